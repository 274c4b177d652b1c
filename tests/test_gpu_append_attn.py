"""GPU tests of the fused draft step (append_kv + draft_decode_attn in one
launch): bit-identical to the two calls in sequence (outputs, lse and pool
contents) and, through that and directly, to the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import synth
from wmtp_testutil import assert_attn_close, bits, host_i32

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    wm.build()
    wm.load()
    wm.device_error(clear=True)
    yield
    assert wm.device_error(clear=True) == 0


def _setup(seed, B, num_slots, H_q, H_kv, D, n_new, lens_list):
    kp = synth.normal_bf16((num_slots, H_kv, D), seed, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), seed + 1, DEV)
    q = synth.normal_bf16((B, 1, H_q, D), seed + 2, DEV)
    # disjoint slot sets per request; the new tokens take the last n_new
    # positions of each row
    perm = synth.permutation(num_slots, seed + 3, DEV)
    stride = max(lens_list)
    table = torch.full((B, stride), -1, dtype=torch.int32, device=DEV)
    off = 0
    for b, L in enumerate(lens_list):
        table[b, :L] = perm[off:off + L]
        off += L
    lens = torch.tensor(lens_list, dtype=torch.int32, device=DEV)
    new_slots = torch.stack([table[b, L - n_new:L] for b, L in enumerate(lens_list)]).contiguous()
    k_new = synth.normal_bf16((B, n_new, H_kv, D), seed + 4, DEV)
    v_new = synth.normal_bf16((B, n_new, H_kv, D), seed + 5, DEV)
    return kp, vp, q, table, lens, new_slots, k_new, v_new


def _two_calls(kp, vp, q, table, lens, new_slots, k_new, v_new, scale, n_split):
    B, n_new, H_kv, D = k_new.shape
    wm.append_kv(k_new.reshape(B * n_new, H_kv, D), v_new.reshape(B * n_new, H_kv, D),
                 new_slots.reshape(-1), kp, vp)
    return wm.draft_decode_attn(q, kp, vp, table, lens, scale, n_split=n_split)


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 8, 2), (128, 4, 4)])
@pytest.mark.parametrize("n_new", [1, 2])
def test_fused_equals_append_then_attend(D, H_q, H_kv, n_new):
    B, num_slots = 3, 9000
    lens_list = [2999, 1500, 64]
    scale = 1 / math.sqrt(D)
    kp, vp, q, table, lens, ns, kn, vn = _setup(D + H_q + n_new, B, num_slots, H_q, H_kv, D, n_new,
                                                lens_list)
    for n_split in (1, 3, 16, 32, 37):
        kp_a, vp_a = kp.clone(), vp.clone()
        kp_b, vp_b = kp.clone(), vp.clone()
        out_a, lse_a = _two_calls(kp_a, vp_a, q, table, lens, ns, kn, vn, scale, n_split)
        out_b, lse_b = wm.draft_decode_attn_append(kn, vn, ns, q, kp_b, vp_b, table, lens, scale,
                                                   n_split=n_split)
        assert torch.equal(out_a, out_b), f"n_split={n_split}: out differs"
        assert torch.equal(lse_a, lse_b), f"n_split={n_split}: lse differs"
        assert torch.equal(kp_a, kp_b) and torch.equal(vp_a, vp_b), f"n_split={n_split}: pools differ"
    # and against the oracle (append then attend, fp64)
    kp_h, vp_h = bits(kp), bits(vp)
    oracle.append_kv(bits(kn.reshape(-1, H_kv, D)), bits(vn.reshape(-1, H_kv, D)),
                     host_i32(ns.reshape(-1)), kp_h, vp_h)
    ro, rl = oracle.draft_decode_attn(bits(q), kp_h, vp_h, host_i32(table), host_i32(lens), scale)
    assert_attn_close(out_b, lse_b, ro, rl, what=f"fused D={D} n_new={n_new}")
    assert np.array_equal(bits(kp_b), kp_h) and np.array_equal(bits(vp_b), vp_h)


def test_fused_sequential_windowed_ring_steps():
    # gamma=6 sequential draft steps on a compact ring (n_sink + W + d slots
    # per request), each appending its own K/V and attending the sink +
    # window table, against the oracle running append then attend.
    B, gamma, n_sink, W, d = 2, 6, 64, 1024, 7
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    R = n_sink + W + d
    S_list = [50_000, 3_000]
    rb_list = synth.ring_bases(B, R, 2 * B, 77)
    ring_base = torch.tensor(rb_list, dtype=torch.int32, device=DEV)
    ring_k = synth.normal_bf16((2 * B * R, H_kv, D), 78, DEV)
    ring_v = synth.normal_bf16((2 * B * R, H_kv, D), 79, DEV)
    o_rk, o_rv = bits(ring_k), bits(ring_v)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    kn = synth.normal_bf16((gamma, B, H_kv, D), 80, DEV)
    vn = synth.normal_bf16((gamma, B, H_kv, D), 81, DEV)
    qs = synth.normal_bf16((gamma, B, 1, H_q, D), 82, DEV)
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=d, windowed=True, stride=n_sink + W)
    tr, lr = wm.build_draft_indices(seq, ring_base=ring_base, **kw)
    otr, olr = oracle.build_draft_indices(np.array(S_list, np.int32),
                                          ring_base=np.array(rb_list, np.int32), **kw)
    reqs = torch.arange(B, dtype=torch.int32, device=DEV)
    for j in range(gamma):
        pos = (seq + j).contiguous()
        rs = wm.ring_map(ring_base, pos, reqs, n_sink, W, d)
        out, lse = wm.draft_decode_attn_append(kn[j], vn[j], rs, qs[j], ring_k, ring_v, tr[j], lr[j],
                                               scale)
        ors = oracle.ring_map(np.array(rb_list, np.int32), host_i32(pos), np.arange(B, dtype=np.int32),
                              n_sink, W, d)
        oracle.append_kv(bits(kn[j]), bits(vn[j]), ors, o_rk, o_rv)
        ro, rl = oracle.draft_decode_attn(bits(qs[j]), o_rk, o_rv, otr[j], olr[j], scale)
        assert_attn_close(out, lse, ro, rl, what=f"ring step {j}")
    assert np.array_equal(bits(ring_k), o_rk) and np.array_equal(bits(ring_v), o_rv)


def test_fused_bad_new_slot_is_latched_like_two_calls():
    D, H_q, H_kv = 128, 8, 2
    B, num_slots = 2, 3000
    lens_list = [700, 300]
    scale = 1 / math.sqrt(D)
    kp, vp, q, table, lens, ns, kn, vn = _setup(5, B, num_slots, H_q, H_kv, D, 1, lens_list)
    # request 1's new token points outside the pool, in its table and its slot
    table[1, 299] = num_slots + 5
    ns[1, 0] = num_slots + 5
    kp_a, vp_a = kp.clone(), vp.clone()
    kp_b, vp_b = kp.clone(), vp.clone()
    wm.device_error(clear=True)
    out_a, lse_a = _two_calls(kp_a, vp_a, q, table, lens, ns, kn, vn, scale, 4)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 1  # WMTP_DEV_SLOT_RANGE
    out_b, lse_b = wm.draft_decode_attn_append(kn, vn, ns, q, kp_b, vp_b, table, lens, scale, n_split=4)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 1  # WMTP_DEV_SLOT_RANGE
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    assert torch.equal(kp_a, kp_b) and torch.equal(vp_a, vp_b)


def test_headline_fused_step_at_one_million_keys():
    """The benchmark's own million-token step, in the launch configuration it
    times: the workload object of the benchmark (B=1, S=1,048,576, H_q=16,
    H_kv=2, D=256, 1 % of K rows x4, permuted page table), its full-context
    arm (six fused append + attention launches over 1,048,577.. keys, the
    split count of wmtp_attn_num_splits, its merge) and its windowed arm.
    Checked: the full-context outputs equal, bit for bit, append_kv followed
    by the unfused attention on a copy of the pools; sampled query heads (two
    per step, one per KV head) and every windowed head match the fp64 oracle
    after its own appends; the index tables match the oracle's; and after the
    six steps both pools equal the oracle's pools bit for bit."""
    import bench

    cfg = bench.WORKLOADS["1m"]
    w = bench.Workload(cfg, DEV)
    g, S = cfg["gamma"], cfg["S"]
    assert w.ns_full == wm.attn_num_splits(1, 1, cfg["H_kv"], S + g, DEV)
    kp_h, vp_h = bits(w.kp), bits(w.vp)
    kp2, vp2 = w.kp.clone(), w.vp.clone()

    w.full_arm()
    torch.cuda.synchronize()
    for j in range(g):
        wm.append_kv(w.kn[j], w.vn[j], w.slots[j], kp2, vp2)
        o2, l2 = wm.draft_decode_attn(w.q[j], kp2, vp2, w.tab_full[j], w.len_full[j], w.scale,
                                      n_split=w.ns_full, workspace=w.ws_full)
        assert torch.equal(o2, w.out_full[j]) and torch.equal(l2, w.lse_full[j]), f"fused != two calls, step {j}"
    assert torch.equal(kp2, w.kp) and torch.equal(vp2, w.vp)
    del kp2, vp2

    seq_h = host_i32(w.seq)
    rtt_h = host_i32(w.rtt)
    tab_f, len_f = oracle.build_draft_indices(seq_h, g, cfg["n_sink"], cfg["W"], g + 1, windowed=False,
                                              req_to_token=rtt_h, stride=w.full_stride)
    assert np.array_equal(host_i32(w.len_full), len_f)
    tab_g = host_i32(w.tab_full)
    for j in range(g):  # entries past a row's length are not written
        assert np.array_equal(tab_g[j, 0, :len_f[j, 0]], tab_f[j, 0, :len_f[j, 0]]), f"full table, step {j}"
    rng = np.random.default_rng(77)
    for j in range(g):
        oracle.append_kv(bits(w.kn[j]), bits(w.vn[j]), host_i32(w.slots[j]), kp_h, vp_h)
        rows = np.array([rng.integers(0, 8), 8 + rng.integers(0, 8)])
        ro, rl = oracle.draft_decode_attn(bits(w.q[j]), kp_h, vp_h, tab_f[j], len_f[j], w.scale, rows=rows)
        assert_attn_close(w.out_full[j], w.lse_full[j], ro, rl, rows=rows, what=f"1M fused full step {j}")
    assert np.array_equal(bits(w.kp), kp_h) and np.array_equal(bits(w.vp), vp_h), "pools differ from the oracle's"

    w.win_arm()
    torch.cuda.synchronize()
    tab_w, len_w = oracle.build_draft_indices(seq_h, g, cfg["n_sink"], cfg["W"], g + 1, windowed=True,
                                              req_to_token=rtt_h, stride=w.win_stride)
    assert np.array_equal(host_i32(w.len_win), len_w)
    tab_g = host_i32(w.tab_win)
    for j in range(g):
        assert np.array_equal(tab_g[j, 0, :len_w[j, 0]], tab_w[j, 0, :len_w[j, 0]]), f"windowed table, step {j}"
    for j in range(g):
        ro, rl = oracle.draft_decode_attn(bits(w.q[j]), kp_h, vp_h, tab_w[j], len_w[j], w.scale)
        assert_attn_close(w.out_win[j], w.lse_win[j], ro, rl, what=f"1M fused windowed step {j}")
    assert np.array_equal(bits(w.kp), kp_h) and np.array_equal(bits(w.vp), vp_h)
