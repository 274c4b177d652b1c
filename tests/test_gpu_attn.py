"""GPU parity of split-KV draft decode attention against the fp64 oracle.

The GPU pipeline (GPU index builder -> GPU append -> GPU attention) and the
oracle pipeline (oracle builder -> oracle append -> oracle attention) run on
the same seeded inputs; outputs must agree within 2e-3 abs + 1e-2 rel
(elementwise) and 1e-2 of each row's largest |value|.  Layout invariants
(windowed == full inside the window, ring == un-ringed) are checked bit for
bit GPU against GPU.
"""
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


def _run_both(q, kp, vp, table, lens, scale, n_split=None, rows=None):
    out, lse = wm.draft_decode_attn(q, kp, vp, table, lens, scale, n_split=n_split)
    ref_out, ref_lse = oracle.draft_decode_attn(bits(q), bits(kp), bits(vp), host_i32(table),
                                                host_i32(lens), scale, rows=rows)
    return out, lse, ref_out, ref_lse


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (16, 2), (4, 1), (6, 3)])
def test_attn_sizes_and_splits(D, H_q, H_kv):
    seed = D + 10 * H_q + H_kv
    num_slots = 3000
    kp = synth.normal_bf16((num_slots, H_kv, D), seed, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), seed + 1, DEV)
    for L in (1, 2, 15, 16, 17, 63, 64, 65, 129, 1000, 2999):
        B = 3
        q = synth.normal_bf16((B, 1, H_q, D), seed + L, DEV)
        table = torch.stack([synth.permutation(num_slots, seed + L + b, DEV) for b in range(B)])
        lens = torch.tensor([L, max(L - 7, 0), min(L + 5, num_slots)], dtype=torch.int32, device=DEV)
        # n_split <= 16 merges through one thread-block cluster; 18, 24, 64
        # and 128 in two levels (clusters of 9, 12, 16 and 16; 2 to 8
        # clusters) where the device holds them; 37 and 136 have no cluster
        # plan: the slice merge where the whole grid fits on the device, else
        # the last CTA in split order
        for n_split in (1, 2, 3, 7, 16, 18, 24, 37, 64, 128, 136, None):
            out, lse, ro, rl = _run_both(q, kp, vp, table, lens, 1 / math.sqrt(D), n_split)
            assert_attn_close(out, lse, ro, rl, what=f"D={D} G={H_q // H_kv} L={L} split={n_split}")


def test_attn_many_query_tokens_and_empty_rows():
    D, H_q, H_kv = 256, 16, 2
    num_slots = 700
    kp = synth.normal_bf16((num_slots, H_kv, D), 21, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 22, DEV)
    B, n_q = 4, 3
    q = synth.normal_bf16((B, n_q, H_q, D), 23, DEV)
    table = torch.stack([synth.permutation(num_slots, 24 + b, DEV) for b in range(B)])
    lens = torch.tensor([0, 700, 1, 333], dtype=torch.int32, device=DEV)
    for n_split in (1, 4, 11, 17, 32, 48):
        out, lse, ro, rl = _run_both(q, kp, vp, table, lens, 0.0625, n_split)
        assert_attn_close(out, lse, ro, rl, what=f"n_q=3 split={n_split}")
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))


@pytest.mark.parametrize("D", [128, 256])
def test_attn_slice_merge_against_oracle_and_last_cta_merge(D):
    """Split counts with no cluster plan at B = 1 (every split merging its
    own output slice after the others arrive, when the grid fits on the
    device), including plans that leave trailing splits empty, against the
    fp64 oracle and against the last-CTA merge of the same partials (the
    workspace-free entry point always merges that way)."""
    H_q, H_kv = 16, 2
    num_slots = 12_000
    kp = synth.normal_bf16((num_slots, H_kv, D), 51, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 52, DEV)
    q = synth.normal_bf16((1, 1, H_q, D), 53, DEV)
    table = synth.permutation(num_slots, 54, DEV).view(1, -1)
    for L, n_split in ((11_999, 17), (11_999, 37), (9_000, 76), (4_000, 76), (11_999, 101), (5_000, 151)):
        lens = torch.tensor([L], dtype=torch.int32, device=DEV)
        out, lse, ro, rl = _run_both(q, kp, vp, table, lens, 1 / math.sqrt(D), n_split)
        assert_attn_close(out, lse, ro, rl, what=f"D={D} L={L} split={n_split}")
        o2 = torch.empty_like(out)
        l2 = torch.empty_like(lse)
        wm.draft_decode_attn_noalloc(q, kp, vp, table, lens, 1 / math.sqrt(D), o2, l2, n_split)
        torch.testing.assert_close(out, o2, atol=2e-3, rtol=1e-2)
        torch.testing.assert_close(lse, l2, atol=2e-3, rtol=1e-2)
        # repeatable bit for bit (the counters are back at zero after each call)
        out_b, lse_b = wm.draft_decode_attn(q, kp, vp, table, lens, 1 / math.sqrt(D), n_split=n_split)
        assert torch.equal(out, out_b) and torch.equal(lse, lse_b)


def test_attn_maximum_split_count():
    D, H_q, H_kv = 128, 8, 2
    num_slots = 70_000
    kp = synth.normal_bf16((num_slots, H_kv, D), 31, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 32, DEV)
    q = synth.normal_bf16((1, 1, H_q, D), 33, DEV)
    table = synth.permutation(num_slots, 34, DEV).view(1, -1)
    lens = torch.tensor([num_slots], dtype=torch.int32, device=DEV)
    out, lse, ro, rl = _run_both(q, kp, vp, table, lens, 1 / math.sqrt(D), 1024)
    assert_attn_close(out, lse, ro, rl, what="n_split=1024")


def test_attn_deterministic_and_split_consistent():
    D, H_q, H_kv = 256, 16, 2
    num_slots = 20_000
    kp = synth.normal_bf16((num_slots, H_kv, D), 41, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 42, DEV)
    q = synth.normal_bf16((2, 1, H_q, D), 43, DEV)
    table = torch.stack([synth.permutation(num_slots, 44 + b, DEV) for b in range(2)])
    lens = torch.tensor([num_slots, 12_345], dtype=torch.int32, device=DEV)
    a = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=9)
    b = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=9)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    c = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=2)
    torch.testing.assert_close(a[0], c[0], atol=2e-3, rtol=1e-2)
    d1 = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=40)
    d2 = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=40)
    assert torch.equal(d1[0], d2[0]) and torch.equal(d1[1], d2[1])
    torch.testing.assert_close(a[0], d1[0], atol=2e-3, rtol=1e-2)
    # two-level merge: the last cluster merges in cluster order
    e1 = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=64)
    e2 = wm.draft_decode_attn(q, kp, vp, table, lens, 0.0625, n_split=64)
    assert torch.equal(e1[0], e2[0]) and torch.equal(e1[1], e2[1])
    torch.testing.assert_close(a[0], e1[0], atol=2e-3, rtol=1e-2)


def test_attn_tiny_windowed_workload():
    # B=1, H_q=8, H_kv=2, D=128, n_sink=64, W=1024, one draft query, pool =
    # seeded permutation; S=8192 windowed and full vs the oracle, and S=1000
    # (inside the window) windowed == full bit for bit on the GPU.
    D, H_q, H_kv, n_sink, W = 128, 8, 2, 64, 1024
    scale = 1 / math.sqrt(D)
    for S in (8192, 1000):
        pool = S + 1
        kp = synth.normal_bf16((pool, H_kv, D), 1000 + S, DEV)
        vp = synth.normal_bf16((pool, H_kv, D), 1001 + S, DEV)
        q = synth.normal_bf16((1, 1, H_q, D), 1002 + S, DEV)
        rtt = synth.permutation(pool, 1003 + S, DEV).view(1, -1)
        seq = torch.tensor([S], dtype=torch.int32, device=DEV)
        outs = {}
        for windowed in (True, False):
            kw = dict(gamma=1, n_sink=n_sink, window=W, depth=2, windowed=windowed, stride=pool)
            tg, lg = wm.build_draft_indices(seq, req_to_token=rtt, **kw)
            out, lse = wm.draft_decode_attn(q, kp, vp, tg[0], lg[0], scale)
            tr, lr = oracle.build_draft_indices(np.array([S], np.int32), req_to_token=host_i32(rtt), **kw)
            ro, rl = oracle.draft_decode_attn(bits(q), bits(kp), bits(vp), tr[0], lr[0], scale)
            assert_attn_close(out, lse, ro, rl, what=f"S={S} windowed={windowed}")
            outs[windowed] = (out, lse)
        if S <= n_sink + W:
            assert torch.equal(outs[True][0], outs[False][0])
            assert torch.equal(outs[True][1], outs[False][1])


@pytest.mark.parametrize("permuted", [True, False])
def test_attn_sequential_draft_steps_131k(permuted):
    # S=131072, gamma=6 draft steps at positions S..S+5, each appending its own
    # K/V before attending; full table and sink+window table.
    S, gamma, n_sink, W = 131072, 6, 64, 4032
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    pool = S + gamma
    kp = synth.normal_bf16((pool, H_kv, D), 2000, DEV)
    vp = synth.normal_bf16((pool, H_kv, D), 2001, DEV)
    kn = synth.normal_bf16((gamma, 1, H_kv, D), 2002, DEV)
    vn = synth.normal_bf16((gamma, 1, H_kv, D), 2003, DEV)
    qs = synth.normal_bf16((gamma, 1, 1, H_q, D), 2004, DEV)
    rtt = (synth.permutation(pool, 2005, DEV) if permuted
           else torch.arange(pool, dtype=torch.int32, device=DEV)).view(1, -1)
    rtt_h = host_i32(rtt)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    kp_h, vp_h = bits(kp), bits(vp)
    tabs = {}
    for windowed in (True, False):
        kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=gamma + 1, windowed=windowed,
                  stride=4096 if windowed else pool)
        tabs[windowed] = (wm.build_draft_indices(seq, req_to_token=rtt, **kw),
                          oracle.build_draft_indices(np.array([S], np.int32), req_to_token=rtt_h, **kw))
    for j in range(gamma):
        slot = rtt[:, S + j].contiguous()
        wm.append_kv(kn[j], vn[j], slot, kp, vp)
        oracle.append_kv(bits(kn[j]), bits(vn[j]), host_i32(slot), kp_h, vp_h)
        for windowed in (True, False):
            (tg, lg), (tr, lr) = tabs[windowed]
            out, lse = wm.draft_decode_attn(qs[j], kp, vp, tg[j], lg[j], scale)
            ro, rl = oracle.draft_decode_attn(bits(qs[j]), kp_h, vp_h, tr[j], lr[j], scale)
            assert_attn_close(out, lse, ro, rl, what=f"step {j} windowed={windowed}")


def test_attn_million_token_step_sampled():
    # S = 1,048,576, 1 % of K rows x4, gamma = 6; windowed rows all checked,
    # full-context rows sampled (two query heads per step, one per KV head).
    S, gamma, n_sink, W = 1_048_576, 6, 64, 4032
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    pool = S + gamma
    kp = synth.normal_bf16((pool, H_kv, D), 3000, DEV)
    synth.scale_random_rows_(kp, 0.01, 4.0, 3001)
    vp = synth.normal_bf16((pool, H_kv, D), 3002, DEV)
    qs = synth.normal_bf16((gamma, 1, 1, H_q, D), 3003, DEV)
    rtt = synth.permutation(pool, 3004, DEV).view(1, -1)
    rtt_h = host_i32(rtt)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    kp_h, vp_h = bits(kp), bits(vp)
    rng = np.random.default_rng(3005)
    for windowed in (True, False):
        kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=gamma + 1, windowed=windowed,
                  stride=4096 if windowed else pool)
        tg, lg = wm.build_draft_indices(seq, req_to_token=rtt, **kw)
        tr, lr = oracle.build_draft_indices(np.array([S], np.int32), req_to_token=rtt_h, **kw)
        for j in range(gamma):
            rows = None if windowed else np.array([rng.integers(0, 8), 8 + rng.integers(0, 8)])
            out, lse = wm.draft_decode_attn(qs[j], kp, vp, tg[j], lg[j], scale)
            ro, rl = oracle.draft_decode_attn(bits(qs[j]), kp_h, vp_h, tr[j], lr[j], scale, rows=rows)
            assert_attn_close(out, lse, ro, rl, rows=rows, what=f"1M step {j} windowed={windowed}")


def test_attn_ring_equals_unringed_batch():
    # B=6 requests at lengths ~U[900K, 1M], ring of n_sink+W+d = 4103 slots per
    # request at seeded ring_base; gamma=6 steps of append + windowed attention.
    # Ring and un-ringed layouts must agree bit for bit; the ring results
    # must match the oracle (which builds its own ring from the logical rows).
    B, gamma, n_sink, W, d = 6, 6, 64, 4032, 7
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    R = n_sink + W + d
    S_list = synth.uniform_lengths(B, 900_000, 1_048_576, 4000)
    ctx = [s + gamma for s in S_list]
    total = sum(ctx)
    flat_k = synth.normal_bf16((total, H_kv, D), 4001, DEV)
    flat_v = synth.normal_bf16((total, H_kv, D), 4002, DEV)
    perm = synth.permutation(total, 4003, DEV)
    max_ctx = max(ctx)
    rtt = torch.zeros((B, max_ctx), dtype=torch.int32, device=DEV)
    off = 0
    for b in range(B):
        rtt[b, :ctx[b]] = perm[off:off + ctx[b]]
        off += ctx[b]
    rb_list = synth.ring_bases(B, R, 2 * B, 4004)
    ring_base = torch.tensor(rb_list, dtype=torch.int32, device=DEV)
    ring_k = torch.zeros((2 * B * R, H_kv, D), dtype=torch.bfloat16, device=DEV)
    ring_v = torch.zeros_like(ring_k)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    # live logical positions before the step: sinks + the window of step 0
    live_pos, live_req = [], []
    for b, S in enumerate(S_list):
        ps = list(range(n_sink)) + list(range(S + 1 - W, S))
        live_pos += ps
        live_req += [b] * len(ps)
    lp = torch.tensor(live_pos, dtype=torch.int32, device=DEV)
    lr_ = torch.tensor(live_req, dtype=torch.int32, device=DEV)
    src_slots = rtt[lr_.long(), lp.long()].contiguous()
    ring_slots = wm.ring_map(ring_base, lp, lr_, n_sink, W, d)
    wm.append_kv(flat_k[src_slots.long()].contiguous(), flat_v[src_slots.long()].contiguous(),
                 ring_slots, ring_k, ring_v)
    # oracle's own ring pool from the same logical rows
    o_rk = np.zeros((2 * B * R, H_kv, D), np.uint16)
    o_rv = np.zeros_like(o_rk)
    o_slots = oracle.ring_map(np.array(rb_list, np.int32), np.array(live_pos, np.int32),
                              np.array(live_req, np.int32), n_sink, W, d)
    oracle.append_kv(bits(flat_k[src_slots.long()]), bits(flat_v[src_slots.long()]), o_slots, o_rk, o_rv)

    kn = synth.normal_bf16((gamma, B, H_kv, D), 4005, DEV)
    vn = synth.normal_bf16((gamma, B, H_kv, D), 4006, DEV)
    qs = synth.normal_bf16((gamma, B, 1, H_q, D), 4007, DEV)
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=d, windowed=True, stride=4096)
    tf, lf = wm.build_draft_indices(seq, req_to_token=rtt, **kw)
    tr, lr = wm.build_draft_indices(seq, ring_base=ring_base, **kw)
    otr, olr = oracle.build_draft_indices(np.array(S_list, np.int32), ring_base=np.array(rb_list, np.int32), **kw)
    assert torch.equal(lf, lr)
    reqs = torch.arange(B, dtype=torch.int32, device=DEV)
    for j in range(gamma):
        pos = (seq + j).contiguous()
        flat_slot = rtt[torch.arange(B, device=DEV), pos.long()].contiguous()
        wm.append_kv(kn[j], vn[j], flat_slot, flat_k, flat_v)
        rs = wm.ring_map(ring_base, pos, reqs, n_sink, W, d)
        wm.append_kv(kn[j], vn[j], rs, ring_k, ring_v)
        ors = oracle.ring_map(np.array(rb_list, np.int32), host_i32(pos), np.arange(B, dtype=np.int32), n_sink, W, d)
        oracle.append_kv(bits(kn[j]), bits(vn[j]), ors, o_rk, o_rv)
        a = wm.draft_decode_attn(qs[j], flat_k, flat_v, tf[j], lf[j], scale)
        b = wm.draft_decode_attn(qs[j], ring_k, ring_v, tr[j], lr[j], scale)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), f"ring != un-ringed at step {j}"
        ro, rl = oracle.draft_decode_attn(bits(qs[j]), o_rk, o_rv, otr[j], olr[j], scale)
        assert_attn_close(b[0], b[1], ro, rl, what=f"ring step {j}")


def test_attn_bad_slot_is_latched_not_faulted():
    D, H_q, H_kv = 128, 8, 2
    kp = synth.normal_bf16((100, H_kv, D), 51, DEV)
    q = synth.normal_bf16((1, 1, H_q, D), 52, DEV)
    table = torch.arange(100, dtype=torch.int32, device=DEV).view(1, -1).clone()
    table[0, 17] = 100  # one past the pool
    lens = torch.tensor([100], dtype=torch.int32, device=DEV)
    out, lse = wm.draft_decode_attn(q, kp, kp, table, lens, 0.1, n_split=2)
    assert wm.device_error(clear=True) == 1
    assert torch.isfinite(out).all()
