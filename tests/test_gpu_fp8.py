"""GPU parity of the fp8 (E4M3) KV path against the fp64 oracle: the
quantising append bit for bit, the attention over E4M3 pools within the
attention tolerance (2e-3 abs + 1e-2 rel elementwise, 1e-2 of each row's
largest |value|) on the same codes and scales."""
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


def _codes(t):
    return t.detach().contiguous().cpu().numpy()


def _quantised_pools(num_slots, H_kv, D, seed, k_scale, v_scale):
    """E4M3 pools holding N(0, 1) bf16 rows quantised by the oracle (host)."""
    kb = bits(synth.normal_bf16((num_slots, H_kv, D), seed, "cpu"))
    vb = bits(synth.normal_bf16((num_slots, H_kv, D), seed + 1, "cpu"))
    kp = np.zeros((num_slots, H_kv, D), np.uint8)
    vp = np.zeros((num_slots, H_kv, D), np.uint8)
    oracle.append_kv_fp8(kb, vb, np.arange(num_slots, dtype=np.int32), k_scale, v_scale, kp, vp)
    return kp, vp


@pytest.mark.parametrize("D,H_kv", [(256, 2), (128, 2), (128, 4), (256, 1)])
def test_append_fp8_bit_exact(D, H_kv):
    n, num_slots = 37, 500
    kn = synth.normal_bf16((n, H_kv, D), 7 + D + H_kv, DEV)
    vn = synth.normal_bf16((n, H_kv, D), 8 + D + H_kv, DEV)
    kn[:3] *= 64  # saturates with the smallest scales below
    # scales: tiny (saturation), typical (amax / 448), large (subnormal codes)
    ks = torch.tensor([0.0625, 4.5 / 448, 7.0, 0.33][:H_kv], dtype=torch.float32, device=DEV)
    vs = torch.tensor([5.0 / 448, 0.9, 0.011, 3.0][:H_kv], dtype=torch.float32, device=DEV)
    slots = synth.permutation(num_slots, 9 + D, DEV)[:n].contiguous()
    kp = synth.e4m3_codes((num_slots, H_kv, D), 10, DEV)
    vp = synth.e4m3_codes((num_slots, H_kv, D), 11, DEV)
    kp_h, vp_h = _codes(kp), _codes(vp)
    wm.append_kv_fp8(kn, vn, slots, ks, vs, kp, vp)
    oracle.append_kv_fp8(bits(kn), bits(vn), host_i32(slots), ks.cpu().numpy(), vs.cpu().numpy(),
                         kp_h, vp_h)
    torch.cuda.synchronize()
    assert np.array_equal(_codes(kp), kp_h)
    assert np.array_equal(_codes(vp), vp_h)


def test_append_fp8_bad_slot_is_latched():
    D, H_kv, num_slots = 128, 2, 64
    kn = synth.normal_bf16((2, H_kv, D), 1, DEV)
    vn = synth.normal_bf16((2, H_kv, D), 2, DEV)
    ones = torch.ones(H_kv, dtype=torch.float32, device=DEV)
    kp = torch.zeros((num_slots, H_kv, D), dtype=torch.uint8, device=DEV)
    vp = torch.zeros_like(kp)
    slots = torch.tensor([3, num_slots + 2], dtype=torch.int32, device=DEV)
    wm.device_error(clear=True)
    wm.append_kv_fp8(kn, vn, slots, ones, ones, kp, vp)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 1  # WMTP_DEV_SLOT_RANGE
    assert int((kp[:3] != 0).sum()) == 0 and int((kp[4:] != 0).sum()) == 0
    assert int((kp[3] != 0).sum()) > 0


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("H_q,H_kv", [(16, 2), (8, 2), (4, 1), (6, 3)])
def test_fp8_attention_sizes_and_splits(D, H_q, H_kv):
    seed = 100 + D + H_q
    num_slots = 3000
    ks = np.linspace(4.0, 6.0, H_kv).astype(np.float32) / 448
    vs = np.linspace(5.0, 3.0, H_kv).astype(np.float32) / 448
    kp_h, vp_h = _quantised_pools(num_slots, H_kv, D, seed, ks, vs)
    kp, vp = torch.from_numpy(kp_h).to(DEV), torch.from_numpy(vp_h).to(DEV)
    ks_d, vs_d = torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV)
    scale = 1 / math.sqrt(D)
    for L in (1, 17, 64, 65, 1000, 2999):
        B = 3
        q = synth.normal_bf16((B, 1, H_q, D), seed + L, DEV)
        table = torch.stack([synth.permutation(num_slots, seed + L + b, DEV) for b in range(B)])
        lens = torch.tensor([L, max(L - 7, 0), min(L + 5, num_slots)], dtype=torch.int32, device=DEV)
        ro, rl = oracle.draft_decode_attn_fp8(bits(q), kp_h, vp_h, ks, vs, host_i32(table),
                                              host_i32(lens), scale)
        for n_split in (1, 3, 16, 24, 37, None):
            out, lse = wm.draft_decode_attn_fp8(q, kp, vp, ks_d, vs_d, table, lens, scale,
                                                n_split=n_split)
            assert_attn_close(out, lse, ro, rl, what=f"fp8 D={D} G={H_q // H_kv} L={L} split={n_split}")


def test_fp8_attention_random_codes_and_outliers():
    # log-uniform codes over 9 octaves, a heavy-tailed score distribution
    D, H_q, H_kv, num_slots = 256, 16, 2, 5000
    kp = synth.e4m3_codes((num_slots, H_kv, D), 21, DEV)
    vp = synth.e4m3_codes((num_slots, H_kv, D), 22, DEV)
    ks = torch.tensor([1 / 64, 1 / 48], dtype=torch.float32, device=DEV)
    vs = torch.tensor([0.5, 1 / 32], dtype=torch.float32, device=DEV)
    q = synth.normal_bf16((2, 3, H_q, D), 23, DEV)
    table = torch.stack([synth.permutation(num_slots, 24 + b, DEV) for b in range(2)])
    lens = torch.tensor([num_slots, 777], dtype=torch.int32, device=DEV)
    ro, rl = oracle.draft_decode_attn_fp8(bits(q), _codes(kp), _codes(vp), ks.cpu().numpy(),
                                          vs.cpu().numpy(), host_i32(table), host_i32(lens), 0.05)
    for n_split in (1, 8, 40):
        out, lse = wm.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.05, n_split=n_split)
        assert_attn_close(out, lse, ro, rl, what=f"fp8 random codes split={n_split}")


def test_fp8_attention_is_deterministic_and_empty_rows():
    D, H_q, H_kv, num_slots = 128, 8, 2, 2000
    kp = synth.e4m3_codes((num_slots, H_kv, D), 31, DEV)
    vp = synth.e4m3_codes((num_slots, H_kv, D), 32, DEV)
    ks = torch.full((H_kv,), 1 / 40, dtype=torch.float32, device=DEV)
    vs = torch.full((H_kv,), 0.25, dtype=torch.float32, device=DEV)
    q = synth.normal_bf16((3, 1, H_q, D), 33, DEV)
    table = torch.stack([synth.permutation(num_slots, 34 + b, DEV) for b in range(3)])
    lens = torch.tensor([1500, 0, 3], dtype=torch.int32, device=DEV)
    a = wm.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.1, n_split=12)
    b = wm.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.1, n_split=12)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.all(a[0][1] == 0) and torch.all(torch.isneginf(a[1][1]))
    ro, rl = oracle.draft_decode_attn_fp8(bits(q), _codes(kp), _codes(vp), ks.cpu().numpy(),
                                          vs.cpu().numpy(), host_i32(table), host_i32(lens), 0.1)
    assert_attn_close(a[0], a[1], ro, rl, what="fp8 empty rows")


def test_fp8_draft_steps_append_then_attend_windowed_ring():
    # gamma = 6 draft steps on a compact ring: each step quantises its own
    # K/V into the ring, then attends the sink + window table; oracle side
    # runs its own append and attention on its own copy of the pools.
    B, gamma, n_sink, W, d = 2, 6, 64, 1024, 7
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    R = n_sink + W + d
    S_list = [50_000, 3_000]
    rb_list = synth.ring_bases(B, R, 2 * B, 41)
    ring_base = torch.tensor(rb_list, dtype=torch.int32, device=DEV)
    ks = torch.tensor([5 / 448, 4 / 448], dtype=torch.float32, device=DEV)
    vs = torch.tensor([4.5 / 448, 6 / 448], dtype=torch.float32, device=DEV)
    o_rk, o_rv = _quantised_pools(2 * B * R, H_kv, D, 42, ks.cpu().numpy(), vs.cpu().numpy())
    ring_k, ring_v = torch.from_numpy(o_rk.copy()).to(DEV), torch.from_numpy(o_rv.copy()).to(DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    kn = synth.normal_bf16((gamma, B, H_kv, D), 43, DEV)
    vn = synth.normal_bf16((gamma, B, H_kv, D), 44, DEV)
    qs = synth.normal_bf16((gamma, B, 1, H_q, D), 45, DEV)
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=d, windowed=True, stride=n_sink + W)
    tr, lr = wm.build_draft_indices(seq, ring_base=ring_base, **kw)
    otr, olr = oracle.build_draft_indices(np.array(S_list, np.int32),
                                          ring_base=np.array(rb_list, np.int32), **kw)
    reqs = torch.arange(B, dtype=torch.int32, device=DEV)
    for j in range(gamma):
        pos = (seq + j).contiguous()
        rs = wm.ring_map(ring_base, pos, reqs, n_sink, W, d)
        wm.append_kv_fp8(kn[j], vn[j], rs, ks, vs, ring_k, ring_v)
        out, lse = wm.draft_decode_attn_fp8(qs[j], ring_k, ring_v, ks, vs, tr[j], lr[j], scale)
        ors = oracle.ring_map(np.array(rb_list, np.int32), host_i32(pos), np.arange(B, dtype=np.int32),
                              n_sink, W, d)
        oracle.append_kv_fp8(bits(kn[j]), bits(vn[j]), ors, ks.cpu().numpy(), vs.cpu().numpy(), o_rk, o_rv)
        ro, rl = oracle.draft_decode_attn_fp8(bits(qs[j]), o_rk, o_rv, ks.cpu().numpy(), vs.cpu().numpy(),
                                              otr[j], olr[j], scale)
        assert_attn_close(out, lse, ro, rl, what=f"fp8 ring step {j}")
    assert np.array_equal(_codes(ring_k), o_rk) and np.array_equal(_codes(ring_v), o_rv)


def test_fp8_million_token_step_sampled():
    # S = 1,048,576 keys of random codes; windowed rows all checked,
    # full-context rows sampled (one query head per KV head).
    S, n_sink, W = 1_048_576, 64, 4032
    D, H_q, H_kv = 256, 16, 2
    scale = 1 / math.sqrt(D)
    pool = S + 1
    kp = synth.e4m3_codes((pool, H_kv, D), 51, DEV)
    vp = synth.e4m3_codes((pool, H_kv, D), 52, DEV)
    ks = torch.tensor([1 / 64, 1 / 80], dtype=torch.float32, device=DEV)
    vs = torch.tensor([1 / 16, 1 / 32], dtype=torch.float32, device=DEV)
    q = synth.normal_bf16((1, 1, H_q, D), 53, DEV)
    rtt = synth.permutation(pool, 54, DEV).view(1, -1)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    kp_h, vp_h = _codes(kp), _codes(vp)
    rng = np.random.default_rng(55)
    for windowed in (True, False):
        kw = dict(gamma=1, n_sink=n_sink, window=W, depth=2, windowed=windowed,
                  stride=4096 if windowed else pool)
        tg, lg = wm.build_draft_indices(seq, req_to_token=rtt, **kw)
        tr, lr = oracle.build_draft_indices(np.array([S], np.int32), req_to_token=host_i32(rtt), **kw)
        rows = None if windowed else np.array([rng.integers(0, 8), 8 + rng.integers(0, 8)])
        out, lse = wm.draft_decode_attn_fp8(q, kp, vp, ks, vs, tg[0], lg[0], scale)
        ro, rl = oracle.draft_decode_attn_fp8(bits(q), kp_h, vp_h, ks.cpu().numpy(), vs.cpu().numpy(),
                                              tr[0], lr[0], scale, rows=rows)
        assert_attn_close(out, lse, ro, rl, rows=rows, what=f"fp8 1M windowed={windowed}")
