"""GPU parity of the ring path without tables: kept prompt positions and the
ring fill bit-exact against the oracle; the implicit-table ring decode step
bit-identical to the table path (same n_split) and within 2e-3 abs + 1e-2 rel
(elementwise) and 1e-2 of each row's largest |value| of the fp64 oracle."""
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


@pytest.mark.parametrize("n_sink,W", [(64, 4032), (4, 16), (0, 8)])
def test_prefill_keep_positions_bit_exact(n_sink, W):
    S_list = [0, 1, n_sink, n_sink + W - 1, n_sink + W, n_sink + W + 1, 5000, 1_048_576]
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    pos, cnt = wm.prefill_keep_positions(seq, n_sink, W)
    pos_h, cnt_h = host_i32(pos), host_i32(cnt)
    for b, want in enumerate(oracle.prefill_keep_positions(S_list, n_sink, W)):
        assert cnt_h[b] == len(want)
        assert np.array_equal(pos_h[b, :len(want)], want)


@pytest.mark.parametrize("tree_k", [1, 4])
def test_ring_fill_bit_exact(tree_k):
    n_sink, W, d = 64, 1024, 7
    D, H_kv = 256, 2
    S_list = [3, 64, 1088, 1089, 50_000]
    B = len(S_list)
    R = n_sink + W + d * tree_k
    rb = synth.ring_bases(B, R, 2 * B, 11)
    ring_base = torch.tensor(rb, dtype=torch.int32, device=DEV)
    k_pool = synth.normal_bf16((2 * B * R, H_kv, D), 12, DEV)
    v_pool = synth.normal_bf16((2 * B * R, H_kv, D), 13, DEV)
    kp_h, vp_h = bits(k_pool), bits(v_pool)
    rows_k = synth.normal_bf16((B, n_sink + W, H_kv, D), 14, DEV)
    rows_v = synth.normal_bf16((B, n_sink + W, H_kv, D), 15, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    wm.ring_fill(rows_k, rows_v, seq, ring_base, n_sink, W, d, k_pool, v_pool, tree_k=tree_k)
    oracle.ring_fill(bits(rows_k), bits(rows_v), S_list, rb, n_sink, W, d, kp_h, vp_h, tree_k=tree_k)
    assert np.array_equal(bits(k_pool), kp_h) and np.array_equal(bits(v_pool), vp_h)


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 8, 2), (128, 4, 4)])
def test_ring_steps_equal_table_path_and_oracle(D, H_q, H_kv):
    # prefill fill, then gamma = 6 fused ring steps; the same steps through
    # ring_map + build_draft_indices (ring) + the fused table call on a copy
    # of the pools must give the same bits; the oracle runs its own pipeline.
    n_sink, W, d, gamma = 64, 1024, 7, 6
    S_list = [10, 1000, 1088, 1089, 70_000]
    B = len(S_list)
    scale = 1 / math.sqrt(D)
    R = n_sink + W + d
    rb = synth.ring_bases(B, R, B + 3, 21 + D)
    ring_base = torch.tensor(rb, dtype=torch.int32, device=DEV)
    pool = (B + 3) * R
    kp = synth.normal_bf16((pool, H_kv, D), 22 + D, DEV)
    vp = synth.normal_bf16((pool, H_kv, D), 23 + D, DEV)
    rows_k = synth.normal_bf16((B, n_sink + W, H_kv, D), 24, DEV)
    rows_v = synth.normal_bf16((B, n_sink + W, H_kv, D), 25, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    kn = synth.normal_bf16((gamma, B, H_kv, D), 26, DEV)
    vn = synth.normal_bf16((gamma, B, H_kv, D), 27, DEV)
    qs = synth.normal_bf16((gamma, B, 1, H_q, D), 28, DEV)
    o_kp, o_vp = bits(kp), bits(vp)
    wm.ring_fill(rows_k, rows_v, seq, ring_base, n_sink, W, d, kp, vp)
    oracle.ring_fill(bits(rows_k), bits(rows_v), S_list, rb, n_sink, W, d, o_kp, o_vp)
    kp_t, vp_t = kp.clone(), vp.clone()
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=d, windowed=True, stride=n_sink + W)
    tr, lr = wm.build_draft_indices(seq, ring_base=ring_base, **kw)
    otr, olr = oracle.build_draft_indices(np.array(S_list, np.int32), ring_base=np.array(rb, np.int32), **kw)
    reqs = torch.arange(B, dtype=torch.int32, device=DEV)
    for j in range(gamma):
        for n_split in (1, 5, 16, 32, None):
            if n_split is not None and j % 2:
                continue
            a_k, a_v = kp.clone(), vp.clone()
            out_r, lse_r = wm.draft_decode_attn_ring(qs[j], a_k, a_v, seq, ring_base, j, n_sink, W, d, scale,
                                                     k_new=kn[j], v_new=vn[j], n_split=n_split)
            b_k, b_v = kp_t.clone(), vp_t.clone()
            rs = wm.ring_map(ring_base, (seq + j).contiguous(), reqs, n_sink, W, d)
            ns = n_split if n_split is not None else wm.attn_num_splits(B, 1, H_kv, n_sink + W)
            out_t, lse_t = wm.draft_decode_attn_append(kn[j], vn[j], rs, qs[j], b_k, b_v, tr[j], lr[j], scale,
                                                       n_split=ns)
            assert torch.equal(out_r, out_t) and torch.equal(lse_r, lse_t), f"step {j} split {n_split}"
            assert torch.equal(a_k, b_k) and torch.equal(a_v, b_v)
        kp, vp, kp_t, vp_t = a_k, a_v, b_k, b_v
        ors = oracle.ring_map(np.array(rb, np.int32), np.array(S_list, np.int32) + j,
                              np.arange(B, dtype=np.int32), n_sink, W, d)
        oracle.append_kv(bits(kn[j]), bits(vn[j]), ors, o_kp, o_vp)
        ro, rl = oracle.draft_decode_attn(bits(qs[j]), o_kp, o_vp, otr[j], olr[j], scale)
        assert_attn_close(out_r, lse_r, ro, rl, what=f"ring step {j}")
    assert np.array_equal(bits(kp), o_kp) and np.array_equal(bits(vp), o_vp)


def test_ring_step_without_append_and_tree_ring_layout():
    # tree_k = 4 ring layout (modulus W + d*k), no fused append, B = 8,
    # contexts from inside the sinks to 1M
    n_sink, W, d, k = 64, 4032, 7, 4
    D, H_q, H_kv = 256, 16, 2
    S_list = [5, 64, 4095, 4096, 4097, 100_000, 777_777, 1_048_576]
    B = len(S_list)
    R = n_sink + W + d * k
    rb = synth.ring_bases(B, R, B, 31)
    ring_base = torch.tensor(rb, dtype=torch.int32, device=DEV)
    kp = synth.normal_bf16((B * R, H_kv, D), 32, DEV)
    vp = synth.normal_bf16((B * R, H_kv, D), 33, DEV)
    q = synth.normal_bf16((B, 1, H_q, D), 34, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    step = 3
    out, lse = wm.draft_decode_attn_ring(q, kp, vp, seq, ring_base, step, n_sink, W, d, 0.0625, tree_k=k)
    kw = dict(gamma=step + 1, n_sink=n_sink, window=W, depth=d, tree_k=k, windowed=True, stride=n_sink + W)
    otr, olr = oracle.build_draft_indices(np.array(S_list, np.int32), ring_base=np.array(rb, np.int32), **kw)
    ro, rl = oracle.draft_decode_attn(bits(q), bits(kp), bits(vp), otr[step], olr[step], 0.0625)
    assert_attn_close(out, lse, ro, rl, what="tree-layout ring step")


def test_ring_bad_base_is_latched_not_faulted():
    n_sink, W, d = 4, 60, 3
    D, H_q, H_kv = 128, 8, 2
    R = n_sink + W + d
    kp = synth.normal_bf16((2 * R, H_kv, D), 41, DEV)
    vp = synth.normal_bf16((2 * R, H_kv, D), 42, DEV)
    q = synth.normal_bf16((2, 1, H_q, D), 43, DEV)
    seq = torch.tensor([100, 100], dtype=torch.int32, device=DEV)
    ring_base = torch.tensor([0, R + 5], dtype=torch.int32, device=DEV)  # request 1's ring runs past the pool
    wm.device_error(clear=True)
    out, lse = wm.draft_decode_attn_ring(q, kp, vp, seq, ring_base, 0, n_sink, W, d, 0.1, n_split=2)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 1  # WMTP_DEV_SLOT_RANGE
    assert torch.all(torch.isfinite(out))
