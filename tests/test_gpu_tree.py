"""GPU parity of tree-draft attention over the ring against the fp64 oracle
("Windowed-MTP" §7, tree speculation; reading R5: node (branch, depth i)
attends keep(S+i+1) with its own branch's draft nodes).  Tolerance as for
the chain: 2e-3 abs + 1e-2 rel elementwise and 1e-2 of each row's max."""
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


def _ring_pool(S_list, n_sink, W, d, k, H_kv, D, seed):
    R = n_sink + W + d * k
    B = len(S_list)
    ring_base = synth.ring_bases(B, R, B + 2, seed)
    n = (B + 2) * R
    kp = synth.normal_bf16((n, H_kv, D), seed + 1, DEV)
    vp = synth.normal_bf16((n, H_kv, D), seed + 2, DEV)
    return (torch.tensor(ring_base, dtype=torch.int32, device=DEV), kp, vp)


def _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed, n_split=None, rows=None):
    rb, kp, vp = _ring_pool(S_list, n_sink, W, d, k, H_kv, D, seed)
    B = len(S_list)
    q = synth.normal_bf16((B, k * d, H_q, D), seed + 3, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    scale = 1 / math.sqrt(D)
    out, lse = wm.tree_draft_attn(q, kp, vp, seq, rb, n_sink, W, d, k, scale, n_split=n_split)
    ro, rl = oracle.tree_draft_attn(bits(q), bits(kp), bits(vp), np.array(S_list, np.int32),
                                    host_i32(rb), n_sink, W, d, k, scale, rows=rows)
    assert_attn_close(out, lse, ro, rl, rows=rows,
                      what=f"S={S_list} sink={n_sink} W={W} d={d} k={k} G={H_q // H_kv} D={D} split={n_split}")
    return out, lse


@pytest.mark.parametrize("n_sink,W,d,k", [(0, 5, 3, 2), (3, 16, 3, 4), (2, 4, 7, 3), (64, 1024, 7, 4),
                                          (5, 40, 1, 1), (4, 9, 7, 1)])
@pytest.mark.parametrize("D,H_q,H_kv", [(128, 8, 2), (256, 16, 2), (256, 4, 1)])
def test_tree_geometries(n_sink, W, d, k, D, H_q, H_kv):
    # committed lengths on both sides of every boundary: empty context, inside
    # the sinks, at the window edge, just past it and far past it
    S_list = sorted({0, 1, max(n_sink - 1, 0), n_sink + W - 3 if n_sink + W > 3 else 1,
                     n_sink + W, n_sink + W + 10, 7 * (n_sink + W) + 5})
    for n_split in (1, 3, None):
        _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed=W + 7 * d + k, n_split=n_split)


def test_tree_width_one_equals_chain_kernel():
    # k = 1: node i is draft step i of the chain (table built by the index
    # builder in the ring layout, attended by the split-KV kernel)
    n_sink, W, d, H_q, H_kv, D = 64, 1024, 7, 16, 2, 256
    S_list = [3000, 70_000, 1100]
    rb, kp, vp = _ring_pool(S_list, n_sink, W, d, 1, H_kv, D, 77)
    B = len(S_list)
    q = synth.normal_bf16((B, d, H_q, D), 78, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    out_t, lse_t = wm.tree_draft_attn(q, kp, vp, seq, rb, n_sink, W, d, 1, 1 / 16)
    tab, lens = wm.build_draft_indices(seq, d, n_sink, W, d, windowed=True, ring_base=rb)
    for i in range(d):
        out_c, lse_c = wm.draft_decode_attn(q[:, i:i + 1].contiguous(), kp, vp, tab[i], lens[i], 1 / 16)
        torch.testing.assert_close(out_t[:, i:i + 1], out_c, atol=2e-3, rtol=1e-2)
        torch.testing.assert_close(lse_t[:, i:i + 1], lse_c, atol=2e-3, rtol=1e-2)


@pytest.mark.parametrize("W", [1024, 2048, 4096, 8192])
def test_tree_drafter_window_sweep(W):
    # B=8 requests, contexts log-uniform in [32K, 1M], k=4, d=7 (28 nodes),
    # H_q=16, H_kv=2, D=256, n_sink=64; ring of n_sink + W + d*k slots.
    n_sink, d, k, H_q, H_kv, D = 64, 7, 4, 16, 2, 256
    S_list = synth.log_uniform_lengths(8, 32_768, 1_048_576, 5000)
    n_rows = 8 * k * d * H_q
    rows = None if W <= 2048 else np.random.default_rng(W).choice(n_rows, 512, replace=False)
    out, lse = _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed=5000 + W, rows=rows)
    # bitwise repeatable
    rb, kp, vp = _ring_pool(S_list, n_sink, W, d, k, H_kv, D, 5000 + W)
    q = synth.normal_bf16((8, k * d, H_q, D), 5000 + W + 3, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    o2, l2 = wm.tree_draft_attn(q, kp, vp, seq, rb, n_sink, W, d, k, 1 / 16)
    assert torch.equal(out, o2) and torch.equal(lse, l2)


def test_tree_bad_ring_base_is_latched():
    n_sink, W, d, k, H_q, H_kv, D = 4, 16, 3, 2, 8, 2, 128
    kp = synth.normal_bf16((40, H_kv, D), 90, DEV)
    q = synth.normal_bf16((1, k * d, H_q, D), 91, DEV)
    seq = torch.tensor([100], dtype=torch.int32, device=DEV)
    rb = torch.tensor([30], dtype=torch.int32, device=DEV)  # ring of 30 slots runs past the pool
    out, lse = wm.tree_draft_attn(q, kp, kp, seq, rb, n_sink, W, d, k, 0.1)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 1


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 8, 2)])
def test_tree_workspace_merges(D, H_q, H_kv):
    # one request, k = 4, d = 7 (224 query rows: two row blocks), more key
    # chunks than a cluster holds: 12, 19 and 37 chunks put the whole grid on
    # the device (every chunk merges its own slice of the outputs; 19 chunks
    # give slices longer than the CTA's threads), 100 do not (the last chunk
    # merges all); against the oracle, and bitwise repeatable
    n_sink, W, d, k = 64, 4096, 7, 4
    S_list = [300_000]
    for n_split in (12, 19, 37, 100):
        out, lse = _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed=900 + n_split, n_split=n_split)
        out2, lse2 = _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed=900 + n_split, n_split=n_split)
        assert torch.equal(out, out2) and torch.equal(lse, lse2), f"split={n_split} not repeatable"


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 8, 2)])
def test_tree_long_chunks(D, H_q, H_kv):
    # chunks of 16 MMA tiles or more (the instance whose gather warps copy K
    # and V rows separately): one chunk, cluster-merged chunks, and 12 / 16
    # chunks merged slice by slice; a request past the window and one inside
    # it (its chunks end early or are empty); sampled rows against the oracle
    n_sink, W, d, k = 64, 16_384, 7, 4
    S_list = [300_000, 9_000]
    n_rows = len(S_list) * k * d * H_q
    rows = np.random.default_rng(D).choice(n_rows, 384, replace=False)
    for n_split in (1, 5, 12, 16):
        _check(S_list, n_sink, W, d, k, H_q, H_kv, D, seed=1300 + n_split, n_split=n_split, rows=rows)
