"""GPU parity of the draft-extend pass (union index table + extend attention)
against the oracle: the table bit-exact, each token's attention within
2e-3 abs + 1e-2 rel of the fp64 attention over its own draft-step table."""
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


def _case(S_list, n_list, n_sink, W, D, H_q, H_kv, windowed, ring, seed, n_q=None, splits=(None,)):
    B = len(S_list)
    n_q = n_q or max(max(n_list), 1)
    scale = 1 / math.sqrt(D)
    d = 7
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    nn = torch.tensor(n_list, dtype=torch.int32, device=DEV)
    if ring:
        R = n_sink + W + d
        rb_list = synth.ring_bases(B, R, B + 1, seed)
        rb = torch.tensor(rb_list, dtype=torch.int32, device=DEV)
        num_slots = (B + 1) * R
        kw = dict(ring_base=rb)
        okw = dict(ring_base=np.array(rb_list, np.int32))
    else:
        ctx = max(S + n for S, n in zip(S_list, n_list)) + 1
        num_slots = B * ctx
        rtt = synth.permutation(num_slots, seed, DEV).view(B, ctx)
        kw = dict(req_to_token=rtt)
        okw = dict(req_to_token=host_i32(rtt))
    kp = synth.normal_bf16((num_slots, H_kv, D), seed + 1, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), seed + 2, DEV)
    q = synth.normal_bf16((B, n_q, H_q, D), seed + 3, DEV)
    stride = None if windowed else (None if not ring else max(S + n for S, n in zip(S_list, n_list)) + 1)
    tab, ln = wm.build_extend_indices(seq, nn, n_sink, W, d, windowed=windowed, stride=stride, **kw)
    otab, oln = oracle.build_extend_indices(np.array(S_list, np.int32), np.array(n_list, np.int32),
                                            n_sink, W, d, windowed=windowed, **okw)
    assert np.array_equal(host_i32(ln), oln)
    for b in range(B):
        assert np.array_equal(host_i32(tab[b, :ln[b]]), otab[b, :oln[b]]), f"table row {b}"
    ro, rl = oracle.draft_extend_attn(bits(q), bits(kp), bits(vp), np.array(S_list, np.int32),
                                      np.array(n_list, np.int32), n_sink, W, scale, windowed=windowed,
                                      depth=d, **okw)
    for n_split in splits:
        out, lse = wm.draft_extend_attn(q, kp, vp, tab, ln, seq, nn, n_sink, W, scale, windowed=windowed,
                                        n_split=n_split)
        assert_attn_close(out, lse, ro, rl, what=f"extend S={S_list} n={n_list} split={n_split}")
        for b, n in enumerate(n_list):
            assert torch.all(out[b, n:] == 0) and torch.all(torch.isneginf(lse[b, n:]))


@pytest.mark.parametrize("ring", [False, True])
@pytest.mark.parametrize("windowed", [True, False])
def test_extend_ragged_batch(ring, windowed):
    # n_sink=64, W=1024: requests inside the sinks, below / across / above the
    # window threshold, and long; ragged counts incl. 0 and 7
    S_list = [10, 1080, 1087, 1090, 5000, 40_000]
    n_list = [3, 7, 2, 0, 5, 1]
    if not windowed and ring:
        S_list = [10, 300, 900]   # a full-context ring table only holds a short context
        n_list = [3, 7, 1]
    _case(S_list, n_list, 64, 1024, 128, 8, 2, windowed, ring, 300 + 10 * ring + windowed,
          splits=(1, 3, 16, 32, 37, None))


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 4, 1)])
def test_extend_shapes_and_small_windows(D, H_q, H_kv):
    _case([0, 4, 9, 25, 300], [7, 5, 7, 4, 6], 4, 9, D, H_q, H_kv, True, False, 400 + D,
          n_q=8, splits=(1, 2, 7, None))


def test_extend_one_token_equals_decode_step():
    D, H_q, H_kv, n_sink, W = 256, 16, 2, 64, 4032
    S = 50_000
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    nn = torch.tensor([1], dtype=torch.int32, device=DEV)
    rtt = synth.permutation(S + 8, 501, DEV).view(1, -1)
    kp = synth.normal_bf16((S + 8, H_kv, D), 502, DEV)
    vp = synth.normal_bf16((S + 8, H_kv, D), 503, DEV)
    q = synth.normal_bf16((1, 1, H_q, D), 504, DEV)
    tab, ln = wm.build_extend_indices(seq, nn, n_sink, W, 7, req_to_token=rtt)
    dt, dl = wm.build_draft_indices(seq, 1, n_sink, W, 7, req_to_token=rtt)
    assert torch.equal(tab[0, :ln[0]], dt[0, 0, :dl[0, 0]])
    a = wm.draft_extend_attn(q, kp, vp, tab, ln, seq, nn, n_sink, W, 1 / 16, n_split=16)
    b = wm.draft_decode_attn(q, kp, vp, dt[0], dl[0], 1 / 16, n_split=16)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("windowed", [True, False])
def test_extend_split_counts_and_fallback(windowed):
    # one-read-per-request launch (rows of >= 1024 keys per split) at 1..8
    # splits; 16+ splits of these rows, 129 splits and n_q = 9 take the
    # per-token launch; all within tolerance of the oracle
    _case([3000, 9000], [5, 2], 64, 1024, 256, 16, 2, windowed, False, 620 + windowed, n_q=6,
          splits=(1, 3, 8, 16, 40, 128, 129))
    _case([70_000, 200_000], [7, 3], 64, 4032, 256, 16, 2, windowed, False, 640 + windowed, n_q=8,
          splits=(None, 100, 128))
    _case([2000], [9], 64, 512, 128, 8, 2, windowed, True, 630 + windowed, n_q=9, splits=(None, 3))


@pytest.mark.parametrize("n_q,n_list", [(3, [3, 1, 2]), (8, [8, 5, 0])])
def test_extend_one_read_head_dim_128(n_q, n_list):
    # long rows take the one-read launch at D = 128 as well (G = 4 heads)
    _case([20_000, 45_000, 9_000], n_list, 64, 1024, 128, 8, 2, False, False, 660 + n_q, n_q=n_q,
          splits=(None, 2, 9))


@pytest.mark.parametrize("windowed,D,H_q,H_kv", [(False, 128, 8, 2), (True, 256, 16, 2)])
def test_extend_tensor_core_path_long_rows(windowed, D, H_q, H_kv):
    # union rows of >= 65536 keys take the tensor-core launch (a request's
    # tokens as one MMA row block over each union key once): one split,
    # cluster merges, workspace merges, a request without new tokens, the
    # ragged tail; the windowed union holds n_sink + W + n - 1 keys
    W = 65_536 if windowed else 1024
    _case([70_001, 150_000, 99_999], [5, 0, 2], 64, W, D, H_q, H_kv, windowed, False, 680 + windowed,
          n_q=5, splits=(None, 1, 4, 8, 100))


def test_extend_tensor_core_path_wrong_union_length_is_latched():
    # a union length that is not the keep set of S + n is latched
    # (WMTP_DEV_LEN_RANGE) on the tensor-core path; the launch reads no entry
    # past the table row and the outputs stay finite
    S, n, n_sink, W, H_q, H_kv, D = 80_000, 3, 64, 1024, 8, 2, 128
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    nn = torch.tensor([n], dtype=torch.int32, device=DEV)
    rtt = synth.permutation(S + 8, 690, DEV).view(1, -1)
    kp = synth.normal_bf16((S + 8, H_kv, D), 691, DEV)
    vp = synth.normal_bf16((S + 8, H_kv, D), 692, DEV)
    q = synth.normal_bf16((1, n, H_q, D), 693, DEV)
    tab, ln = wm.build_extend_indices(seq, nn, n_sink, W, 7, windowed=False, req_to_token=rtt)
    assert tab.shape[-1] >= 65_536 and int(ln[0]) == S + n
    wm.device_error(clear=True)
    out, lse = wm.draft_extend_attn(q, kp, vp, tab, ln - 1, seq, nn, n_sink, W, 0.1, windowed=False,
                                    n_split=16)
    torch.cuda.synchronize()
    assert wm.device_error(clear=True) == 3  # WMTP_DEV_LEN_RANGE
    assert torch.all(torch.isfinite(out))


def test_extend_tensor_core_path_ring_layout():
    # a windowed union of n_sink + W + n - 1 >= 65536 keys over per-request
    # rings: the union row's slots run consecutively, so the tensor-core
    # launch brings them in as TMA boxes (runs of 32 and 8 slots, the ring
    # wrap and the sink seam by cp.async)
    _case([70_001, 150_000, 99_999], [5, 0, 2], 64, 65_536, 256, 16, 2, True, True, 700,
          n_q=5, splits=(None, 1, 8, 100))
