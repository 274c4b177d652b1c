"""The attention entry point that allocates nothing.

Some callers cannot give the library a workspace: an engine that has reserved
nearly all device memory for its KV pool behind its own allocator (where a
cudaMalloc fails or stalls the device), or a plugin boundary that passes only
input and output pointers.  For them wmtp_draft_decode_attn_noalloc merges the
split partials in a fixed scratch array that the library keeps on the device.

These tests call it through the C ABI (and once through the Python binding)
and check it against the regular entry point, which uses a caller-provided
workspace, on several calls in a row with different shapes, so that each call
runs on scratch left over by the one before.  The no-workspace call always
merges through the scratch with the "last CTA merges" path; where the regular
call takes that same path -- more splits than one cluster holds in a grid
larger than the device holds at once, or no cluster plan that fits -- the two
must agree bit for bit.  Where the regular call merges through a thread-block
cluster, they must agree within the attention tolerance of the other parity
tests.  One
case is also checked against the fp64 oracle.  The file is named to be
collected last.
"""
import ctypes
import math

import pytest
import torch

import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import synth

NULL = None
P = ctypes.c_void_p(256)  # never dereferenced: the call below fails validation first

# Largest split count whose partials fit the scratch at B=1, n_q=1, H_q=16,
# D=256: the counter region takes WMTP_NOALLOC_MAX_COUNTERS * 4 bytes, the
# lse partials 16 * n_split floats (rounded up to 256 bytes) and the output
# partials 16 * n_split * 256 floats.
SCRATCH = 8 << 20
COUNTERS = 4096


def _partials(rows_q, D, n_split):
    return (rows_q * n_split * 4 + 255) // 256 * 256 + rows_q * n_split * D * 4


LIMIT_SPLITS = max(n for n in range(1, 1025) if _partials(16, 256, n) <= SCRATCH - COUNTERS * 4)


def test_scratch_limit_arithmetic():
    assert LIMIT_SPLITS == 509
    assert _partials(16, 256, 509) == SCRATCH - COUNTERS * 4  # exactly full


def test_noalloc_rejects_oversized_scratch():
    wm.build()
    lib = wm.load()
    # 64 requests x 16 heads x 1024 splits x 256 dims of fp32 partials is far
    # beyond the fixed scratch; rejected before anything is launched.
    st = lib.wmtp_draft_decode_attn_noalloc(P, 64, 1, 16, 2, 256, P, P, 10, P, 10, P, 0.1, P, NULL,
                                            1024, NULL)
    assert st == wm.WMTP_ECAPACITY
    # more merge counters than the scratch reserves
    st = lib.wmtp_draft_decode_attn_noalloc(P, 4097, 1, 2, 1, 128, P, P, 10, P, 10, P, 0.1, P, NULL,
                                            2, NULL)
    assert st == wm.WMTP_ECAPACITY
    # one split past the partials limit
    st = lib.wmtp_draft_decode_attn_noalloc(P, 1, 1, 16, 2, 256, P, P, 10, P, 10, P, 0.1, P, NULL,
                                            LIMIT_SPLITS + 1, NULL)
    assert st == wm.WMTP_ECAPACITY


def test_noalloc_binding_checks_shapes():
    """Mismatched pools, a short table or lens, or outputs of the wrong shape
    are refused by the binding before the library is called (checked on
    host tensors: the shape checks come first)."""
    q = torch.zeros((2, 1, 16, 128), dtype=torch.bfloat16)
    kp = torch.zeros((50, 2, 128), dtype=torch.bfloat16)
    table = torch.zeros((2, 40), dtype=torch.int32)
    lens = torch.zeros((2,), dtype=torch.int32)
    out = torch.zeros((2, 1, 16, 128))
    lse = torch.zeros((2, 1, 16))
    f = wm.draft_decode_attn_noalloc
    with pytest.raises(ValueError, match="v_pool shape"):
        f(q, kp, torch.zeros((49, 2, 128), dtype=torch.bfloat16), table, lens, 0.1, out, lse, 2)
    with pytest.raises(ValueError, match="head dim"):
        f(q, torch.zeros((50, 2, 256), dtype=torch.bfloat16), torch.zeros((50, 2, 256), dtype=torch.bfloat16),
          table, lens, 0.1, out, lse, 2)
    with pytest.raises(ValueError, match="smaller than B rows"):
        f(q, kp, kp, table[:1], lens, 0.1, out, lse, 2)
    with pytest.raises(ValueError, match="smaller than B rows"):
        f(q, kp, kp, table, lens[:1], 0.1, out, lse, 2)
    with pytest.raises(ValueError, match="out shape"):
        f(q, kp, kp, table, lens, 0.1, out[:1], lse, 2)
    with pytest.raises(ValueError, match="lse shape"):
        f(q, kp, kp, table, lens, 0.1, out, lse[:, :, :8], 2)
    with pytest.raises(ValueError, match="must be passed in"):
        f(q, kp, kp, table, lens, 0.1, None, lse, 2)
    # the regular entry point makes the same checks on outputs it is given
    with pytest.raises(ValueError, match="out shape"):
        wm.draft_decode_attn(q, kp, kp, table, lens, 0.1, out=out[:, :, :8])


def _call_c_abi(lib, q, kp, vp, table, lens, scale, out, lse, n_split):
    B, n_q, H_q, D = q.shape
    num_slots, H_kv, _ = kp.shape
    st = lib.wmtp_draft_decode_attn_noalloc(
        ctypes.c_void_p(q.data_ptr()), B, n_q, H_q, H_kv, D, ctypes.c_void_p(kp.data_ptr()),
        ctypes.c_void_p(vp.data_ptr()), num_slots, ctypes.c_void_p(table.data_ptr()),
        table.shape[-1], ctypes.c_void_p(lens.data_ptr()), float(scale),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()), n_split,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == wm.WMTP_OK, st


def _inputs(B, H_q, H_kv, D, L, pool, seed, dev):
    kp = synth.normal_bf16((pool, H_kv, D), seed, dev)
    vp = synth.normal_bf16((pool, H_kv, D), seed + 1, dev)
    q = synth.normal_bf16((B, 1, H_q, D), seed + 2, dev)
    table = torch.stack([synth.permutation(pool, seed + 3 + b, dev)[:L] for b in range(B)])
    lens = torch.tensor([L - 37 * (b % 3) for b in range(B)], dtype=torch.int32, device=dev)
    return kp, vp, q, table.contiguous(), lens


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    wm.build()
    lib = wm.load()
    dev = torch.device("cuda:0")
    cases = [
        # (B, H_q, H_kv, D, keys, pool, n_split, bit-exact expected)
        (2, 16, 2, 256, 20_000, 20_000, 9, False),   # regular call merges in a cluster of 9
        (12, 8, 2, 128, 7_000, 7_000, 37, True),     # 888 CTAs, more than the device holds at once
        (1, 16, 2, 256, LIMIT_SPLITS * 64, LIMIT_SPLITS * 64, LIMIT_SPLITS, True),  # scratch exactly full, 1018 CTAs
        (COUNTERS // 2, 2, 2, 128, 130, 5_000, 2, True),  # WMTP_NOALLOC_MAX_COUNTERS merge counters
        (2, 16, 2, 256, 3_000, 3_000, 1, True),      # one split: no scratch at all
        (12, 8, 2, 128, 7_000, 7_000, 37, True),     # repeat: leftover counters and partials
    ]
    for i, (B, H_q, H_kv, D, L, pool, n_split, exact) in enumerate(cases):
        kp, vp, q, table, lens = _inputs(B, H_q, H_kv, D, L, pool, 500 + 10 * i, dev)
        scale = 1 / math.sqrt(D)
        ref_out, ref_lse = wm.draft_decode_attn(q, kp, vp, table, lens, scale, n_split=n_split)
        out = torch.full((B, 1, H_q, D), float("nan"), device=dev)
        lse = torch.full((B, 1, H_q), float("nan"), device=dev)
        _call_c_abi(lib, q, kp, vp, table, lens, scale, out, lse, n_split)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all(), f"case {i}"
        if exact:
            assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), f"case {i}: not bit-identical"
        else:
            torch.testing.assert_close(out, ref_out, atol=2e-3, rtol=1e-2)
            torch.testing.assert_close(lse, ref_lse, atol=2e-3, rtol=1e-2)
    assert wm.device_error(clear=True) == 0


@pytest.mark.gpu
def test_noalloc_binding_matches_oracle():
    """The Python binding of the same call, twice in a row, against the fp64
    oracle over a row whose split plan leaves some splits empty."""
    import oracle
    from wmtp_testutil import assert_attn_close, bits, host_i32

    wm.build()
    dev = torch.device("cuda:0")
    B, H_q, H_kv, D, L, n_split = 2, 16, 2, 256, 3_000, 37
    kp, vp, q, table, lens = _inputs(B, H_q, H_kv, D, L, L, 900, dev)
    scale = 1 / math.sqrt(D)
    ref, ref_lse = oracle.draft_decode_attn(bits(q), bits(kp), bits(vp), host_i32(table), host_i32(lens), scale)
    for _ in range(2):
        out = torch.full((B, 1, H_q, D), float("nan"), device=dev)
        lse = torch.full((B, 1, H_q), float("nan"), device=dev)
        wm.draft_decode_attn_noalloc(q, kp, vp, table, lens, scale, out, lse, n_split)
        torch.cuda.synchronize()
        assert_attn_close(out, lse, ref, ref_lse, what="noalloc vs oracle")
    assert wm.device_error(clear=True) == 0
