"""The attention entry point that allocates nothing.

Some callers cannot give the library a workspace: an engine that has reserved
nearly all device memory for its KV pool behind its own allocator (where a
cudaMalloc fails or stalls the device), or a plugin boundary that passes only
input and output pointers.  For them wmtp_draft_decode_attn_noalloc merges the
split partials in a fixed scratch array that the library keeps on the device.

These tests call it through the C ABI and check it against the regular entry
point (which uses a caller-provided workspace) within the attention tolerance
of the other parity tests, on two calls in a row with different shapes, so
that the second call runs on scratch left over by the first.  The file is
named to be collected last.
"""
import ctypes
import math

import pytest
import torch

import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import synth

NULL = None
P = ctypes.c_void_p(256)  # never dereferenced: the call below fails validation first


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


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice():
    wm.build()
    lib = wm.load()
    dev = torch.device("cuda:0")
    cases = [
        # (B, H_q, H_kv, D, keys, n_split): merge through the scratch in both
        (2, 16, 2, 256, 20_000, 9),
        (3, 8, 2, 128, 7_000, 40),
    ]
    for i, (B, H_q, H_kv, D, L, n_split) in enumerate(cases):
        kp = synth.normal_bf16((L, H_kv, D), 500 + i, dev)
        vp = synth.normal_bf16((L, H_kv, D), 510 + i, dev)
        q = synth.normal_bf16((B, 1, H_q, D), 520 + i, dev)
        table = torch.stack([synth.permutation(L, 530 + i + b, dev) for b in range(B)])
        lens = torch.tensor([L - 37 * b for b in range(B)], dtype=torch.int32, device=dev)
        scale = 1 / math.sqrt(D)
        ref_out, ref_lse = wm.draft_decode_attn(q, kp, vp, table, lens, scale, n_split=n_split)
        out = torch.full((B, 1, H_q, D), float("nan"), device=dev)
        lse = torch.full((B, 1, H_q), float("nan"), device=dev)
        _call_c_abi(lib, q, kp, vp, table, lens, scale, out, lse, n_split)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        torch.testing.assert_close(out, ref_out, atol=2e-3, rtol=1e-2)
        torch.testing.assert_close(lse, ref_lse, atol=2e-3, rtol=1e-2)
    assert wm.device_error(clear=True) == 0
