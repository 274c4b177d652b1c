"""Shared helpers for the parity tests: tensor <-> oracle marshalling and the
attention tolerance.

Tolerance for fp32 attention outputs against the fp64 oracle, bf16 K/V: every
element must satisfy |gpu - ref| <= 2e-3 + 1e-2 * |ref| (2e-3 absolute /
1e-2 relative).  Because long rows give outputs far below 2e-3 in
magnitude, the tests also require max |gpu - ref| <= 1e-2 * max |ref| over
each query row, which keeps the check meaningful at any output scale.
"""
from __future__ import annotations

import numpy as np
import torch

ATOL = 2e-3
RTOL = 1e-2
ROW_RTOL = 1e-2


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.int32, copy=False)


def assert_attn_close(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what=""):
    """Compare GPU fp32 attention with the fp64 oracle.

    out_*: [..., D]; lse_*: [...]; ``rows`` selects flattened query rows
    (others are NaN in the oracle output)."""
    og = out_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(-1, out_gpu.shape[-1])
    lg = lse_gpu.detach().float().cpu().numpy().astype(np.float64).reshape(-1)
    orf = np.asarray(out_ref, np.float64).reshape(-1, og.shape[-1])
    lrf = np.asarray(lse_ref, np.float64).reshape(-1)
    if rows is not None:
        rows = np.asarray(rows)
        og, lg, orf, lrf = og[rows], lg[rows], orf[rows], lrf[rows]
    assert np.all(np.isfinite(og)), f"{what}: non-finite GPU output"
    err = np.abs(og - orf)
    bound = ATOL + RTOL * np.abs(orf)
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {bad.size} elements outside 2e-3 abs + 1e-2 rel; "
        f"max abs err {err.max():.3e}, worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    row_scale = np.abs(orf).max(axis=1)
    row_err = err.max(axis=1)
    ok_rows = row_err <= ROW_RTOL * row_scale + 1e-30
    assert ok_rows.all(), (
        f"{what}: row-relative error {np.max(row_err / np.maximum(row_scale, 1e-30)):.3e} > {ROW_RTOL}")
    fin = np.isfinite(lrf)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lrf)), f"{what}: -inf lse mismatch"
    lerr = np.abs(lg[fin] - lrf[fin])
    assert np.all(lerr <= ATOL + RTOL * np.abs(lrf[fin])), f"{what}: lse max err {lerr.max():.3e}"
    return float(err.max()), float(np.max(row_err / np.maximum(row_scale, 1e-30)))
