"""GB300 (sm_103a) library for the Windowed-MTP draft-attention hot path.

Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
Context" (arXiv 2607.21535).  The compute runs in the CUDA library
``_lib/libwmtp.so`` (C ABI: ``include/wmtp.h``).  This module only marshals
torch tensors into pointers, sizes and the current CUDA stream; it performs no
arithmetic of the method and has no CPU fallback: if the library is missing it
raises.

Calls (same names as the C ABI without the ``wmtp_`` prefix):
  build_draft_indices  draft KV-index tables (sink + window, or full context)
  ring_map             logical position -> ring slot
  append_kv            write draft K/V rows into the pool
  draft_decode_attn    split-KV flash-decode attention with LSE merge
  draft_decode_attn_append  append_kv + draft_decode_attn in one launch
  build_extend_indices / draft_extend_attn  the draft forward over a request's
                       accepted tokens in one launch (each token its own keys)
  build_far_indices    the far-key tables (positions the keep rule drops)
  attn_mass_diagnostics  in-window mass, win_perturb, tail out-frac per query,
                       from the windowed and the far-key attention
  append_kv_fp8 / draft_decode_attn_fp8  the same over E4M3 KV pools with
                       per-KV-head scales
  prefill_keep_positions / ring_fill  pruned draft prefill: the kept prompt
                       positions and their KV written into the ring
  draft_decode_attn_ring  a draft step over the ring with no table (slots
                       from the ring rule in the kernel), append fused
  (overlap_hold=...)   draft_decode_attn_append / draft_decode_attn_ring as
                       chained steps (``*_overlap`` in the C ABI): copies of
                       every key but the last few start while the previous
                       step on the stream finishes; the same bits
  draft_decode_attn_noalloc  the attention without a caller workspace
  tree_draft_attn      tree-draft attention over the ring (tree-causal mask)
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

from . import _build

__all__ = [
    "WmtpError", "load", "build", "version", "device_error",
    "build_draft_indices", "build_extend_indices", "build_far_indices", "ring_map", "append_kv", "draft_decode_attn",
    "draft_decode_attn_append", "draft_extend_attn", "attn_mass_diagnostics",
    "attn_workspace_bytes", "attn_num_splits", "extend_num_splits", "AttnWorkspace", "draft_decode_attn_noalloc",
    "tree_draft_attn", "tree_workspace_bytes", "tree_num_splits",
    "append_kv_fp8", "draft_decode_attn_fp8", "prefill_keep_positions", "ring_fill",
    "draft_decode_attn_ring",
]

WMTP_OK = 0
WMTP_EINVAL = -1
WMTP_ECAPACITY = -2
WMTP_ECUDA = -3
WMTP_EDEVICE = -4

DEV_ERRORS = {0: "ok", 1: "slot out of range", 2: "table overflow", 3: "lens out of range",
              4: "pipeline wait timeout", 5: "device argument out of range"}


class WmtpError(RuntimeError):
    def __init__(self, what: str, status: int):
        super().__init__(f"{what}: status {status} ({_STATUS.get(status, 'unknown')})")
        self.status = status


_STATUS = {WMTP_OK: "ok", WMTP_EINVAL: "invalid argument", WMTP_ECAPACITY: "capacity",
           WMTP_ECUDA: "CUDA error", WMTP_EDEVICE: "device check failed"}

_lock = threading.Lock()
_lib = None
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libwmtp.so`` for sm_103a (nvcc) if it is missing or stale."""
    return _build.build(force=force, verbose=verbose)


def load():
    """Load the CUDA library; raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise ImportError(f"libwmtp.so is not built ({path}); run "
                              "speculative_decoding_draft_build_gb300.build()")
        lib = ctypes.CDLL(path)
        lib.wmtp_version.restype = _i32
        lib.wmtp_status_string.restype = ctypes.c_char_p
        lib.wmtp_status_string.argtypes = [_i32]
        lib.wmtp_get_device_error.restype = _i32
        lib.wmtp_get_device_error.argtypes = [ctypes.POINTER(_i32), _i32]
        lib.wmtp_build_draft_indices.restype = _i32
        lib.wmtp_build_draft_indices.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp]
        lib.wmtp_build_extend_indices.restype = _i32
        lib.wmtp_build_extend_indices.argtypes = [
            _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i64, _vp, _vp]
        lib.wmtp_draft_extend_attn.restype = _i32
        lib.wmtp_draft_extend_attn.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _i32,
            _i32, ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_attn_mass_diagnostics.restype = _i32
        lib.wmtp_attn_mass_diagnostics.argtypes = [_vp, _vp, _vp, _vp, _i64, _i32, _vp, _vp, _vp, _vp,
                                                   _vp, _vp]
        lib.wmtp_build_far_indices.restype = _i32
        lib.wmtp_build_far_indices.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64,
                                               _vp, _vp]
        lib.wmtp_ring_map.restype = _i32
        lib.wmtp_ring_map.argtypes = [_vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp]
        lib.wmtp_append_kv.restype = _i32
        lib.wmtp_append_kv.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _i64, _vp]
        lib.wmtp_attn_workspace_bytes.restype = ctypes.c_size_t
        lib.wmtp_attn_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
        lib.wmtp_attn_workspace_init.restype = _i32
        lib.wmtp_attn_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
        lib.wmtp_attn_num_splits.restype = _i32
        lib.wmtp_attn_num_splits.argtypes = [_i32, _i32, _i32, _i64]
        lib.wmtp_draft_decode_attn.restype = _i32
        lib.wmtp_draft_decode_attn.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, ctypes.c_float,
            _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_draft_decode_attn_append.restype = _i32
        lib.wmtp_draft_decode_attn_append.argtypes = [
            _vp, _vp, _vp, _i32,
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, ctypes.c_float,
            _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_draft_decode_attn_append_overlap.restype = _i32
        lib.wmtp_draft_decode_attn_append_overlap.argtypes = [
            _vp, _vp, _vp, _i32,
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, ctypes.c_float,
            _vp, _vp, _vp, ctypes.c_size_t, _i32, _i32, _vp]
        lib.wmtp_tree_workspace_bytes.restype = ctypes.c_size_t
        lib.wmtp_tree_workspace_bytes.argtypes = [_i32] * 7
        lib.wmtp_tree_num_splits.restype = _i32
        lib.wmtp_tree_num_splits.argtypes = [_i32] * 7
        lib.wmtp_tree_draft_attn.restype = _i32
        lib.wmtp_tree_draft_attn.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32,
            ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_append_kv_fp8.restype = _i32
        lib.wmtp_append_kv_fp8.argtypes = [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64,
                                           _vp]
        lib.wmtp_extend_num_splits.restype = _i32
        lib.wmtp_extend_num_splits.argtypes = [_i32, _i32, _i32, _i64]
        lib.wmtp_attn_num_splits_fp8.restype = _i32
        lib.wmtp_attn_num_splits_fp8.argtypes = [_i32, _i32, _i32, _i64]
        lib.wmtp_draft_decode_attn_fp8.restype = _i32
        lib.wmtp_draft_decode_attn_fp8.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _i64, _vp,
            ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_prefill_keep_positions.restype = _i32
        lib.wmtp_prefill_keep_positions.argtypes = [_vp, _i32, _i32, _i32, _vp, _i64, _vp, _vp]
        lib.wmtp_ring_fill.restype = _i32
        lib.wmtp_ring_fill.argtypes = [_vp, _vp, _vp, _i32, _i64, _i32, _i32, _vp, _i32, _i32, _i32, _i32,
                                       _vp, _vp, _i64, _vp]
        lib.wmtp_draft_decode_attn_ring.restype = _i32
        lib.wmtp_draft_decode_attn_ring.argtypes = [
            _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _i32, _vp]
        lib.wmtp_draft_decode_attn_ring_overlap.restype = _i32
        lib.wmtp_draft_decode_attn_ring_overlap.argtypes = [
            _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
            ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _i32, _i32, _vp]
        lib.wmtp_draft_decode_attn_noalloc.restype = _i32
        lib.wmtp_draft_decode_attn_noalloc.argtypes = [
            _vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _i64, _vp, _i64, _vp, ctypes.c_float,
            _vp, _vp, _i32, _vp]
        _lib = lib
        return lib


def version() -> int:
    return int(load().wmtp_version())


def _check(status: int, what: str) -> None:
    if status != WMTP_OK:
        raise WmtpError(what, int(status))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on(dev):
    """Make `dev` the current CUDA device for a library call (the library
    keeps per-device state); a no-op when it already is."""
    idx = dev.index if isinstance(dev, torch.device) else int(dev)
    if idx is None or idx == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(idx)


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, device=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def device_error(clear: bool = True) -> int:
    """Device-side error code latched by the kernels (0 = none). Synchronises."""
    code = _i32(0)
    _check(load().wmtp_get_device_error(ctypes.byref(code), int(clear)), "get_device_error")
    return int(code.value)


# ---------------------------------------------------------------- a1
def build_draft_indices(seq_lens: torch.Tensor, gamma: int, n_sink: int, window: int,
                        depth: int, tree_k: int = 1, windowed: bool = True,
                        req_to_token: torch.Tensor | None = None,
                        req_pool_idx: torch.Tensor | None = None,
                        ring_base: torch.Tensor | None = None, stride: int | None = None,
                        table: torch.Tensor | None = None, lens: torch.Tensor | None = None,
                        stream=None):
    """Draft KV-index tables for ``gamma`` draft steps (``wmtp_build_draft_indices``).

    Returns ``(table[gamma, B, stride] int32, lens[gamma, B] int32)``.  When
    ``stride`` is omitted it is ``n_sink + window`` (windowed) or
    ``req_to_token.shape[1]`` (full, paged layout).
    """
    _need(seq_lens, "seq_lens", torch.int32)
    dev = seq_lens.device
    B = seq_lens.shape[0]
    if req_to_token is not None:
        _need(req_to_token, "req_to_token", torch.int32, dev)
        if req_pool_idx is not None:
            _need(req_pool_idx, "req_pool_idx", torch.int32, dev)
    if ring_base is not None:
        _need(ring_base, "ring_base", torch.int32, dev)
    if stride is None:
        if table is not None:
            stride = table.shape[-1]
        elif windowed:
            stride = n_sink + window
        elif req_to_token is not None:
            stride = req_to_token.shape[1]
        else:
            raise ValueError("stride is required for a full-context ring table")
    if table is None:
        table = torch.empty((gamma, B, stride), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((gamma, B), dtype=torch.int32, device=dev)
    _need(table, "table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev)
    rtt_stride = req_to_token.shape[1] if req_to_token is not None else 0
    with _on(dev):
        _check(load().wmtp_build_draft_indices(
            _ptr(seq_lens), B, gamma, n_sink, window, depth, tree_k, int(bool(windowed)),
            _ptr(req_to_token), _ptr(req_pool_idx), rtt_stride, _ptr(ring_base), _ptr(table),
            stride, _ptr(lens), _stream(stream)), "build_draft_indices")
    return table, lens


def build_far_indices(seq_lens: torch.Tensor, gamma: int, n_sink: int, window: int,
                      req_to_token: torch.Tensor, req_pool_idx: torch.Tensor | None = None,
                      stride: int | None = None, table: torch.Tensor | None = None,
                      lens: torch.Tensor | None = None, stream=None):
    """Far-key tables (``wmtp_build_far_indices``): per draft step j, the
    positions [n_sink, kv_len - W) the keep rule drops (none while kv_len <=
    n_sink + W), through ``req_to_token``.  Returns ``(table[gamma, B,
    stride], lens[gamma, B])``; ``stride`` defaults to ``req_to_token.shape[1]``."""
    _need(seq_lens, "seq_lens", torch.int32)
    dev = seq_lens.device
    B = seq_lens.shape[0]
    _need(req_to_token, "req_to_token", torch.int32, dev)
    if req_pool_idx is not None:
        _need(req_pool_idx, "req_pool_idx", torch.int32, dev)
    if stride is None:
        stride = table.shape[-1] if table is not None else req_to_token.shape[1]
    if table is None:
        table = torch.empty((gamma, B, stride), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((gamma, B), dtype=torch.int32, device=dev)
    _need(table, "table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev)
    if table.numel() < gamma * B * stride or lens.numel() < gamma * B:
        raise ValueError("build_far_indices: table/lens smaller than gamma * B rows")
    with _on(dev):
        _check(load().wmtp_build_far_indices(
            _ptr(seq_lens), B, gamma, n_sink, window, _ptr(req_to_token), _ptr(req_pool_idx),
            req_to_token.shape[1], _ptr(table), stride, _ptr(lens), _stream(stream)), "build_far_indices")
    return table, lens


def build_extend_indices(seq_lens: torch.Tensor, n_new: torch.Tensor, n_sink: int, window: int,
                         depth: int, tree_k: int = 1, windowed: bool = True,
                         req_to_token: torch.Tensor | None = None,
                         req_pool_idx: torch.Tensor | None = None,
                         ring_base: torch.Tensor | None = None, stride: int | None = None,
                         table: torch.Tensor | None = None, lens: torch.Tensor | None = None,
                         stream=None):
    """Union index table of a draft-extend pass (``wmtp_build_extend_indices``).

    Returns ``(table[B, stride] int32, lens[B] int32)``.  When ``stride`` is
    omitted it is ``n_sink + window + max_new - 1`` with ``max_new`` =
    ``n_new.max()`` (windowed), or ``req_to_token.shape[1]`` (full, paged).
    """
    _need(seq_lens, "seq_lens", torch.int32)
    dev = seq_lens.device
    _need(n_new, "n_new", torch.int32, dev)
    B = seq_lens.shape[0]
    if req_to_token is not None:
        _need(req_to_token, "req_to_token", torch.int32, dev)
        if req_pool_idx is not None:
            _need(req_pool_idx, "req_pool_idx", torch.int32, dev)
    if ring_base is not None:
        _need(ring_base, "ring_base", torch.int32, dev)
    if stride is None:
        if table is not None:
            stride = table.shape[-1]
        elif windowed:
            stride = n_sink + window + max(int(n_new.max().item()) if B else 1, 1) - 1
        elif req_to_token is not None:
            stride = req_to_token.shape[1]
        else:
            raise ValueError("stride is required for a full-context ring table")
    if table is None:
        table = torch.empty((B, stride), dtype=torch.int32, device=dev)
    if lens is None:
        lens = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(table, "table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev)
    rtt_stride = req_to_token.shape[1] if req_to_token is not None else 0
    with _on(dev):
        _check(load().wmtp_build_extend_indices(
            _ptr(seq_lens), _ptr(n_new), B, n_sink, window, depth, tree_k, int(bool(windowed)),
            _ptr(req_to_token), _ptr(req_pool_idx), rtt_stride, _ptr(ring_base), _ptr(table),
            stride, _ptr(lens), _stream(stream)), "build_extend_indices")
    return table, lens


# ---------------------------------------------------------------- a2
def ring_map(ring_base: torch.Tensor, pos: torch.Tensor, req_of: torch.Tensor, n_sink: int,
             window: int, depth: int, tree_k: int = 1, branch: torch.Tensor | None = None,
             slots: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Ring slots of logical positions (``wmtp_ring_map``)."""
    _need(ring_base, "ring_base", torch.int32)
    dev = ring_base.device
    _need(pos, "pos", torch.int32, dev)
    _need(req_of, "req_of", torch.int32, dev)
    if branch is not None:
        _need(branch, "branch", torch.int32, dev)
    n = pos.numel()
    if slots is None:
        slots = torch.empty(n, dtype=torch.int32, device=dev)
    _need(slots, "slots", torch.int32, dev)
    with _on(dev):
        _check(load().wmtp_ring_map(_ptr(ring_base), _ptr(pos), _ptr(branch), _ptr(req_of), n,
                                    n_sink, window, depth, tree_k, _ptr(slots), _stream(stream)),
               "ring_map")
    return slots


def append_kv(k_new: torch.Tensor, v_new: torch.Tensor, slots: torch.Tensor,
              k_pool: torch.Tensor, v_pool: torch.Tensor, stream=None) -> None:
    """Write each new token's K/V rows into pool slot ``slots[i]`` (``wmtp_append_kv``)."""
    _need(k_pool, "k_pool", torch.bfloat16)
    dev = k_pool.device
    for t, nm in ((v_pool, "v_pool"), (k_new, "k_new"), (v_new, "v_new")):
        _need(t, nm, torch.bfloat16, dev)
    _need(slots, "slots", torch.int32, dev)
    n, H_kv, D = k_new.shape
    if v_new.shape != k_new.shape or k_pool.shape[1:] != (H_kv, D) or v_pool.shape != k_pool.shape:
        raise ValueError("append_kv: shape mismatch")
    with _on(dev):
        _check(load().wmtp_append_kv(_ptr(k_new), _ptr(v_new), _ptr(slots), n, H_kv, D,
                                     _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _stream(stream)),
               "append_kv")


def append_kv_fp8(k_new: torch.Tensor, v_new: torch.Tensor, slots: torch.Tensor,
                  k_scale: torch.Tensor, v_scale: torch.Tensor, k_pool: torch.Tensor,
                  v_pool: torch.Tensor, stream=None) -> None:
    """Quantise each new token's bf16 K/V rows to E4M3 codes with the per-KV-head
    scales and write them to pool slot ``slots[i]`` (``wmtp_append_kv_fp8``).
    k_new/v_new: [n, H_kv, D] bf16; k_scale/v_scale: [H_kv] fp32; pools:
    [num_slots, H_kv, D] uint8."""
    _need(k_pool, "k_pool", torch.uint8)
    dev = k_pool.device
    _need(v_pool, "v_pool", torch.uint8, dev)
    for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, nm, torch.bfloat16, dev)
    for t, nm in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, nm, torch.float32, dev)
    _need(slots, "slots", torch.int32, dev)
    n, H_kv, D = k_new.shape
    if (v_new.shape != k_new.shape or k_pool.shape[1:] != (H_kv, D) or v_pool.shape != k_pool.shape
            or k_scale.numel() != H_kv or v_scale.numel() != H_kv or slots.numel() != n):
        raise ValueError("append_kv_fp8: shape mismatch")
    with _on(dev):
        _check(load().wmtp_append_kv_fp8(_ptr(k_new), _ptr(v_new), _ptr(slots), n, H_kv, D,
                                         _ptr(k_scale), _ptr(v_scale), _ptr(k_pool), _ptr(v_pool),
                                         k_pool.shape[0], _stream(stream)), "append_kv_fp8")


# ---------------------------------------------------------------- a3 + a4
def attn_workspace_bytes(B: int, n_q: int, H_q: int, H_kv: int, D: int, n_split: int) -> int:
    return int(load().wmtp_attn_workspace_bytes(B, n_q, H_q, H_kv, D, n_split))


def attn_num_splits(B: int, n_q: int, H_kv: int, max_len: int, device=None, fp8: bool = False) -> int:
    dev = device if device is not None else torch.cuda.current_device()
    fn = load().wmtp_attn_num_splits_fp8 if fp8 else load().wmtp_attn_num_splits
    with _on(dev):
        return int(fn(B, n_q, H_kv, int(max_len)))


def extend_num_splits(B: int, n_q: int, H_kv: int, max_len: int, device=None) -> int:
    """Usual split count of :func:`draft_extend_attn` (``wmtp_extend_num_splits``)."""
    dev = device if device is not None else torch.cuda.current_device()
    with _on(dev):
        return int(load().wmtp_extend_num_splits(B, n_q, H_kv, int(max_len)))


class AttnWorkspace:
    """Device scratch for the split-KV partials, zeroed once at creation.

    Every completed ``draft_decode_attn`` call leaves the merge counters at
    zero, so one workspace serves any number of calls (not concurrent ones).
    A CUDA graph that captured a call keeps the workspace's address: keep the
    object alive as long as the graph (``torch.cuda.graph`` empties the
    allocator cache when a capture starts, so a dropped workspace can be
    unmapped before the replay).
    """

    def __init__(self, nbytes: int, device, stream=None):
        self.nbytes = int(nbytes)
        self.buf = torch.empty(max(self.nbytes, 256), dtype=torch.uint8, device=device)
        with _on(self.buf.device):
            _check(load().wmtp_attn_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)),
                   "attn_workspace_init")

    def ensure(self, nbytes: int, stream=None) -> "AttnWorkspace":
        if nbytes <= self.nbytes:
            return self
        return AttnWorkspace(nbytes, self.buf.device, stream)


_ws_cache: dict = {}


def draft_decode_attn(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                      table: torch.Tensor, lens: torch.Tensor, scale: float,
                      out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      n_split: int | None = None, max_len: int | None = None,
                      workspace: AttnWorkspace | None = None, stream=None):
    """Split-KV flash-decode attention over a block table (``wmtp_draft_decode_attn``).

    q: [B, n_q, H_q, D] bf16; k_pool/v_pool: [num_slots, H_kv, D] bf16;
    table: [B, stride] int32 (or [..., stride] with B rows); lens: [B] int32.
    ``n_split`` defaults to ``attn_num_splits`` for ``max_len`` (default: the
    table stride).  Returns ``(out [B, n_q, H_q, D] fp32, lse [B, n_q, H_q] fp32)``.
    """
    return _attn(None, q, k_pool, v_pool, table, lens, scale, out, lse, n_split, max_len,
                 workspace, stream)


def draft_decode_attn_append(k_new: torch.Tensor, v_new: torch.Tensor, new_slots: torch.Tensor,
                             q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                             table: torch.Tensor, lens: torch.Tensor, scale: float,
                             out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                             n_split: int | None = None, max_len: int | None = None,
                             workspace: AttnWorkspace | None = None, stream=None,
                             overlap_hold: int | None = None):
    """``append_kv`` then ``draft_decode_attn`` in one launch
    (``wmtp_draft_decode_attn_append``).

    k_new/v_new: [B, n_new, H_kv, D] bf16 (or [B, H_kv, D] for n_new = 1);
    new_slots: [B, n_new] (or [B]) int32 pool slots.  Other arguments and the
    result as :func:`draft_decode_attn`; the pools are written.
    ``overlap_hold`` not None: a chained step (``wmtp_draft_decode_attn_append_overlap``):
    -1 for the first step of a chain (nothing read early), >= 0 to start the
    copies of every entry but the last ``overlap_hold`` of a row while the
    preceding kernel on the stream finishes (2 for steps >= 1 of consecutive
    fused steps); same results bit for bit."""
    if overlap_hold is not None and int(overlap_hold) < -1:
        raise ValueError("overlap_hold must be -1 or >= 0 (None: not a chained step)")
    return _attn((k_new, v_new, new_slots, overlap_hold), q, k_pool, v_pool, table, lens, scale, out, lse,
                 n_split, max_len, workspace, stream)


def draft_extend_attn(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                      table: torch.Tensor, lens: torch.Tensor, seq_lens: torch.Tensor,
                      n_new: torch.Tensor, n_sink: int, window: int, scale: float,
                      windowed: bool = True, out: torch.Tensor | None = None,
                      lse: torch.Tensor | None = None, n_split: int | None = None,
                      max_len: int | None = None, workspace: AttnWorkspace | None = None,
                      stream=None):
    """Draft-extend attention over a union table (``wmtp_draft_extend_attn``):
    row t of request b attends the keys draft step t sees; rows t >= n_new[b]
    give zeros and lse = -inf.  q: [B, n_q, H_q, D] bf16; table/lens from
    :func:`build_extend_indices`.  Returns ``(out, lse)`` as
    :func:`draft_decode_attn`."""
    _need(seq_lens, "seq_lens", torch.int32, q.device)
    _need(n_new, "n_new", torch.int32, q.device)
    return _attn(("extend", seq_lens, n_new, n_sink, window, windowed), q, k_pool, v_pool, table,
                 lens, scale, out, lse, n_split, max_len, workspace, stream)


def draft_decode_attn_fp8(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                          k_scale: torch.Tensor, v_scale: torch.Tensor, table: torch.Tensor,
                          lens: torch.Tensor, scale: float, out: torch.Tensor | None = None,
                          lse: torch.Tensor | None = None, n_split: int | None = None,
                          max_len: int | None = None, workspace: AttnWorkspace | None = None,
                          stream=None):
    """:func:`draft_decode_attn` over E4M3 pools (``wmtp_draft_decode_attn_fp8``):
    k_pool/v_pool [num_slots, H_kv, D] uint8 codes, element = code *
    k_scale[g] (or v_scale[g]), k_scale/v_scale [H_kv] fp32."""
    for t, nm in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        _need(t, nm, torch.float32, q.device)
    if k_scale.numel() != k_pool.shape[1] or v_scale.numel() != k_pool.shape[1]:
        raise ValueError("draft_decode_attn_fp8: one scale per KV head expected")
    return _attn(("fp8", k_scale, v_scale), q, k_pool, v_pool, table, lens, scale, out, lse,
                 n_split, max_len, workspace, stream)


def _attn_shapes(what, q, k_pool, v_pool, table, lens, out, lse):
    """Shape checks of an attention call, made before anything else (the
    kernels index every buffer from these sizes, so a short buffer would be
    read or written past its end).  q [B, n_q, H_q, D]; k_pool and v_pool
    [num_slots, H_kv, D]; table rows of `stride` entries (at least B rows);
    lens at least B entries; out, lse (when given) exactly [B, n_q, H_q, D]
    and [B, n_q, H_q].  Returns (B, n_q, H_q, D, num_slots, H_kv, stride)."""
    if q.dim() != 4 or k_pool.dim() != 3:
        raise ValueError(f"{what}: q must be [B, n_q, H_q, D] and k_pool [num_slots, H_kv, D]")
    B, n_q, H_q, D = q.shape
    num_slots, H_kv, Dk = k_pool.shape
    if Dk != D:
        raise ValueError(f"{what}: k_pool head dim {Dk} differs from q's {D}")
    if v_pool.shape != k_pool.shape:
        raise ValueError(f"{what}: v_pool shape {tuple(v_pool.shape)} differs from k_pool's "
                         f"{tuple(k_pool.shape)}")
    stride = table.shape[-1] if table.dim() > 0 else 0
    if stride < 1 or table.numel() < B * stride or lens.numel() < B:
        raise ValueError(f"{what}: table/lens smaller than B rows")
    if out is not None and tuple(out.shape) != (B, n_q, H_q, D):
        raise ValueError(f"{what}: out shape {tuple(out.shape)}, expected {(B, n_q, H_q, D)}")
    if lse is not None and tuple(lse.shape) != (B, n_q, H_q):
        raise ValueError(f"{what}: lse shape {tuple(lse.shape)}, expected {(B, n_q, H_q)}")
    return B, n_q, H_q, D, num_slots, H_kv, stride


def _attn(append, q, k_pool, v_pool, table, lens, scale, out, lse, n_split, max_len, workspace,
          stream):
    B, n_q, H_q, D, num_slots, H_kv, stride = _attn_shapes("draft_decode_attn", q, k_pool, v_pool,
                                                           table, lens, out, lse)
    _need(q, "q", torch.bfloat16)
    dev = q.device
    pool_dtype = torch.uint8 if (append is not None and append[0] == "fp8") else torch.bfloat16
    for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, nm, pool_dtype, dev)
    _need(table, "table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev)
    if out is None:
        out = torch.empty((B, n_q, H_q, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, n_q, H_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    if n_split is None:
        ml = max_len if max_len is not None else stride
        if append is not None and append[0] == "extend":
            with _on(dev):
                n_split = int(load().wmtp_extend_num_splits(B, n_q, H_kv, int(ml)))
        else:
            n_split = attn_num_splits(B, n_q, H_kv, ml, dev, fp8=pool_dtype == torch.uint8)
    need = attn_workspace_bytes(B, n_q, H_q, H_kv, D, n_split)
    if workspace is None:
        # one zero-initialised workspace per (device, stream, layout): the merge
        # counters sit at layout-dependent offsets
        sid = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream
        key = (dev, sid, B * n_q * H_kv, H_q, D, n_split)
        ws = _ws_cache.get(key)
        if ws is None:
            ws = AttnWorkspace(need, dev, stream)
            _ws_cache[key] = ws
        workspace = ws
    elif workspace.nbytes < need:
        raise ValueError(f"workspace holds {workspace.nbytes} bytes, {need} needed")
    if append is None:
        with _on(dev):
            _check(load().wmtp_draft_decode_attn(
                _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(table),
                stride, _ptr(lens), float(scale), _ptr(out), _ptr(lse), _ptr(workspace.buf),
                workspace.nbytes, n_split, _stream(stream)), "draft_decode_attn")
        return out, lse
    if append[0] == "fp8":
        _, k_scale, v_scale = append
        with _on(dev):
            _check(load().wmtp_draft_decode_attn_fp8(
                _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), _ptr(k_scale),
                _ptr(v_scale), num_slots, _ptr(table), stride, _ptr(lens), float(scale), _ptr(out),
                _ptr(lse), _ptr(workspace.buf), workspace.nbytes, n_split, _stream(stream)),
                "draft_decode_attn_fp8")
        return out, lse
    if append[0] == "extend":
        _, seq_lens, n_new, n_sink, window, windowed = append
        with _on(dev):
            _check(load().wmtp_draft_extend_attn(
                _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(table),
                stride, _ptr(lens), _ptr(seq_lens), _ptr(n_new), n_sink, window, int(bool(windowed)),
                float(scale), _ptr(out), _ptr(lse), _ptr(workspace.buf), workspace.nbytes, n_split,
                _stream(stream)), "draft_extend_attn")
        return out, lse
    k_new, v_new, new_slots, hold = append
    _need(k_new, "k_new", torch.bfloat16, dev)
    _need(v_new, "v_new", torch.bfloat16, dev)
    _need(new_slots, "new_slots", torch.int32, dev)
    n_new = new_slots.numel() // max(B, 1)
    if (new_slots.numel() != B * n_new or k_new.numel() != B * n_new * H_kv * D
            or v_new.shape != k_new.shape or k_new.shape[-2:] != (H_kv, D)):
        raise ValueError("draft_decode_attn_append: k_new/v_new/new_slots shape mismatch")
    with _on(dev):
        if hold is None:
            _check(load().wmtp_draft_decode_attn_append(
                _ptr(k_new), _ptr(v_new), _ptr(new_slots), n_new,
                _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(table),
                stride, _ptr(lens), float(scale), _ptr(out), _ptr(lse), _ptr(workspace.buf),
                workspace.nbytes, n_split, _stream(stream)), "draft_decode_attn_append")
        else:
            _check(load().wmtp_draft_decode_attn_append_overlap(
                _ptr(k_new), _ptr(v_new), _ptr(new_slots), n_new,
                _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(table),
                stride, _ptr(lens), float(scale), _ptr(out), _ptr(lse), _ptr(workspace.buf),
                workspace.nbytes, n_split, int(hold), _stream(stream)), "draft_decode_attn_append_overlap")
    return out, lse


def attn_mass_diagnostics(o_win: torch.Tensor, lse_win: torch.Tensor, o_far: torch.Tensor,
                          lse_far: torch.Tensor, o_full: torch.Tensor | None = None,
                          lse_full: torch.Tensor | None = None, stream=None):
    """Per query row: (in_win, win_perturb, tail_out_frac) from the windowed
    attention and the attention over the far keys of the same queries
    (``wmtp_attn_mass_diagnostics``).  o_*: [..., D] fp32; lse_*: [...] fp32.
    Returns three fp32 tensors shaped like lse_win; when ``o_full`` /
    ``lse_full`` are given, the merged full-context attention is written
    there too."""
    for t, nm in ((o_win, "o_win"), (lse_win, "lse_win"), (o_far, "o_far"), (lse_far, "lse_far")):
        _need(t, nm, torch.float32, o_win.device)
    D = o_win.shape[-1]
    rows = lse_win.numel()
    if o_win.numel() != rows * D or o_far.numel() != rows * D or lse_far.numel() != rows:
        raise ValueError("attn_mass_diagnostics: shape mismatch")
    if o_full is not None:
        _need(o_full, "o_full", torch.float32, o_win.device)
        if o_full.numel() != rows * D:
            raise ValueError("attn_mass_diagnostics: o_full shape mismatch")
    if lse_full is not None:
        _need(lse_full, "lse_full", torch.float32, o_win.device)
        if lse_full.numel() != rows:
            raise ValueError("attn_mass_diagnostics: lse_full shape mismatch")
    res = [torch.empty_like(lse_win) for _ in range(3)]
    with _on(o_win.device):
        _check(load().wmtp_attn_mass_diagnostics(
            _ptr(o_win), _ptr(lse_win), _ptr(o_far), _ptr(lse_far), rows, D, _ptr(res[0]),
            _ptr(res[1]), _ptr(res[2]), _ptr(o_full), _ptr(lse_full), _stream(stream)),
            "attn_mass_diagnostics")
    return tuple(res)


def draft_decode_attn_noalloc(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                              table: torch.Tensor, lens: torch.Tensor, scale: float,
                              out: torch.Tensor, lse: torch.Tensor, n_split: int, stream=None):
    """``wmtp_draft_decode_attn_noalloc``: the same attention as
    :func:`draft_decode_attn`, for callers that cannot provide a workspace
    (the library uses a fixed scratch array it holds on the device).  The
    outputs must be passed in; nothing is allocated on this path.  The first
    call on a device looks up the scratch address: make it before any stream
    capture.  Calls that overlap on the GPU share the scratch and race.
    Shapes are checked as for :func:`draft_decode_attn`; `out` and `lse` must
    be exactly [B, n_q, H_q, D] and [B, n_q, H_q]."""
    if out is None or lse is None:
        raise ValueError("draft_decode_attn_noalloc: out and lse must be passed in")
    B, n_q, H_q, D, num_slots, H_kv, stride = _attn_shapes(
        "draft_decode_attn_noalloc", q, k_pool, v_pool, table, lens, out, lse)
    _need(q, "q", torch.bfloat16)
    dev = q.device
    for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, nm, torch.bfloat16, dev)
    _need(table, "table", torch.int32, dev)
    _need(lens, "lens", torch.int32, dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    with _on(dev):
        _check(load().wmtp_draft_decode_attn_noalloc(
            _ptr(q), B, n_q, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(table),
            stride, _ptr(lens), float(scale), _ptr(out), _ptr(lse), int(n_split),
            _stream(stream)), "draft_decode_attn_noalloc")
    return out, lse


def tree_workspace_bytes(B: int, H_q: int, H_kv: int, D: int, depth: int, tree_k: int,
                         n_split: int) -> int:
    return int(load().wmtp_tree_workspace_bytes(B, H_q, H_kv, D, depth, tree_k, n_split))


def tree_num_splits(B: int, H_q: int, H_kv: int, depth: int, tree_k: int, n_sink: int,
                    window: int, device=None) -> int:
    dev = device if device is not None else torch.cuda.current_device()
    with _on(dev):
        return int(load().wmtp_tree_num_splits(B, H_q, H_kv, depth, tree_k, n_sink, window))


def tree_draft_attn(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                    seq_lens: torch.Tensor, ring_base: torch.Tensor, n_sink: int, window: int,
                    depth: int, tree_k: int, scale: float, out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None, n_split: int | None = None,
                    workspace: AttnWorkspace | None = None, stream=None):
    """Tree-draft attention over the ring (``wmtp_tree_draft_attn``).

    q: [B, tree_k*depth, H_q, D] bf16 (node t = branch*depth + i); k_pool /
    v_pool: [num_slots, H_kv, D] bf16 holding each request's ring at
    ``ring_base``; seq_lens: committed lengths [B] int32.
    Returns ``(out [B, k*d, H_q, D] fp32, lse [B, k*d, H_q] fp32)``.
    """
    _need(q, "q", torch.bfloat16)
    dev = q.device
    for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, nm, torch.bfloat16, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    _need(ring_base, "ring_base", torch.int32, dev)
    B, n_nodes, H_q, D = q.shape
    if n_nodes != tree_k * depth:
        raise ValueError("q must hold tree_k * depth nodes per request")
    num_slots, H_kv, _ = k_pool.shape
    if out is None:
        out = torch.empty((B, n_nodes, H_q, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, n_nodes, H_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    if n_split is None:
        n_split = tree_num_splits(B, H_q, H_kv, depth, tree_k, n_sink, window, dev)
    need = tree_workspace_bytes(B, H_q, H_kv, D, depth, tree_k, n_split)
    if workspace is None:
        sid = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream
        key = ("tree", dev, sid, B, H_q, H_kv, D, depth, tree_k, n_split)
        ws = _ws_cache.get(key)
        if ws is None:
            ws = AttnWorkspace(need, dev, stream)
            _ws_cache[key] = ws
        workspace = ws
    elif workspace.nbytes < need:
        raise ValueError(f"workspace holds {workspace.nbytes} bytes, {need} needed")
    with _on(dev):
        _check(load().wmtp_tree_draft_attn(
            _ptr(q), B, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots, _ptr(seq_lens),
            _ptr(ring_base), n_sink, window, depth, tree_k, float(scale), _ptr(out), _ptr(lse),
            _ptr(workspace.buf), workspace.nbytes, n_split, _stream(stream)), "tree_draft_attn")
    return out, lse


# ---------------------------------------------------------------- ring path without tables
def prefill_keep_positions(seq_lens: torch.Tensor, n_sink: int, window: int, stride: int | None = None,
                           positions: torch.Tensor | None = None, counts: torch.Tensor | None = None,
                           stream=None):
    """Prompt positions whose draft KV the windowed draft needs after the
    prompt (``wmtp_prefill_keep_positions``).  Returns ``(positions[B, stride],
    counts[B])`` int32; ``stride`` defaults to ``n_sink + window``."""
    _need(seq_lens, "seq_lens", torch.int32)
    dev = seq_lens.device
    B = seq_lens.numel()
    stride = stride if stride is not None else n_sink + window
    if positions is None:
        positions = torch.empty((B, stride), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((B,), dtype=torch.int32, device=dev)
    _need(positions, "positions", torch.int32, dev)
    _need(counts, "counts", torch.int32, dev)
    with _on(dev):
        _check(load().wmtp_prefill_keep_positions(_ptr(seq_lens), B, n_sink, window, _ptr(positions),
                                                  positions.shape[-1], _ptr(counts), _stream(stream)),
               "prefill_keep_positions")
    return positions, counts


def ring_fill(k_rows: torch.Tensor, v_rows: torch.Tensor, seq_lens: torch.Tensor, ring_base: torch.Tensor,
              n_sink: int, window: int, depth: int, k_pool: torch.Tensor, v_pool: torch.Tensor,
              tree_k: int = 1, stream=None) -> None:
    """Write each request's draft K/V of its kept prompt positions (rows in
    keep order, ``[B, stride, H_kv, D]`` bf16) into its ring (``wmtp_ring_fill``)."""
    _need(k_pool, "k_pool", torch.bfloat16)
    dev = k_pool.device
    for t, nm in ((v_pool, "v_pool"), (k_rows, "k_rows"), (v_rows, "v_rows")):
        _need(t, nm, torch.bfloat16, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    _need(ring_base, "ring_base", torch.int32, dev)
    B, stride, H_kv, D = k_rows.shape
    if v_rows.shape != k_rows.shape or k_pool.shape[1:] != (H_kv, D) or v_pool.shape != k_pool.shape:
        raise ValueError("ring_fill: shape mismatch")
    with _on(dev):
        _check(load().wmtp_ring_fill(_ptr(k_rows), _ptr(v_rows), _ptr(seq_lens), B, stride, H_kv, D,
                                     _ptr(ring_base), n_sink, window, depth, tree_k, _ptr(k_pool),
                                     _ptr(v_pool), k_pool.shape[0], _stream(stream)), "ring_fill")


def draft_decode_attn_ring(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           seq_lens: torch.Tensor, ring_base: torch.Tensor, step: int, n_sink: int,
                           window: int, depth: int, scale: float, k_new: torch.Tensor | None = None,
                           v_new: torch.Tensor | None = None, tree_k: int = 1,
                           out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                           n_split: int | None = None, workspace: AttnWorkspace | None = None,
                           stream=None, overlap_hold: int | None = None):
    """Draft step ``step`` over the ring with no table (``wmtp_draft_decode_attn_ring``):
    q [B, 1, H_q, D] (or [B, H_q, D]) bf16; k_new/v_new [B, H_kv, D] bf16 appended at
    position S + step first (optional).  Returns ``(out [B, 1, H_q, D], lse [B, 1, H_q])``.
    ``overlap_hold`` not None: a chained step as in :func:`draft_decode_attn_append`
    (``wmtp_draft_decode_attn_ring_overlap``; needs k_new / v_new)."""
    if overlap_hold is not None and int(overlap_hold) < -1:
        raise ValueError("overlap_hold must be -1 or >= 0 (None: not a chained step)")
    if overlap_hold is not None and k_new is None:
        raise ValueError("draft_decode_attn_ring: a chained step appends (give k_new and v_new)")
    _need(q, "q", torch.bfloat16)
    dev = q.device
    for t, nm in ((k_pool, "k_pool"), (v_pool, "v_pool")):
        _need(t, nm, torch.bfloat16, dev)
    _need(seq_lens, "seq_lens", torch.int32, dev)
    _need(ring_base, "ring_base", torch.int32, dev)
    B = seq_lens.numel()
    D = q.shape[-1]
    H_q = q.numel() // (B * D) if B else 0
    num_slots, H_kv, Dk = k_pool.shape
    if Dk != D or v_pool.shape != k_pool.shape:
        raise ValueError("draft_decode_attn_ring: pool shape mismatch")
    if (k_new is None) != (v_new is None):
        raise ValueError("draft_decode_attn_ring: give both k_new and v_new, or neither")
    if k_new is not None:
        _need(k_new, "k_new", torch.bfloat16, dev)
        _need(v_new, "v_new", torch.bfloat16, dev)
        if k_new.numel() != B * H_kv * D or v_new.shape != k_new.shape:
            raise ValueError("draft_decode_attn_ring: k_new/v_new shape mismatch")
    if out is None:
        out = torch.empty((B, 1, H_q, D), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, 1, H_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev)
    _need(lse, "lse", torch.float32, dev)
    if n_split is None:
        n_split = attn_num_splits(B, 1, H_kv, n_sink + window, dev)
    need = attn_workspace_bytes(B, 1, H_q, H_kv, D, n_split)
    if workspace is None:
        sid = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream.cuda_stream
        key = (dev, sid, B * H_kv, H_q, D, n_split)
        workspace = _ws_cache.get(key)
        if workspace is None:
            workspace = AttnWorkspace(need, dev, stream)
            _ws_cache[key] = workspace
    elif workspace.nbytes < need:
        raise ValueError(f"workspace holds {workspace.nbytes} bytes, {need} needed")
    with _on(dev):
        if overlap_hold is None:
            _check(load().wmtp_draft_decode_attn_ring(
                _ptr(k_new), _ptr(v_new), _ptr(q), B, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots,
                _ptr(seq_lens), _ptr(ring_base), int(step), n_sink, window, depth, tree_k, float(scale),
                _ptr(out), _ptr(lse), _ptr(workspace.buf), workspace.nbytes, n_split, _stream(stream)),
                "draft_decode_attn_ring")
        else:
            _check(load().wmtp_draft_decode_attn_ring_overlap(
                _ptr(k_new), _ptr(v_new), _ptr(q), B, H_q, H_kv, D, _ptr(k_pool), _ptr(v_pool), num_slots,
                _ptr(seq_lens), _ptr(ring_base), int(step), n_sink, window, depth, tree_k, float(scale),
                _ptr(out), _ptr(lse), _ptr(workspace.buf), workspace.nbytes, n_split, int(overlap_hold),
                _stream(stream)), "draft_decode_attn_ring_overlap")
    return out, lse
