"""ctypes front end of the C oracle (``wmtp_oracle.c``).

Test infrastructure only; see the package docstring.  Each wrapper names the
passage of "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
Million-Token Context" (arXiv 2607.21535) that the C function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ORC_OK = 0
ORC_EINVAL = -1
ORC_ECAPACITY = -2
ORC_EBOUNDS = -4

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wmtp_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, OpenMP over output rows).

    No -ffast-math: every floating-point operation keeps the order written in
    the C source.
    """
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC",
               "-shared", "-Wall", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_keep.restype = _i64
        lib.orc_keep.argtypes = [_i64, _i64, _i64, ctypes.c_int, _i64p]
        lib.orc_ring_slot.restype = _i64
        lib.orc_ring_slot.argtypes = [_i64] * 7
        lib.orc_ring_map.restype = ctypes.c_int
        lib.orc_ring_map.argtypes = [_i32p, _i32p, _i32p, _i32p, _i64, _i64,
                                     _i64, _i64, _i64, _i32p]
        lib.orc_build_draft_indices.restype = ctypes.c_int
        lib.orc_build_draft_indices.argtypes = [
            _i32p, _i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_int,
            _i32p, _i32p, _i64, _i32p, _i32p, _i64, _i32p]
        lib.orc_append_kv.restype = ctypes.c_int
        lib.orc_append_kv.argtypes = [_u16p, _u16p, _i32p, _i64, _i64, _i64,
                                      _u16p, _u16p, _i64]
        lib.orc_draft_decode_attn.restype = ctypes.c_int
        lib.orc_draft_decode_attn.argtypes = [
            _u16p, _i64, _i64, _i64, _i64, _i64, _u16p, _u16p, _i64, _i32p,
            _i64, _i32p, ctypes.c_double, _i64p, _i64, _f64p, _f64p, _f64p,
            _i64, ctypes.c_int]
        lib.orc_tree_draft_attn.restype = ctypes.c_int
        lib.orc_tree_draft_attn.argtypes = [
            _u16p, _i64, _i64, _i64, _i64, _u16p, _u16p, _i64, _i32p, _i32p,
            _i64, _i64, _i64, _i64, ctypes.c_double, _i64p, _i64, _f64p,
            _f64p, ctypes.c_int]
        lib.orc_e4m3_to_f64.restype = ctypes.c_double
        lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.orc_f32_to_e4m3.restype = ctypes.c_uint8
        lib.orc_f32_to_e4m3.argtypes = [ctypes.c_float]
        lib.orc_append_kv_fp8.restype = ctypes.c_int
        lib.orc_append_kv_fp8.argtypes = [_u16p, _u16p, _i32p, _i64, _i64, _i64,
                                          _f32p, _f32p, _u8p, _u8p, _i64]
        lib.orc_draft_decode_attn_fp8.restype = ctypes.c_int
        lib.orc_draft_decode_attn_fp8.argtypes = [
            _u16p, _i64, _i64, _i64, _i64, _i64, _u8p, _u8p, _f32p, _f32p, _i64,
            _i32p, _i64, _i32p, ctypes.c_double, _i64p, _i64, _f64p, _f64p, _f64p,
            _i64, ctypes.c_int]
        lib.orc_acceptance_length.restype = ctypes.c_double
        lib.orc_acceptance_length.argtypes = [_f64p, _i64, _f64p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _as(a, dtype) -> np.ndarray | None:
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _check(status: int, what: str) -> None:
    if status != ORC_OK:
        raise ValueError(f"oracle {what} failed with status {status}")


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use by default."""
    return int(_load().orc_num_threads())


def keep(s_kv: int, n_sink: int, window: int, windowed: bool = True) -> np.ndarray:
    """Positions a draft step with kv length ``s_kv`` attends (App. A
    pseudocode): sinks then the last ``window`` positions, or all of them."""
    lib = _load()
    n = lib.orc_keep(s_kv, n_sink, window, int(windowed), None)
    out = np.empty(max(n, 0), dtype=np.int64)
    lib.orc_keep(s_kv, n_sink, window, int(windowed), _ptr(out, ctypes.c_int64))
    return out


def far_positions(s_kv: int, n_sink: int, window: int) -> np.ndarray:
    """Positions a windowed draft step with kv length ``s_kv`` does NOT
    attend: every position of [0, s_kv) outside :func:`keep` (§5 "A
    partition-function view": the full key set is the kept set plus these
    far keys), ascending.  Written as the set difference itself."""
    kept = set(int(x) for x in keep(s_kv, n_sink, window, True))
    return np.array([p for p in range(max(s_kv, 0)) if p not in kept], dtype=np.int64)


def build_far_indices(seq_lens, gamma, n_sink, window, req_to_token, req_pool_idx=None,
                      stride=None):
    """Far-key tables: for draft step j of request b (kv length S_b + j + 1,
    as the draft tables), the slots req_to_token[row b] of
    :func:`far_positions`.  Returns ``(table[gamma, B, stride] int32,
    lens[gamma, B] int32)``; entries past ``lens`` are -1."""
    sl = _as(seq_lens, np.int64)
    rtt = _as(req_to_token, np.int32)
    B = sl.shape[0]
    stride = rtt.shape[1] if stride is None else int(stride)
    table = np.full((gamma, B, stride), -1, np.int32)
    lens = np.zeros((gamma, B), np.int32)
    for j in range(gamma):
        for b in range(B):
            row = int(req_pool_idx[b]) if req_pool_idx is not None else b
            pos = far_positions(int(sl[b]) + j + 1, n_sink, window)
            if len(pos) > stride:
                raise ValueError("build_far_indices: a row needs more than stride entries")
            lens[j, b] = len(pos)
            table[j, b, :len(pos)] = rtt[row, pos]
    return table, lens


def ring_slot(ring_base: int, p: int, branch: int, n_sink: int, window: int,
              depth: int, tree_k: int = 1) -> int:
    """Ring slot of logical position ``p`` (App. A; §7 tree sizing)."""
    return int(_load().orc_ring_slot(ring_base, p, branch, n_sink, window,
                                     depth, tree_k))


def ring_map(ring_base, pos, req_of, n_sink, window, depth, tree_k=1,
             branch=None) -> np.ndarray:
    """Vector form of :func:`ring_slot` over (request, position, branch)."""
    rb = _as(ring_base, np.int32)
    p = _as(pos, np.int32)
    r = _as(req_of, np.int32)
    br = _as(branch, np.int32)
    out = np.empty(p.shape[0], dtype=np.int32)
    _check(_load().orc_ring_map(_ptr(rb, ctypes.c_int32), _ptr(p, ctypes.c_int32),
                                _ptr(br, ctypes.c_int32), _ptr(r, ctypes.c_int32),
                                p.shape[0], n_sink, window, depth, tree_k,
                                _ptr(out, ctypes.c_int32)), "ring_map")
    return out


def build_draft_indices(seq_lens, gamma, n_sink, window, depth, tree_k=1,
                        windowed=True, req_to_token=None, req_pool_idx=None,
                        ring_base=None, stride=None):
    """Draft KV-index tables for ``gamma`` draft steps (§4 Mechanism; App. A).

    Returns ``(table[gamma, B, stride] int32, lens[gamma, B] int32)``; entries
    past ``lens`` are left at -1.
    """
    sl = _as(seq_lens, np.int32)
    B = sl.shape[0]
    rtt = _as(req_to_token, np.int32)
    rpi = _as(req_pool_idx, np.int32)
    rb = _as(ring_base, np.int32)
    if rtt is not None and rpi is None:
        rpi = np.arange(B, dtype=np.int32)
    if stride is None:
        stride = max([int(len(keep(int(s) + j + 1, n_sink, window, windowed)))
                      for s in sl for j in range(gamma)] + [1])
    table = np.full((gamma, B, stride), -1, dtype=np.int32)
    lens = np.zeros((gamma, B), dtype=np.int32)
    rtt_stride = rtt.shape[1] if rtt is not None else 0
    _check(_load().orc_build_draft_indices(
        _ptr(sl, ctypes.c_int32), B, gamma, n_sink, window, depth, tree_k,
        int(windowed), _ptr(rtt, ctypes.c_int32), _ptr(rpi, ctypes.c_int32),
        rtt_stride, _ptr(rb, ctypes.c_int32), _ptr(table, ctypes.c_int32),
        stride, _ptr(lens, ctypes.c_int32)), "build_draft_indices")
    return table, lens


def append_kv(k_new, v_new, slots, k_pool, v_pool) -> None:
    """Copy each new token's K/V rows into pool slot ``slots[i]`` (in place)."""
    kn = _as(k_new, np.uint16)
    vn = _as(v_new, np.uint16)
    sl = _as(slots, np.int32)
    assert k_pool.dtype == np.uint16 and k_pool.flags["C_CONTIGUOUS"]
    assert v_pool.dtype == np.uint16 and v_pool.flags["C_CONTIGUOUS"]
    n, H_kv, D = kn.shape
    _check(_load().orc_append_kv(_ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16),
                                 _ptr(sl, ctypes.c_int32), n, H_kv, D,
                                 _ptr(k_pool, ctypes.c_uint16),
                                 _ptr(v_pool, ctypes.c_uint16), k_pool.shape[0]),
           "append_kv")


def draft_decode_attn(q, k_pool, v_pool, table, lens, scale, rows=None,
                      nthreads=None):
    """fp64 softmax attention over a block table (§4 Mechanism).

    q: [B, n_q, H_q, D] bf16 bits; k_pool/v_pool: [num_slots, H_kv, D] bf16
    bits; table: [B, stride] int32; lens: [B].  ``rows`` optionally selects
    flattened (b*n_q + t)*H_q + h rows; the others come back as NaN.
    Returns ``(out[B, n_q, H_q, D] float64, lse[B, n_q, H_q] float64)``.
    """
    q = _as(q, np.uint16)
    kp = _as(k_pool, np.uint16)
    vp = _as(v_pool, np.uint16)
    tb = _as(table, np.int32)
    ln = _as(lens, np.int32)
    B, n_q, H_q, D = q.shape
    num_slots, H_kv, _ = kp.shape
    rws = _as(rows, np.int64)
    nthreads = nthreads or num_threads()
    out = np.full((B, n_q, H_q, D), np.nan, dtype=np.float64)
    lse = np.full((B, n_q, H_q), np.nan, dtype=np.float64)
    scratch_len = max(int(ln.max()) if ln.size else 0, 1)
    scratch = np.empty(scratch_len * nthreads, dtype=np.float64)
    _check(_load().orc_draft_decode_attn(
        _ptr(q, ctypes.c_uint16), B, n_q, H_q, H_kv, D, _ptr(kp, ctypes.c_uint16),
        _ptr(vp, ctypes.c_uint16), num_slots, _ptr(tb, ctypes.c_int32),
        tb.shape[-1], _ptr(ln, ctypes.c_int32), float(scale),
        _ptr(rws, ctypes.c_int64), 0 if rws is None else rws.shape[0],
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        _ptr(scratch, ctypes.c_double), scratch_len, nthreads),
        "draft_decode_attn")
    return out, lse


def tree_draft_attn(q, k_pool, v_pool, seq_lens, ring_base, n_sink, window,
                    depth, tree_k, scale, rows=None, nthreads=None):
    """fp64 tree-draft attention over the ring (§7 tree speculation).

    q: [B, tree_k*depth, H_q, D]; node t = branch*depth + i.
    Returns ``(out float64, lse float64)`` shaped like q without / with D.
    """
    q = _as(q, np.uint16)
    kp = _as(k_pool, np.uint16)
    vp = _as(v_pool, np.uint16)
    sl = _as(seq_lens, np.int32)
    rb = _as(ring_base, np.int32)
    B, n_nodes, H_q, D = q.shape
    assert n_nodes == tree_k * depth
    num_slots, H_kv, _ = kp.shape
    rws = _as(rows, np.int64)
    nthreads = nthreads or num_threads()
    out = np.full((B, n_nodes, H_q, D), np.nan, dtype=np.float64)
    lse = np.full((B, n_nodes, H_q), np.nan, dtype=np.float64)
    _check(_load().orc_tree_draft_attn(
        _ptr(q, ctypes.c_uint16), B, H_q, H_kv, D, _ptr(kp, ctypes.c_uint16),
        _ptr(vp, ctypes.c_uint16), num_slots, _ptr(sl, ctypes.c_int32),
        _ptr(rb, ctypes.c_int32), n_sink, window, depth, tree_k, float(scale),
        _ptr(rws, ctypes.c_int64), 0 if rws is None else rws.shape[0],
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double), nthreads),
        "tree_draft_attn")
    return out, lse


def acceptance_length(hist):
    """(alpha[1..gamma], AL) from an acceptance histogram (§5, Eq. 4)."""
    h = _as(hist, np.float64)
    gamma = h.shape[0] - 1
    alpha = np.zeros(max(gamma, 0), dtype=np.float64)
    al = _load().orc_acceptance_length(_ptr(h, ctypes.c_double), gamma,
                                       _ptr(alpha, ctypes.c_double))
    return alpha, float(al)


# ------------------------------------------------------------ draft extend
# A draft-extend pass is the draft forward over the n tokens a request
# accepted, at positions S..S+n-1, in one call.  Token t is exactly draft
# step t of build_draft_indices (kv_len = S + t + 1, §4 Mechanism; App. A
# keep rule), so both functions below compose the pinned functions above
# and add no arithmetic of their own.

def build_extend_indices(seq_lens, n_new, n_sink, window, depth, tree_k=1,
                         windowed=True, req_to_token=None, req_pool_idx=None,
                         ring_base=None, stride=None):
    """Union, in ascending position order, of the keep sets of steps
    0..n_new[b]-1 of each request, mapped to slots like build_draft_indices.

    Returns ``(table[B, stride] int32, lens[B] int32)``; entries past lens
    are -1."""
    sl = _as(seq_lens, np.int32)
    nn = _as(n_new, np.int32)
    B = sl.shape[0]
    rtt = _as(req_to_token, np.int32)
    rpi = _as(req_pool_idx, np.int32)
    rb = _as(ring_base, np.int32)
    if rtt is not None and rpi is None:
        rpi = np.arange(B, dtype=np.int32)
    rows = []
    for b in range(B):
        pos = set()
        for t in range(max(int(nn[b]), 0)):
            pos.update(int(p) for p in keep(int(sl[b]) + t + 1, n_sink, window, windowed))
        pos = np.array(sorted(pos), dtype=np.int64)
        if rtt is not None:
            slots = rtt[int(rpi[b])][pos] if pos.size else np.zeros(0, np.int32)
        else:
            slots = ring_map(np.array([rb[b]], np.int32), pos.astype(np.int32),
                             np.zeros(pos.size, np.int32), n_sink, window, depth, tree_k)
        rows.append(np.asarray(slots, dtype=np.int32))
    if stride is None:
        stride = max([r.size for r in rows] + [1])
    table = np.full((B, stride), -1, dtype=np.int32)
    lens = np.zeros(B, dtype=np.int32)
    for b, r in enumerate(rows):
        n = min(r.size, stride)
        table[b, :n] = r[:n]
        lens[b] = r.size
    return table, lens


def draft_extend_attn(q, k_pool, v_pool, seq_lens, n_new, n_sink, window,
                      scale, windowed=True, req_to_token=None, req_pool_idx=None,
                      ring_base=None, depth=1, tree_k=1):
    """Row t < n_new[b] of request b: draft_decode_attn over the table of
    draft step t (build_draft_indices); rows t >= n_new[b]: out 0, lse -inf.

    q: [B, n_q, H_q, D] bf16 bits.  Returns ``(out float64, lse float64)``."""
    q = _as(q, np.uint16)
    sl = _as(seq_lens, np.int32)
    nn = _as(n_new, np.int32)
    B, n_q, H_q, D = q.shape
    out = np.zeros((B, n_q, H_q, D), dtype=np.float64)
    lse = np.full((B, n_q, H_q), -np.inf, dtype=np.float64)
    if B == 0 or n_q == 0:
        return out, lse
    gamma = max(int(min(nn.max(), n_q)), 0)
    if gamma == 0:
        return out, lse
    tables, lens = build_draft_indices(sl, gamma, n_sink, window, depth, tree_k,
                                       windowed, req_to_token, req_pool_idx,
                                       ring_base)
    for b in range(B):
        for t in range(min(max(int(nn[b]), 0), n_q)):
            o, l = draft_decode_attn(q[b:b + 1, t:t + 1], k_pool, v_pool,
                                     tables[t][b:b + 1], lens[t][b:b + 1], scale)
            out[b, t] = o[0, 0]
            lse[b, t] = l[0, 0]
    return out, lse


# ------------------------------------------------- attention-mass diagnostics
def attn_mass(q, k_pool, v_pool, table_full, len_full, table_win, len_win, scale):
    """App. C, Table 12 quantities for every query row, straight from their
    definitions in fp64: logits z over the full table row, the kept set =
    the slots of the windowed row; in_win = sum_kept e^z / sum_all e^z,
    win_perturb = ||o_full - o_win|| / ||o_full|| with o_win the softmax
    read-out over the kept keys alone, tail_out_frac = ||sum_far p v|| /
    ||o_full|| with p the full softmax.  Plain numpy (test sizes).

    q: [B, n_q, H_q, D] bf16 bits; tables [B, stride].  Returns three float64
    arrays [B, n_q, H_q]."""
    q = _as(q, np.uint16)
    kp = _as(k_pool, np.uint16)
    vp = _as(v_pool, np.uint16)
    tf, lf = _as(table_full, np.int32), _as(len_full, np.int32)
    tw, lw = _as(table_win, np.int32), _as(len_win, np.int32)
    B, n_q, H_q, D = q.shape
    H_kv = kp.shape[1]
    G = H_q // H_kv

    def f64(u):
        return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)

    res = np.zeros((3, B, n_q, H_q), dtype=np.float64)
    for b in range(B):
        slots = tf[b, :lf[b]]
        kept = np.isin(slots, tw[b, :lw[b]])
        for h in range(H_q):
            g = h // G
            K = f64(kp[slots, g])
            V = f64(vp[slots, g])
            for t in range(n_q):
                z = scale * (K @ f64(q[b, t, h]))
                e = np.exp(z - z.max()) if z.size else z
                Z, Zw = e.sum(), e[kept].sum()
                o_full = (e[:, None] * V).sum(0) / Z if Z > 0 else np.zeros(D)
                o_win = (e[kept][:, None] * V[kept]).sum(0) / Zw if Zw > 0 else np.zeros(D)
                o_far = (e[~kept][:, None] * V[~kept]).sum(0) / Z if Z > 0 else np.zeros(D)
                nf = np.linalg.norm(o_full)
                res[0, b, t, h] = Zw / Z if Z > 0 else 0.0
                res[1, b, t, h] = np.linalg.norm(o_full - o_win) / nf if nf > 0 else 0.0
                res[2, b, t, h] = np.linalg.norm(o_far) / nf if nf > 0 else 0.0
    return res[0], res[1], res[2]


# --- fp8 (E4M3) KV with per-KV-head scales ([WMTP] §6, "Robustness to
# KV-cache quantization"; reading R13) ---

def e4m3_to_f64(code: int) -> float:
    """Value of one OCP FP8 E4M3 code (bias 7, subnormals m * 2^-9, no inf)."""
    return float(_load().orc_e4m3_to_f64(int(code) & 0xFF))


def f32_to_e4m3(x: float) -> int:
    """Nearest E4M3 code to the fp32 value x, ties to even, saturating at 448."""
    return int(_load().orc_f32_to_e4m3(float(np.float32(x))))


def e4m3_table() -> np.ndarray:
    """float64[256]: the value of every code (NaN for 0x7F and 0xFF)."""
    return np.array([e4m3_to_f64(c) for c in range(256)], dtype=np.float64)


def append_kv_fp8(k_new, v_new, slots, k_scale, v_scale, k_pool, v_pool) -> None:
    """Quantise each new token's bf16 K/V rows to E4M3 codes,
    code = E4M3(fp32(x) * fp32(1 / scale[h])), into pool slot ``slots[i]``
    (uint8 pools [num_slots, H_kv, D], in place)."""
    kn = _as(k_new, np.uint16)
    vn = _as(v_new, np.uint16)
    sl = _as(slots, np.int32)
    ks = _as(k_scale, np.float32)
    vs = _as(v_scale, np.float32)
    assert k_pool.dtype == np.uint8 and k_pool.flags["C_CONTIGUOUS"]
    assert v_pool.dtype == np.uint8 and v_pool.flags["C_CONTIGUOUS"]
    n, H_kv, D = kn.shape
    assert ks.shape == (H_kv,) and vs.shape == (H_kv,)
    _check(_load().orc_append_kv_fp8(_ptr(kn, ctypes.c_uint16), _ptr(vn, ctypes.c_uint16),
                                     _ptr(sl, ctypes.c_int32), n, H_kv, D,
                                     _ptr(ks, ctypes.c_float), _ptr(vs, ctypes.c_float),
                                     _ptr(k_pool, ctypes.c_uint8),
                                     _ptr(v_pool, ctypes.c_uint8), k_pool.shape[0]),
           "append_kv_fp8")


def draft_decode_attn_fp8(q, k_pool, v_pool, k_scale, v_scale, table, lens, scale,
                          rows=None, nthreads=None):
    """fp64 softmax attention over E4M3 pools: key i of KV head g is
    code * k_scale[g], its value code * v_scale[g]; otherwise as
    ``draft_decode_attn``."""
    q = _as(q, np.uint16)
    kp = _as(k_pool, np.uint8)
    vp = _as(v_pool, np.uint8)
    ks = _as(k_scale, np.float32)
    vs = _as(v_scale, np.float32)
    tb = _as(table, np.int32)
    ln = _as(lens, np.int32)
    B, n_q, H_q, D = q.shape
    num_slots, H_kv, _ = kp.shape
    rws = _as(rows, np.int64)
    nthreads = nthreads or num_threads()
    out = np.full((B, n_q, H_q, D), np.nan, dtype=np.float64)
    lse = np.full((B, n_q, H_q), np.nan, dtype=np.float64)
    scratch_len = max(int(ln.max()) if ln.size else 0, 1)
    scratch = np.empty(scratch_len * nthreads, dtype=np.float64)
    _check(_load().orc_draft_decode_attn_fp8(
        _ptr(q, ctypes.c_uint16), B, n_q, H_q, H_kv, D, _ptr(kp, ctypes.c_uint8),
        _ptr(vp, ctypes.c_uint8), _ptr(ks, ctypes.c_float), _ptr(vs, ctypes.c_float),
        num_slots, _ptr(tb, ctypes.c_int32), tb.shape[-1], _ptr(ln, ctypes.c_int32),
        float(scale), _ptr(rws, ctypes.c_int64), 0 if rws is None else rws.shape[0],
        _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double),
        _ptr(scratch, ctypes.c_double), scratch_len, nthreads),
        "draft_decode_attn_fp8")
    return out, lse


# --- pruned draft prefill ([WMTP] §7 "Prefill sparsification and TTFT";
# reading R14: the draft KV kept after a prompt of S positions is keep(S)) ---

def prefill_keep_positions(seq_lens, n_sink, window):
    """Per request, the prompt positions whose draft KV the windowed draft
    reads after the prompt: keep(S) (App. A keep rule at kv length S)."""
    return [keep(int(S), n_sink, window, True) for S in np.asarray(seq_lens).reshape(-1)]


def ring_fill(k_rows, v_rows, seq_lens, ring_base, n_sink, window, depth, k_pool, v_pool, tree_k=1):
    """Write row i of request b (its draft K/V at the i-th kept position, rows
    [B, stride, H_kv, D] bf16 bits) to that position's ring slot (in place):
    the keep rule, the ring rule and append_kv, composed."""
    kr = _as(k_rows, np.uint16)
    vr = _as(v_rows, np.uint16)
    rb = _as(ring_base, np.int32)
    for b, pos in enumerate(prefill_keep_positions(seq_lens, n_sink, window)):
        n = min(len(pos), kr.shape[1])
        if n == 0:
            continue
        slots = ring_map(rb, pos[:n].astype(np.int32), np.full(n, b, np.int32), n_sink, window, depth,
                         tree_k)
        append_kv(kr[b, :n], vr[b, :n], slots, k_pool, v_pool)
