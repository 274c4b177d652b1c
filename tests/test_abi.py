"""CPU checks of the C-ABI library: it builds, loads, exports every symbol that
include/wmtp.h declares, and its host-side argument checks reject bad calls
before touching the GPU.  No compute call runs here (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wmtp.h")


@pytest.fixture(scope="module")
def lib():
    wm.build()
    return wm.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wmtp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("wmtp_build_draft_indices", "wmtp_ring_map", "wmtp_append_kv", "wmtp_draft_decode_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (wmtp_[a-z0-9_]+)", out))
    missing = [n for n in _declared() if n not in exported]
    assert not missing, missing
    for n in _declared():
        getattr(lib, n)


def test_library_does_not_link_the_oracle(lib):
    out = subprocess.run(["readelf", "-d", _build.LIB_PATH], capture_output=True, text=True).stdout
    assert "oracle" not in out
    pkg = os.path.dirname(wm.__file__)
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "wmtp_oracle" not in src and "liboracle" not in src, f


def test_version_and_status_strings(lib):
    assert lib.wmtp_version() == 1000
    assert lib.wmtp_status_string(0) == b"ok"
    assert lib.wmtp_status_string(-1) == b"invalid argument"
    assert lib.wmtp_status_string(-2).startswith(b"output")


def test_workspace_size(lib):
    assert lib.wmtp_attn_workspace_bytes(1, 1, 16, 2, 256, 1) == 0
    small = lib.wmtp_attn_workspace_bytes(1, 1, 16, 2, 256, 2)
    big = lib.wmtp_attn_workspace_bytes(1, 1, 16, 2, 256, 76)
    assert 0 < small < big
    # partials of 16 heads x 76 splits x 256 dims must fit
    assert big >= 16 * 76 * 256 * 4
    assert lib.wmtp_attn_workspace_bytes(-1, 1, 16, 2, 256, 2) == 0


def test_split_heuristic_without_a_device(lib):
    # No device here: the heuristic assumes 152 SMs and no cluster capacity,
    # so short rows stay within one cluster of 16.
    ns = lib.wmtp_attn_num_splits
    assert ns(1, 1, 2, 4096) == 16           # short row: two key tiles per split, one cluster
    assert ns(1, 1, 2, 1_048_582) == 76      # long row: one CTA per SM
    assert ns(8, 1, 2, 4096) == 8            # 16 rows fill the SMs at 9 splits; 8 cover the 64 tiles
    assert ns(1, 1, 2, 1088) == 6            # 17 tiles: 8 splits of 3 tiles leave 2 empty
    assert ns(1, 1, 2, 100) == 1
    assert ns(1, 1, 1, 200 * 64) == 16
    assert ns(1, 1, 2, 0) == 1
    # the fp8 instance: one CTA per SM as well
    ns8 = lib.wmtp_attn_num_splits_fp8
    assert ns8(1, 1, 2, 1_048_582) == 76
    assert ns8(1, 1, 2, 4096) == 16
    assert ns8(8, 1, 2, 4096) == 8
    assert ns8(1, 1, 2, 100) == 1


NULL = None
P = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first


def test_attention_argument_checks(lib):
    f = lib.wmtp_draft_decode_attn
    args = dict(q=P, B=1, n_q=1, H_q=16, H_kv=2, D=256, k=P, v=P, num_slots=10, table=P,
                stride=10, lens=P, scale=0.1, out=P, lse=NULL, ws=P, ws_bytes=1 << 20, n_split=1,
                stream=NULL)

    def call(**over):
        a = dict(args, **over)
        return f(a["q"], a["B"], a["n_q"], a["H_q"], a["H_kv"], a["D"], a["k"], a["v"],
                 a["num_slots"], a["table"], a["stride"], a["lens"], a["scale"], a["out"],
                 a["lse"], a["ws"], a["ws_bytes"], a["n_split"], a["stream"])

    assert call(D=64) == wm.WMTP_EINVAL
    assert call(H_q=15) == wm.WMTP_EINVAL            # not a multiple of H_kv
    assert call(H_q=32) == wm.WMTP_EINVAL            # group of 16 > 8
    assert call(n_split=0) == wm.WMTP_EINVAL
    assert call(n_split=1025) == wm.WMTP_EINVAL
    assert call(q=NULL) == wm.WMTP_EINVAL
    assert call(k=ctypes.c_void_p(24)) == wm.WMTP_EINVAL  # pool not 16-byte aligned
    assert call(n_split=4, ws=ctypes.c_void_p(256), ws_bytes=16) == wm.WMTP_ECAPACITY
    assert call(n_split=4, ws=ctypes.c_void_p(16 + 128)) == wm.WMTP_EINVAL  # workspace alignment
    assert call(B=0) == wm.WMTP_OK                   # nothing to do, nothing launched


def test_builder_and_ring_argument_checks(lib):
    b = lib.wmtp_build_draft_indices
    assert b(P, 1, 1, 64, 0, 7, 1, 1, P, NULL, 10, NULL, P, 10, P, NULL) == wm.WMTP_EINVAL  # W < 1
    assert b(P, 1, 1, -1, 8, 7, 1, 1, P, NULL, 10, NULL, P, 10, P, NULL) == wm.WMTP_EINVAL
    assert b(P, 1, 1, 4, 8, 7, 1, 1, NULL, NULL, 10, NULL, P, 10, P, NULL) == wm.WMTP_EINVAL  # no layout
    assert b(P, 300, 300, 4, 8, 7, 1, 1, P, NULL, 10, NULL, P, 10, P, NULL) == wm.WMTP_EINVAL
    assert b(P, 0, 6, 4, 8, 7, 1, 1, P, NULL, 10, NULL, P, 10, P, NULL) == wm.WMTP_OK
    f = lib.wmtp_build_far_indices
    assert f(P, 1, 1, 64, 0, P, NULL, 10, P, 10, P, NULL) == wm.WMTP_EINVAL   # W < 1
    assert f(P, 1, 1, -1, 8, P, NULL, 10, P, 10, P, NULL) == wm.WMTP_EINVAL  # n_sink < 0
    assert f(P, 1, 1, 4, 8, NULL, NULL, 10, P, 10, P, NULL) == wm.WMTP_EINVAL  # paged layout only
    assert f(P, 1, 1, 4, 8, P, NULL, 0, P, 10, P, NULL) == wm.WMTP_EINVAL     # rtt_stride < 1
    assert f(P, 300, 300, 4, 8, P, NULL, 10, P, 10, P, NULL) == wm.WMTP_EINVAL
    assert f(P, 0, 6, 4, 8, P, NULL, 10, P, 10, P, NULL) == wm.WMTP_OK
    m = lib.wmtp_attn_mass_diagnostics
    assert m(P, P, P, P, 4, 256, NULL, NULL, NULL, NULL, NULL, NULL) == wm.WMTP_EINVAL  # no output
    assert m(P, NULL, P, P, 4, 256, P, NULL, NULL, NULL, NULL, NULL) == wm.WMTP_EINVAL  # null input
    assert m(P, P, P, P, 4, 0, P, NULL, NULL, NULL, NULL, NULL) == wm.WMTP_EINVAL       # D < 1
    assert m(P, P, P, P, 0, 256, P, NULL, NULL, NULL, NULL, NULL) == wm.WMTP_OK
    r = lib.wmtp_ring_map
    assert r(P, P, NULL, P, 5, 4, 8, 0, 1, P, NULL) == wm.WMTP_EINVAL  # depth < 1
    assert r(P, P, NULL, P, 5, 4, 8, 7, 0, P, NULL) == wm.WMTP_EINVAL  # tree_k < 1
    assert r(P, P, NULL, P, 0, 4, 8, 7, 1, P, NULL) == wm.WMTP_OK
    a = lib.wmtp_append_kv
    assert a(P, P, P, 3, 2, 250, P, P, 10, NULL) == wm.WMTP_EINVAL  # D % 8
    assert a(ctypes.c_void_p(20), P, P, 3, 2, 256, P, P, 10, NULL) == wm.WMTP_EINVAL


def test_overlapped_step_argument_checks(lib):
    f = lib.wmtp_draft_decode_attn_append_overlap
    args = dict(kn=P, vn=P, slots=P, n_new=1, q=P, B=1, n_q=1, H_q=16, H_kv=2, D=256, k=P, v=P,
                num_slots=10, table=P, stride=10, lens=P, scale=0.1, out=P, lse=NULL, ws=P,
                ws_bytes=1 << 20, n_split=1, hold=2, stream=NULL)

    def call(**over):
        a = dict(args, **over)
        return f(a["kn"], a["vn"], a["slots"], a["n_new"], a["q"], a["B"], a["n_q"], a["H_q"], a["H_kv"],
                 a["D"], a["k"], a["v"], a["num_slots"], a["table"], a["stride"], a["lens"], a["scale"],
                 a["out"], a["lse"], a["ws"], a["ws_bytes"], a["n_split"], a["hold"], a["stream"])

    assert call(hold=-2) == wm.WMTP_EINVAL           # -1 is "no overlap", below that is an error
    assert call(n_new=0) == wm.WMTP_EINVAL
    assert call(D=64) == wm.WMTP_EINVAL
    assert call(kn=ctypes.c_void_p(24)) == wm.WMTP_EINVAL  # new rows not 16-byte aligned
    assert call(B=0) == wm.WMTP_OK
    assert call(B=0, hold=-1) == wm.WMTP_OK
    r = lib.wmtp_draft_decode_attn_ring_overlap
    # k_new, v_new, q, B, H_q, H_kv, D, k, v, num_slots, seq_lens, ring_base, step, n_sink, W,
    # depth, tree_k, scale, out, lse, ws, ws_bytes, n_split, hold, stream
    ring = [P, P, P, 1, 16, 2, 256, P, P, 4200, P, P, 0, 64, 4032, 7, 1, 0.1, P, NULL, P, 1 << 20, 1]
    assert r(*ring, -2, NULL) == wm.WMTP_EINVAL
    assert r(*ring[:12], -1, *ring[13:], 2, NULL) == wm.WMTP_EINVAL  # step < 0
    assert r(*ring[:3], 0, *ring[4:], 2, NULL) == wm.WMTP_OK          # B = 0
    assert r(NULL, NULL, *ring[2:], 2, NULL) == wm.WMTP_EINVAL      # a chained ring step appends
