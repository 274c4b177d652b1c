"""Plain fp64 CPU oracle for the Windowed-MTP draft-attention hot path.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs import this package.  The CUDA
library never links, imports or calls it, and it shares no code with it.

The arithmetic lives in ``wmtp_oracle.c`` (plain loops, fp64); this module
compiles it with gcc on first use and marshals numpy arrays through ctypes.
bf16 tensors travel as ``numpy.uint16`` bit patterns.
"""
from .oracle import (  # noqa: F401
    ORC_OK,
    acceptance_length,
    append_kv,
    append_kv_fp8,
    attn_mass,
    build,
    build_draft_indices,
    build_extend_indices,
    build_far_indices,
    draft_decode_attn,
    draft_decode_attn_fp8,
    draft_extend_attn,
    e4m3_table,
    e4m3_to_f64,
    f32_to_e4m3,
    far_positions,
    keep,
    num_threads,
    prefill_keep_positions,
    ring_fill,
    ring_map,
    ring_slot,
    tree_draft_attn,
)
