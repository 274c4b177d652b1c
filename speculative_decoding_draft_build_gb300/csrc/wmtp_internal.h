// wmtp_internal.h -- host-side helpers shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "wmtp.h"

namespace wmtp {

// 3-D TMA map of a [num_slots][H_kv][D] bf16 pool: boxes of 64 dims x 1 head
// x `rows` consecutive slots, 128-byte swizzle (defined in wmtp_tree.cu).
// False if the driver entry point is missing or the encoding is refused.
bool pool_tensor_map(CUtensorMap *map, const void *pool, int64_t num_slots, int H_kv, int D, int rows);

// Each translation unit keeps its own device error word (no relocatable
// device code is needed); these read-and-optionally-clear them.
cudaError_t read_index_error(int32_t *code, bool clear);
cudaError_t read_attn_error(int32_t *code, bool clear);
cudaError_t read_tree_tc_error(int32_t *code, bool clear);
size_t tree_tc_workspace_bytes(int64_t B, int64_t H_kv, int64_t R, int D, int n_split);
wmtp_status tree_tc_launch(const uint16_t *q, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                           const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                           const int32_t *seq_lens, const int32_t *ring_base, int32_t n_sink,
                           int32_t window, int32_t depth, int32_t tree_k, float scale, float *out,
                           float *lse, void *workspace, int32_t n_split, cudaStream_t stream);

// Draft extend with one K/V read per request (wmtp_extend.cu): up to
// kMaxExtendTokens tokens per request, up to kMaxExtendSplits splits; the
// partials use the split-order workspace layout of the decode attention.
constexpr int kMaxExtendTokens = 8;
constexpr int kMaxExtendSplits = 128;
// Rows (table strides) of at least this many keys per split take the
// one-read launch; shorter rows, where a CTA sees a few tiles and latency
// dominates, are faster as one set of CTAs per token (L2 serves the rereads).
constexpr int kExtendMinKeysPerSplit = 1024;
cudaError_t read_extend_error(int32_t *code, bool clear);
wmtp_status extend_multi_launch(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t D,
                                const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                                const int32_t *table, int64_t table_stride, const int32_t *lens,
                                const int32_t *seq_lens, const int32_t *n_new, int32_t n_sink, int32_t window,
                                int32_t windowed, float scale, float *out, float *lse, int32_t *counters,
                                float *lse_part, float *o_part, int32_t n_split, cudaStream_t stream);

// Draft extend on the tensor cores (wmtp_tree.cu): a chain of n_q nodes per
// request over the union table row, for rows of at least kTreeExtendMinKeys
// keys and up to kTreeExtendMaxSplits splits; the partials of a split-order
// merge use the decode attention's workspace layout (counters zero at rest).
constexpr int64_t kTreeExtendMinKeys = 65536;
constexpr int kTreeExtendMaxSplits = 128;
wmtp_status tree_extend_launch(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv,
                               int32_t D, const uint16_t *k_pool, const uint16_t *v_pool,
                               int64_t num_slots, const int32_t *table, int64_t table_stride,
                               const int32_t *lens, const int32_t *seq_lens, const int32_t *n_new,
                               int32_t n_sink, int32_t window, int32_t windowed, float scale,
                               float *out, float *lse, int32_t *ws_counters, float *ws_lse_part,
                               float *ws_o_part, int32_t n_split, cudaStream_t stream);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline wmtp_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

// Launch configuration with programmatic stream serialization: the kernel may
// begin launching while the previous kernel in the stream drains; every
// kernel of this library calls griddepcontrol.wait before touching global
// memory, so ordering is unchanged and only launch latency is hidden.
struct PdlLaunch {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attrs[2]{};
    PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t stream) {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attrs;
        cfg.numAttrs = 1;
    }
    void add_cluster(unsigned x) {
        attrs[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
        attrs[cfg.numAttrs].val.clusterDim.x = x;
        attrs[cfg.numAttrs].val.clusterDim.y = 1;
        attrs[cfg.numAttrs].val.clusterDim.z = 1;
        ++cfg.numAttrs;
    }
};

}  // namespace wmtp
