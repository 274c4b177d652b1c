// wmtp_index.cu -- draft KV-index builder, ring slot mapper and draft KV
// append for sm_103a, plus the library's status and device-error calls.
//
// Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
// Million-Token Context" (arXiv 2607.21535), §4 Mechanism and App. A "The
// windowing change (pseudocode)"; ring sizing from §6 Memory and §7
// "Compatibility with tree speculation".
//
// All three kernels move int32 / bf16 rows and are bandwidth- or
// launch-bound: coalesced loads and stores, no shared memory.
#include <cuda_runtime.h>
#include <stdint.h>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"
#include "wmtp_ring.cuh"

namespace wmtp {
namespace {

__device__ int32_t g_index_error = 0;

__device__ __forceinline__ void latch(int32_t code) { atomicCAS(&g_index_error, 0, code); }

// Table entries per thread of the index builder: long rows take many per
// thread (loads in flight), short rows one (more CTAs, less latency).
constexpr int kIndexPerThreadLong = 8;
constexpr int64_t kIndexLongRow = 65536;

// One grid row (blockIdx.y) per (draft step j, request b); the x dimension
// strides over the row's entries, kIndexPerThread per thread.  Entry e of a
// windowed row is position e for the sinks and e + (kv_len - W - n_sink) for
// the window.  `windowed` == 2 builds the far list instead: the positions
// the keep rule drops, [n_sink, kv_len - W) when kv_len > n_sink + W (else
// none), entry e being position n_sink + e (paged layout only).
template <int kIndexPerThread>
__global__ void __launch_bounds__(256) build_indices_kernel(
    const int32_t *__restrict__ seq_lens, int32_t B, int32_t n_sink, int32_t window,
    int32_t depth, int32_t tree_k, int32_t windowed,
    const int32_t *__restrict__ req_to_token, const int32_t *__restrict__ req_pool_idx,
    int64_t rtt_stride, const int32_t *__restrict__ ring_base, int32_t *__restrict__ table,
    int64_t stride, int32_t *__restrict__ lens, const int32_t *__restrict__ n_new) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t row = blockIdx.y;
    const int32_t j = row / B;
    const int32_t b = row - j * B;
    int64_t kv_len = (int64_t)seq_lens[b] + j + 1;
    int64_t keep_w = window;  // window of the keep rule (the ring keeps `window`)
    if (n_new) {
        // extend: the union of the key sets of the n new tokens at positions
        // S..S+n-1 = the keep rule at kv_len S + n with window W + n - 1
        int32_t nn = n_new[b];
        if (nn < 0) {
            if (blockIdx.x == 0 && threadIdx.x == 0) latch(WMTP_DEV_ARG_RANGE);
            nn = 0;
        }
        kv_len = nn == 0 ? 0 : (int64_t)seq_lens[b] + nn;
        keep_w = (int64_t)window + (nn > 0 ? nn - 1 : 0);
    }
    const bool far = windowed == 2;
    const bool win = windowed && kv_len > (int64_t)n_sink + keep_w;
    const int64_t n = kv_len <= 0 ? 0
                      : far       ? (win ? kv_len - keep_w - n_sink : 0)
                                  : (win ? (int64_t)n_sink + keep_w : kv_len);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        lens[row] = (int32_t)n;
        if (n > stride) latch(WMTP_DEV_TABLE_OVERFLOW);
    }
    const int64_t n_write = n < stride ? n : stride;
    // position of entry e: e + shift past the sinks (all of a far row)
    const int64_t shift = far ? n_sink : (win ? kv_len - keep_w - n_sink : 0);
    const int64_t first_shifted = far ? 0 : n_sink;
    int32_t *__restrict__ out = table + (int64_t)row * stride;
    // Each thread takes kIndexPerThread entries a block apart: coalesced
    // accesses, and that many independent loads in flight per thread.
    const int64_t span = (int64_t)blockDim.x * kIndexPerThread;
    const int64_t step = (int64_t)gridDim.x * span;
    if (req_to_token) {
        const int32_t pool_row = req_pool_idx ? req_pool_idx[b] : b;
        const int32_t *__restrict__ src = req_to_token + (int64_t)pool_row * rtt_stride;
        for (int64_t e0 = (int64_t)blockIdx.x * span + threadIdx.x; e0 < n_write; e0 += step) {
            int32_t v[kIndexPerThread];
#pragma unroll
            for (int u = 0; u < kIndexPerThread; ++u) {
                const int64_t e = e0 + (int64_t)u * blockDim.x;
                const int64_t p = (win && e >= first_shifted) ? e + shift : e;
                v[u] = (e < n_write && p < rtt_stride) ? __ldg(src + p) : 0;
            }
#pragma unroll
            for (int u = 0; u < kIndexPerThread; ++u) {
                const int64_t e = e0 + (int64_t)u * blockDim.x;
                const int64_t p = (win && e >= first_shifted) ? e + shift : e;
                if (e >= n_write) break;
                if (p >= rtt_stride) {
                    latch(WMTP_DEV_ARG_RANGE);
                    continue;
                }
                out[e] = v[u];
            }
        }
    } else {
        const int64_t base = ring_base[b];
        for (int64_t e0 = (int64_t)blockIdx.x * span + threadIdx.x; e0 < n_write; e0 += step) {
#pragma unroll
            for (int u = 0; u < kIndexPerThread; ++u) {
                const int64_t e = e0 + (int64_t)u * blockDim.x;
                if (e >= n_write) break;
                const int64_t p = (win && e >= first_shifted) ? e + shift : e;
                out[e] = (int32_t)ring_slot(base, p, 0, n_sink, window, depth, tree_k);
            }
        }
    }
}

__global__ void __launch_bounds__(256) ring_map_kernel(
    const int32_t *__restrict__ ring_base, const int32_t *__restrict__ pos,
    const int32_t *__restrict__ branch, const int32_t *__restrict__ req_of, int32_t n,
    int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k, int32_t *__restrict__ slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int32_t br = branch ? branch[i] : 0;
    const int32_t p = pos[i];
    if (br < 0 || br >= tree_k || p < 0) {
        latch(WMTP_DEV_ARG_RANGE);
        slots[i] = -1;
        return;
    }
    slots[i] = (int32_t)ring_slot(ring_base[req_of[i]], p, br, n_sink, window, depth, tree_k);
}

// One thread per 16-byte chunk of a token's K row set and V row set.
__global__ void __launch_bounds__(256) append_kv_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int32_t *__restrict__ slots, int64_t total, int32_t chunks_per_token,
    uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool, int64_t num_slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int64_t i = idx / chunks_per_token;
    const int64_t e = idx - i * chunks_per_token;
    const int64_t slot = slots[i];
    if (slot < 0 || slot >= num_slots) {
        latch(WMTP_DEV_SLOT_RANGE);
        return;
    }
    k_pool[slot * chunks_per_token + e] = k_new[idx];
    v_pool[slot * chunks_per_token + e] = v_new[idx];
}

// fp8 KV append: one thread per 8 elements of one token's K rows and V rows
// (16 bytes of bf16 in, 8 bytes of E4M3 codes out).  Element x of KV head h
// becomes E4M3_rn_satfinite(x * (1 / scale[h])), the reciprocal and the
// product each rounded once in fp32.
__global__ void __launch_bounds__(256) append_kv_fp8_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
    const int32_t *__restrict__ slots, int64_t total, int32_t chunks_per_token, int32_t chunks_per_head,
    const float *__restrict__ k_scale, const float *__restrict__ v_scale, uint2 *__restrict__ k_pool,
    uint2 *__restrict__ v_pool, int64_t num_slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int64_t i = idx / chunks_per_token;
    const int64_t e = idx - i * chunks_per_token;
    const int64_t slot = slots[i];
    if (slot < 0 || slot >= num_slots) {
        latch(WMTP_DEV_SLOT_RANGE);
        return;
    }
    const int h = (int)(e / chunks_per_head);
    const float ik = __frcp_rn(k_scale[h]), iv = __frcp_rn(v_scale[h]);
    k_pool[slot * chunks_per_token + e] = quant_e4m3x8(k_new[idx], ik);
    v_pool[slot * chunks_per_token + e] = quant_e4m3x8(v_new[idx], iv);
}

// Pruned draft prefill ("Windowed-MTP", §7 "Prefill sparsification and
// TTFT"): after a prompt of S positions the windowed draft needs only its KV
// of keep(S) = [0, n_sink) u [S - W, S) (all S positions when S <= n_sink + W).
// Entry i of request b's kept list is position i (sinks, or a short prompt)
// or S - W + (i - n_sink).
__device__ __forceinline__ int64_t kept_position(int64_t S, int64_t i, int32_t n_sink, int32_t window) {
    const bool win = S > (int64_t)n_sink + window;
    return (win && i >= n_sink) ? S - window + (i - n_sink) : i;
}

__device__ __forceinline__ int64_t kept_count(int64_t S, int32_t n_sink, int32_t window) {
    if (S <= 0) return 0;
    return S > (int64_t)n_sink + window ? (int64_t)n_sink + window : S;
}

// One grid row per request; writes the kept prompt positions and their count.
__global__ void __launch_bounds__(256) keep_positions_kernel(const int32_t *__restrict__ seq_lens,
                                                             int32_t n_sink, int32_t window,
                                                             int32_t *__restrict__ positions, int64_t stride,
                                                             int32_t *__restrict__ counts) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t b = blockIdx.y;
    const int64_t S = seq_lens[b];
    const int64_t n = kept_count(S, n_sink, window);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (S < 0) latch(WMTP_DEV_LEN_RANGE);
        if (n > stride) latch(WMTP_DEV_TABLE_OVERFLOW);
        counts[b] = (int32_t)(n < stride ? n : stride);
    }
    const int64_t n_write = n < stride ? n : stride;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_write;
         i += (int64_t)gridDim.x * blockDim.x)
        positions[(int64_t)b * stride + i] = (int32_t)kept_position(S, i, n_sink, window);
}

// Ring fill from the pruned prefill: row i of request b (its draft K and V at
// kept position i, bf16 [B][stride][H_kv][D]) goes to the ring slot of that
// position.  One thread per 16-byte chunk; grid row = request.
__global__ void __launch_bounds__(256) ring_fill_kernel(
    const uint4 *__restrict__ k_rows, const uint4 *__restrict__ v_rows, const int32_t *__restrict__ seq_lens,
    const int32_t *__restrict__ ring_base, int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k,
    int64_t stride, int32_t chunks_per_row, uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
    int64_t num_slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int32_t b = blockIdx.y;
    const int64_t S = seq_lens[b];
    int64_t n = kept_count(S, n_sink, window);
    if (blockIdx.x == 0 && threadIdx.x == 0 && n > stride) latch(WMTP_DEV_TABLE_OVERFLOW);
    if (n > stride) n = stride;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n * chunks_per_row) return;
    const int64_t i = idx / chunks_per_row;
    const int64_t e = idx - i * chunks_per_row;
    const int64_t slot =
        ring_slot(ring_base[b], kept_position(S, i, n_sink, window), 0, n_sink, window, depth, tree_k);
    if (slot < 0 || slot >= num_slots) {
        latch(WMTP_DEV_SLOT_RANGE);
        return;
    }
    const int64_t src = ((int64_t)b * stride + i) * chunks_per_row + e;
    k_pool[slot * chunks_per_row + e] = k_rows[src];
    v_pool[slot * chunks_per_row + e] = v_rows[src];
}

}  // namespace

cudaError_t read_index_error(int32_t *code, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(code, g_index_error, sizeof(int32_t));
    if (err != cudaSuccess || !clear) return err;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_index_error, &zero, sizeof(int32_t));
}

}  // namespace wmtp

using namespace wmtp;

extern "C" {

int32_t wmtp_version(void) { return 1000; }

const char *wmtp_status_string(int32_t status) {
    switch (status) {
        case WMTP_OK: return "ok";
        case WMTP_EINVAL: return "invalid argument";
        case WMTP_ECAPACITY: return "output or workspace too small";
        case WMTP_ECUDA: return "CUDA launch or runtime error";
        case WMTP_EDEVICE: return "device-side check failed";
        default: return "unknown status";
    }
}

wmtp_status wmtp_get_device_error(int32_t *code, int32_t clear) {
    if (!code) return WMTP_EINVAL;
    if (cudaDeviceSynchronize() != cudaSuccess) return WMTP_ECUDA;
    int32_t a = 0, b = 0, t = 0, x = 0;
    if (read_index_error(&a, clear != 0) != cudaSuccess) return WMTP_ECUDA;
    if (read_attn_error(&b, clear != 0) != cudaSuccess) return WMTP_ECUDA;
    if (read_tree_tc_error(&t, clear != 0) != cudaSuccess) return WMTP_ECUDA;
    if (read_extend_error(&x, clear != 0) != cudaSuccess) return WMTP_ECUDA;
    *code = a ? a : (b ? b : (t ? t : x));
    return WMTP_OK;
}

wmtp_status wmtp_build_draft_indices(const int32_t *seq_lens, int32_t B, int32_t gamma,
                                     int32_t n_sink, int32_t window, int32_t depth,
                                     int32_t tree_k, int32_t windowed,
                                     const int32_t *req_to_token,
                                     const int32_t *req_pool_idx, int64_t rtt_stride,
                                     const int32_t *ring_base, int32_t *table,
                                     int64_t stride, int32_t *lens, void *stream) {
    if (B < 0 || gamma < 0 || n_sink < 0 || window < 1 || depth < 1 || tree_k < 1 ||
        stride < 1)
        return WMTP_EINVAL;
    if ((int64_t)gamma * B > 65535) return WMTP_EINVAL;
    if (B == 0 || gamma == 0) return WMTP_OK;
    if (!seq_lens || !table || !lens) return WMTP_EINVAL;
    if (!req_to_token && !ring_base) return WMTP_EINVAL;
    if (req_to_token && rtt_stride < 1) return WMTP_EINVAL;
    windowed = windowed ? 1 : 0;
    // kIndexPerThreadLong entries per thread on long rows, up to 8192 CTAs per row.
    constexpr int kThreads = 256;
    const bool long_rows = stride >= kIndexLongRow;
    const int per = long_rows ? kIndexPerThreadLong : 1;
    int64_t gx = (stride + kThreads * per - 1) / (kThreads * per);
    if (gx > 8192) gx = 8192;
    PdlLaunch L(dim3((unsigned)gx, (unsigned)(gamma * B)), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, long_rows ? build_indices_kernel<kIndexPerThreadLong> : build_indices_kernel<1>, seq_lens, B, n_sink, window, depth,
                              tree_k, windowed, req_to_token, req_pool_idx, rtt_stride, ring_base,
                              table, stride, lens, static_cast<const int32_t *>(nullptr)) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

wmtp_status wmtp_build_far_indices(const int32_t *seq_lens, int32_t B, int32_t gamma,
                                   int32_t n_sink, int32_t window, const int32_t *req_to_token,
                                   const int32_t *req_pool_idx, int64_t rtt_stride, int32_t *table,
                                   int64_t stride, int32_t *lens, void *stream) {
    if (B < 0 || gamma < 0 || n_sink < 0 || window < 1 || stride < 1) return WMTP_EINVAL;
    if ((int64_t)gamma * B > 65535) return WMTP_EINVAL;
    if (B == 0 || gamma == 0) return WMTP_OK;
    if (!seq_lens || !table || !lens || !req_to_token || rtt_stride < 1) return WMTP_EINVAL;
    constexpr int kThreads = 256;
    const bool long_rows = stride >= kIndexLongRow;
    const int per = long_rows ? kIndexPerThreadLong : 1;
    int64_t gx = (stride + kThreads * per - 1) / (kThreads * per);
    if (gx > 8192) gx = 8192;
    PdlLaunch L(dim3((unsigned)gx, (unsigned)(gamma * B)), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, long_rows ? build_indices_kernel<kIndexPerThreadLong> : build_indices_kernel<1>,
                              seq_lens, B, n_sink, window, 1, 1, 2, req_to_token, req_pool_idx, rtt_stride,
                              static_cast<const int32_t *>(nullptr), table, stride, lens,
                              static_cast<const int32_t *>(nullptr)) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

wmtp_status wmtp_build_extend_indices(const int32_t *seq_lens, const int32_t *n_new, int32_t B,
                                      int32_t n_sink, int32_t window, int32_t depth,
                                      int32_t tree_k, int32_t windowed,
                                      const int32_t *req_to_token,
                                      const int32_t *req_pool_idx, int64_t rtt_stride,
                                      const int32_t *ring_base, int32_t *table,
                                      int64_t stride, int32_t *lens, void *stream) {
    if (B < 0 || n_sink < 0 || window < 1 || depth < 1 || tree_k < 1 || stride < 1 || B > 65535)
        return WMTP_EINVAL;
    if (B == 0) return WMTP_OK;
    if (!seq_lens || !n_new || !table || !lens) return WMTP_EINVAL;
    if (!req_to_token && !ring_base) return WMTP_EINVAL;
    if (req_to_token && rtt_stride < 1) return WMTP_EINVAL;
    windowed = windowed ? 1 : 0;
    constexpr int kThreads = 256;
    const bool long_rows = stride >= kIndexLongRow;
    const int per = long_rows ? kIndexPerThreadLong : 1;
    int64_t gx = (stride + kThreads * per - 1) / (kThreads * per);
    if (gx > 8192) gx = 8192;
    PdlLaunch L(dim3((unsigned)gx, (unsigned)B), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, long_rows ? build_indices_kernel<kIndexPerThreadLong> : build_indices_kernel<1>, seq_lens, B, n_sink, window, depth,
                              tree_k, windowed, req_to_token, req_pool_idx, rtt_stride, ring_base,
                              table, stride, lens, n_new) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

wmtp_status wmtp_ring_map(const int32_t *ring_base, const int32_t *pos,
                          const int32_t *branch, const int32_t *req_of, int32_t n,
                          int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k,
                          int32_t *slots, void *stream) {
    if (n < 0 || n_sink < 0 || window < 1 || depth < 1 || tree_k < 1) return WMTP_EINVAL;
    if (n == 0) return WMTP_OK;
    if (!ring_base || !pos || !req_of || !slots) return WMTP_EINVAL;
    constexpr int kThreads = 256;
    PdlLaunch L(dim3((unsigned)((n + kThreads - 1) / kThreads)), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, ring_map_kernel, ring_base, pos, branch, req_of, n, n_sink,
                              window, depth, tree_k, slots) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

wmtp_status wmtp_append_kv(const uint16_t *k_new, const uint16_t *v_new,
                           const int32_t *slots, int32_t n, int32_t H_kv, int32_t D,
                           uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots,
                           void *stream) {
    if (n < 0 || H_kv < 1 || D < 1 || (D % 8) != 0 || num_slots < 0) return WMTP_EINVAL;
    if (n == 0) return WMTP_OK;
    if (!k_new || !v_new || !slots || !k_pool || !v_pool) return WMTP_EINVAL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return WMTP_EINVAL;
    const int32_t chunks = H_kv * D / 8;
    const int64_t total = (int64_t)n * chunks;
    constexpr int kThreads = 256;
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    PdlLaunch L(dim3((unsigned)blocks), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, append_kv_kernel, reinterpret_cast<const uint4 *>(k_new),
                              reinterpret_cast<const uint4 *>(v_new), slots, total, chunks,
                              reinterpret_cast<uint4 *>(k_pool), reinterpret_cast<uint4 *>(v_pool),
                              num_slots) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"

extern "C" {

wmtp_status wmtp_append_kv_fp8(const uint16_t *k_new, const uint16_t *v_new,
                               const int32_t *slots, int32_t n, int32_t H_kv, int32_t D,
                               const float *k_scale, const float *v_scale, uint8_t *k_pool,
                               uint8_t *v_pool, int64_t num_slots, void *stream) {
    if (n < 0 || H_kv < 1 || D < 1 || (D % 16) != 0 || num_slots < 0) return WMTP_EINVAL;
    if (n == 0) return WMTP_OK;
    if (!k_new || !v_new || !slots || !k_scale || !v_scale || !k_pool || !v_pool) return WMTP_EINVAL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return WMTP_EINVAL;
    const int32_t chunks = H_kv * D / 8;
    const int64_t total = (int64_t)n * chunks;
    constexpr int kThreads = 256;
    const int64_t blocks = (total + kThreads - 1) / kThreads;
    PdlLaunch L(dim3((unsigned)blocks), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, append_kv_fp8_kernel, reinterpret_cast<const uint4 *>(k_new),
                              reinterpret_cast<const uint4 *>(v_new), slots, total, chunks, D / 8, k_scale,
                              v_scale, reinterpret_cast<uint2 *>(k_pool), reinterpret_cast<uint2 *>(v_pool),
                              num_slots) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"

extern "C" {

wmtp_status wmtp_prefill_keep_positions(const int32_t *seq_lens, int32_t B, int32_t n_sink,
                                        int32_t window, int32_t *positions, int64_t stride,
                                        int32_t *counts, void *stream) {
    if (B < 0 || n_sink < 0 || window < 1 || stride < 1 || B > 65535) return WMTP_EINVAL;
    if (B == 0) return WMTP_OK;
    if (!seq_lens || !positions || !counts) return WMTP_EINVAL;
    constexpr int kThreads = 256;
    const int64_t need = (int64_t)n_sink + window < stride ? (int64_t)n_sink + window : stride;
    int64_t gx = (need + kThreads - 1) / kThreads;
    if (gx < 1) gx = 1;
    PdlLaunch L(dim3((unsigned)gx, (unsigned)B), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, keep_positions_kernel, seq_lens, n_sink, window, positions, stride,
                              counts) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

wmtp_status wmtp_ring_fill(const uint16_t *k_rows, const uint16_t *v_rows, const int32_t *seq_lens,
                           int32_t B, int64_t stride, int32_t H_kv, int32_t D, const int32_t *ring_base,
                           int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k, uint16_t *k_pool,
                           uint16_t *v_pool, int64_t num_slots, void *stream) {
    if (B < 0 || B > 65535 || stride < 1 || H_kv < 1 || D < 1 || (D % 8) != 0 || n_sink < 0 || window < 1 ||
        depth < 1 || tree_k < 1 || num_slots < 0)
        return WMTP_EINVAL;
    if (B == 0) return WMTP_OK;
    if (!k_rows || !v_rows || !seq_lens || !ring_base || !k_pool || !v_pool) return WMTP_EINVAL;
    if (!aligned16(k_rows) || !aligned16(v_rows) || !aligned16(k_pool) || !aligned16(v_pool)) return WMTP_EINVAL;
    const int32_t chunks = H_kv * D / 8;
    const int64_t rows = (int64_t)n_sink + window < stride ? (int64_t)n_sink + window : stride;
    constexpr int kThreads = 256;
    const int64_t gx = (rows * chunks + kThreads - 1) / kThreads;
    PdlLaunch L(dim3((unsigned)gx, (unsigned)B), dim3(kThreads), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, ring_fill_kernel, reinterpret_cast<const uint4 *>(k_rows),
                              reinterpret_cast<const uint4 *>(v_rows), seq_lens, ring_base, n_sink, window, depth,
                              tree_k, stride, chunks, reinterpret_cast<uint4 *>(k_pool),
                              reinterpret_cast<uint4 *>(v_pool), num_slots) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"
