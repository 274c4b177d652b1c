// wmtp_tree.cu -- tree-draft attention over the ring for sm_103a.
//
// Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
// Million-Token Context" (arXiv 2607.21535), §7 "Compatibility with tree
// speculation": windowing changes only which KV the draft reads, not the
// tree; a tree of width k reserves n_sink + W + d*k ring slots and its
// candidates share the sink + window prefix and diverge over the last d
// positions.  Reading used here (the pages leave the tree open): node
// (branch b, depth i) of a request with committed length S sits at position
// S + i and attends keep(S + i + 1) of App. A's pseudocode, with the draft
// positions S..S+i taken from its own branch.  For k = 1 this is the chain.
//
// Kernel design (one CTA = 112 query rows x one key chunk of one request and
// KV head):
//   * the request's key list is implicit: sinks || committed window of the
//     shallowest node || the k*d draft nodes, with ring slots computed in the
//     kernel (no table read);
//   * all 224 query rows of a KV head (28 nodes x 8 heads at k=4, d=7) form a
//     dense contraction: rows are the MMA M dimension (16 per warp, 7 warps),
//     keys N, head dim K, on mma.sync bf16 with fp32 accumulation;
//   * K/V tiles of 64 keys are gathered by all warps with 16-byte cp.async
//     into padded shared memory (two stages); Q rows stay in shared memory;
//   * a per-(row, key) predicate applies the tree-causal mask; online softmax
//     in base 2; the weights are split into bf16 head + tail for PV;
//   * key chunks are split over CTAs; the last CTA of a (request, KV head,
//     row block) merges the partials from the workspace in split order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"
#include "wmtp_ring.cuh"

namespace wmtp {
namespace {

__device__ int32_t g_tree_error = 0;

__device__ __forceinline__ void latch(int32_t code) { atomicCAS(&g_tree_error, 0, code); }

constexpr int kWarps = 7;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = kWarps * 16;  // query rows (node, head) per CTA
constexpr int kTileKeys = 64;
constexpr int kStages = 2;
constexpr int kMaxTreeSplits = 64;
constexpr int kTcRows = 128;  // query rows per CTA of the tcgen05 kernel
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct TCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kPitch = kRowBytes + 16;  // padded: conflict-free ldmatrix
    static constexpr int kQBytes = kRowsPerCta * kPitch;
    static constexpr int kTileBytes = kTileKeys * kPitch;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
    static constexpr int kKVOffset = kQBytes;
    static constexpr int kFlagOffset = kKVOffset + kStages * kStageBytes;
    static constexpr int kSmemBytes = kFlagOffset + 16;
    static_assert(kRowsPerCta * kMaxTreeSplits * 4 <= kStages * kStageBytes, "merge weights must fit");
};

struct TreeWs {
    int32_t *counters;  // [B][H_kv][row blocks]
    float *lse_part;    // [B][H_kv][R][n_split], base 2
    float *o_part;      // [B][H_kv][R][n_split][D]
};

__host__ __device__ inline size_t align256t(size_t x) { return (x + 255) & ~size_t(255); }

inline size_t tree_ws_bytes(int64_t B, int64_t H_kv, int64_t R, int64_t n_rb, int D, int n_split) {
    if (n_split <= 1) return 0;
    return align256t(B * H_kv * n_rb * 4) + align256t(B * H_kv * R * n_split * 4) +
           (size_t)B * H_kv * R * n_split * D * 4;
}

// The request's key list: sinks [0, ns), committed window [lo0, S) of the
// shallowest node (all of [0, S) when no node is windowed yet), then the
// n_nodes draft nodes (branch-major).
struct Geo {
    int64_t S, ns, lo0, Uc, U;
};

__device__ __forceinline__ Geo geometry(int64_t S, int n_sink, int window, int n_nodes) {
    Geo g;
    g.S = S;
    g.ns = S < n_sink ? S : n_sink;
    const bool windowed0 = S + 1 > (int64_t)n_sink + window;
    g.lo0 = windowed0 ? S + 1 - window : g.ns;
    g.Uc = g.ns + (S - g.lo0);
    g.U = g.Uc + n_nodes;
    return g;
}

// Logical position and branch of entry e (< U) of the key list.
__device__ __forceinline__ void entry_pos(const Geo &g, int64_t e, int depth, int64_t &p,
                                          int &br, int &dep) {
    if (e < g.Uc) {
        p = e < g.ns ? e : g.lo0 + (e - g.ns);
        br = 0;
        dep = -1;
    } else {
        const int64_t n = e - g.Uc;
        br = (int)(n / depth);
        dep = (int)(n - (int64_t)br * depth);
        p = g.S + dep;
    }
}

// A query row: node (branch, depth); keys below `lo` other than sinks are
// outside its window (lo = 0 when its key set is not windowed).
struct RowInfo {
    bool live;
    int br, dep;
    int64_t lo;
};

__device__ __forceinline__ bool visible(const RowInfo &rw, int64_t p, int br, int dep, int n_sink) {
    if (!rw.live) return false;
    const bool in_window = p < n_sink || p >= rw.lo;
    if (dep < 0) return in_window;                        // committed key
    return br == rw.br && dep <= rw.dep && in_window;     // draft node on its own path
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) tree_decode_kernel(
    const __nv_bfloat16 *__restrict__ q, int32_t H_q, int32_t H_kv, int32_t G, int32_t n_nodes,
    const __nv_bfloat16 *__restrict__ k_pool, const __nv_bfloat16 *__restrict__ v_pool,
    int64_t num_slots, const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ ring_base,
    int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k, float scale_log2,
    float *__restrict__ out, float *__restrict__ lse, TreeWs ws, int32_t n_split, int32_t n_rb) {
    using C = TCfg<D>;
    constexpr int KD = D / 16;
    constexpr int kChunks = C::kRowBytes / 16;
    extern __shared__ __align__(128) uint8_t smem[];
    volatile int32_t *flags = reinterpret_cast<volatile int32_t *>(smem + C::kFlagOffset);

    griddep_launch_dependents();
    griddep_wait();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int split = blockIdx.x;
    const int g = blockIdx.y % H_kv;
    const int rb = blockIdx.y / H_kv;
    const int64_t b = blockIdx.z;
    const int R = n_nodes * G;

    int64_t S = seq_lens[b];
    if (S < 0) {
        if (tid == 0) latch(WMTP_DEV_ARG_RANGE);
        S = 0;
    }
    const int64_t base = ring_base[b];
    const Geo geo = geometry(S, n_sink, window, n_nodes);
    int64_t chunk = (geo.U + n_split - 1) / n_split;
    chunk = (chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
    const int64_t start = (int64_t)split * chunk;
    const int64_t cnt = geo.U - start < 0 ? 0 : (geo.U - start < chunk ? geo.U - start : chunk);
    const int n_tiles = (int)((cnt + kTileKeys - 1) / kTileKeys);

    // ------------------------------------------------- Q rows -> smem
    const uint32_t q_addr = smem_addr(smem);
    const uint64_t keep = l2_policy_evict_last();
    for (int idx = tid; idx < kRowsPerCta * kChunks; idx += kThreads) {
        const int i = idx / kChunks, c16 = idx - i * kChunks;
        const int rq = rb * kRowsPerCta + i;
        const bool live = rq < R;
        const int t = live ? rq / G : 0;
        const int h = g * G + (live ? rq % G : 0);
        const __nv_bfloat16 *src = q + ((b * n_nodes + t) * H_q + h) * (int64_t)D + c16 * 8;
        cp_async_16(q_addr + i * C::kPitch + c16 * 16, src, live ? 16u : 0u, keep);
    }

    // ------------------------------------------------- K/V gathers
    const uint8_t *kbase = reinterpret_cast<const uint8_t *>(k_pool) + (size_t)g * C::kRowBytes;
    const uint8_t *vbase = reinterpret_cast<const uint8_t *>(v_pool) + (size_t)g * C::kRowBytes;
    const size_t slot_bytes = (size_t)H_kv * C::kRowBytes;
    const uint32_t kv_addr = smem_addr(smem + C::kKVOffset);
    auto issue = [&](int t, int st) {
        const uint32_t kdst = kv_addr + st * C::kStageBytes;
        const uint32_t vdst = kdst + C::kTileBytes;
        for (int k = warp; k < kTileKeys; k += kWarps) {
            const int64_t kk = (int64_t)t * kTileKeys + k;
            bool ok = kk < cnt;
            int64_t slot = 0;
            if (ok) {
                int64_t p;
                int br, dep;
                entry_pos(geo, start + kk, depth, p, br, dep);
                slot = ring_slot(base, p, br, n_sink, window, depth, tree_k);
                if (slot < 0 || slot >= num_slots) {
                    ok = false;
                    if (lane == 0) latch(WMTP_DEV_SLOT_RANGE);
                }
            }
            const uint8_t *ks = kbase + (ok ? (size_t)slot * slot_bytes : 0);
            const uint8_t *vs = vbase + (ok ? (size_t)slot * slot_bytes : 0);
            for (int c16 = lane; c16 < kChunks; c16 += 32) {
                cp_async_16(kdst + k * C::kPitch + c16 * 16, ks + c16 * 16, ok ? 16u : 0u, keep);
                cp_async_16(vdst + k * C::kPitch + c16 * 16, vs + c16 * 16, ok ? 16u : 0u, keep);
            }
        }
    };

    if (n_tiles > 0) issue(0, 0);
    cp_async_commit();  // Q rows + tile 0

    // ------------------------------------------------- this thread's rows
    const int r = lane >> 2, c = lane & 3;
    RowInfo rows[2];
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        const int rq = rb * kRowsPerCta + warp * 16 + r + 8 * hi;
        RowInfo &rw = rows[hi];
        rw.live = rq < R;
        const int t = rw.live ? rq / G : 0;
        rw.br = t / depth;
        rw.dep = t - rw.br * depth;
        const int64_t kv = S + rw.dep + 1;
        rw.lo = kv > (int64_t)n_sink + window ? kv - window : 0;
    }

    float o[D / 8][4];
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    const uint32_t a_base = q_addr + (warp * 16 + (lane & 15)) * C::kPitch + (lane >> 4) * 16;
    const uint32_t kb_off = ((lane & 7) + ((lane >> 4) << 3)) * C::kPitch + ((lane >> 3) & 1) * 16;
    const uint32_t vb_off = ((lane & 7) + (((lane >> 3) & 1) << 3)) * C::kPitch + (lane >> 4) * 16;

    for (int it = 0; it < n_tiles; ++it) {
        if (it + 1 < n_tiles) issue(it + 1, (it + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const uint32_t kt = kv_addr + (it & 1) * C::kStageBytes;
        const uint32_t vt = kt + C::kTileBytes;

        // S = Q K^T for 16 rows x 64 keys (8 n-tiles of 8 keys)
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(a_base + kd * 32, a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t x0, x1, x2, x3;
                ldsm_x4(kt + np * 16 * C::kPitch + kb_off + kd * 32, x0, x1, x2, x3);
                mma_bf16_16816(s[2 * np], a0, a1, a2, a3, x0, x1);
                mma_bf16_16816(s[2 * np + 1], a0, a1, a2, a3, x2, x3);
            }
        }

        // tree-causal mask, online softmax (rows r and r+8 of this warp)
        const int64_t tile_e0 = start + (int64_t)it * kTileKeys;
        const int64_t tile_cnt = cnt - (int64_t)it * kTileKeys;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int kk = nt * 8 + 2 * c + j;
                bool v0 = false, v1 = false;
                if (kk < tile_cnt) {
                    int64_t p;
                    int br, dep;
                    entry_pos(geo, tile_e0 + kk, depth, p, br, dep);
                    v0 = visible(rows[0], p, br, dep, n_sink);
                    v1 = visible(rows[1], p, br, dep, n_sink);
                }
                s[nt][j] = v0 ? s[nt][j] * scale_log2 : -INFINITY;
                s[nt][2 + j] = v1 ? s[nt][2 + j] * scale_log2 : -INFINITY;
                mx[0] = fmaxf(mx[0], s[nt][j]);
                mx[1] = fmaxf(mx[1], s[nt][2 + j]);
            }
        }
        float alpha[2], muse[2];
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            mx[hi] = fmaxf(mx[hi], __shfl_xor_sync(0xffffffffu, mx[hi], 1));
            mx[hi] = fmaxf(mx[hi], __shfl_xor_sync(0xffffffffu, mx[hi], 2));
            const float mn = fmaxf(m[hi], mx[hi]);
            muse[hi] = mn == -INFINITY ? 0.f : mn;
            alpha[hi] = exp2f(m[hi] - muse[hi]);
            m[hi] = mn;
        }
        float rs[2] = {0.f, 0.f};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            s[nt][0] = exp2f(s[nt][0] - muse[0]);
            s[nt][1] = exp2f(s[nt][1] - muse[0]);
            s[nt][2] = exp2f(s[nt][2] - muse[1]);
            s[nt][3] = exp2f(s[nt][3] - muse[1]);
            rs[0] += s[nt][0] + s[nt][1];
            rs[1] += s[nt][2] + s[nt][3];
        }
        l[0] = l[0] * alpha[0] + rs[0];
        l[1] = l[1] * alpha[1] + rs[1];
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) {
                o[nt][0] *= alpha[0];
                o[nt][1] *= alpha[0];
                o[nt][2] *= alpha[1];
                o[nt][3] *= alpha[1];
            }
        }

        // O += P V, P split into bf16 head + tail sharing each V fragment
#pragma unroll
        for (int kk16 = 0; kk16 < 4; ++kk16) {
            const float *pa = s[2 * kk16], *pb = s[2 * kk16 + 1];
            const uint32_t h0 = pack_bf16x2(pa[0], pa[1]), h1 = pack_bf16x2(pa[2], pa[3]);
            const uint32_t h2 = pack_bf16x2(pb[0], pb[1]), h3 = pack_bf16x2(pb[2], pb[3]);
            const uint32_t t0 = pack_bf16x2(pa[0] - bf16_lo_to_f32(h0), pa[1] - bf16_hi_to_f32(h0));
            const uint32_t t1 = pack_bf16x2(pa[2] - bf16_lo_to_f32(h1), pa[3] - bf16_hi_to_f32(h1));
            const uint32_t t2 = pack_bf16x2(pb[0] - bf16_lo_to_f32(h2), pb[1] - bf16_hi_to_f32(h2));
            const uint32_t t3 = pack_bf16x2(pb[2] - bf16_lo_to_f32(h3), pb[3] - bf16_hi_to_f32(h3));
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t y0, y1, y2, y3;
                ldsm_x4_trans(vt + kk16 * 16 * C::kPitch + vb_off + dp * 32, y0, y1, y2, y3);
                mma_bf16_16816(o[2 * dp], h0, h1, h2, h3, y0, y1);
                mma_bf16_16816(o[2 * dp + 1], h0, h1, h2, h3, y2, y3);
                mma_bf16_16816(o[2 * dp], t0, t1, t2, t3, y0, y1);
                mma_bf16_16816(o[2 * dp + 1], t0, t1, t2, t3, y2, y3);
            }
        }
        __syncthreads();  // the stage is overwritten by the next issue
    }
    cp_async_wait<0>();

#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        l[hi] += __shfl_xor_sync(0xffffffffu, l[hi], 1);
        l[hi] += __shfl_xor_sync(0xffffffffu, l[hi], 2);
    }

    // ------------------------------------------------- partial or final rows
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        if (!rows[hi].live) continue;
        const int rq = rb * kRowsPerCta + warp * 16 + r + 8 * hi;
        const int t = rq / G, h = g * G + rq % G;
        const float inv = l[hi] > 0.f ? 1.f / l[hi] : 0.f;
        const float lse2 = l[hi] > 0.f ? m[hi] + log2f(l[hi]) : -INFINITY;
        float *dst;
        if (n_split == 1) {
            const int64_t orow = (b * n_nodes + t) * H_q + h;
            dst = out + orow * D;
            if (c == 0 && lse) lse[orow] = lse2 * kLn2;
        } else {
            const int64_t prow = ((b * H_kv + g) * R + rq) * n_split + split;
            dst = ws.o_part + prow * D;
            if (c == 0) ws.lse_part[prow] = lse2;
        }
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt)
            *reinterpret_cast<float2 *>(dst + nt * 8 + 2 * c) =
                make_float2(o[nt][2 * hi] * inv, o[nt][2 * hi + 1] * inv);
    }
    if (n_split == 1) return;

    // ------------------------------------------ ticket; the last CTA merges
    __threadfence();
    __syncthreads();
    const int64_t cidx = (b * H_kv + g) * n_rb + rb;
    if (tid == 0) {
        const int32_t ticket = atomicAdd(&ws.counters[cidx], 1);
        flags[0] = (ticket == n_split - 1);
    }
    __syncthreads();
    if (!flags[0]) return;
    __threadfence();

    const int row0 = rb * kRowsPerCta;
    const int n_rows = R - row0 < kRowsPerCta ? R - row0 : kRowsPerCta;
    float *wts = reinterpret_cast<float *>(smem + C::kKVOffset);  // [rows][n_split]
    const int64_t prow0 = (b * H_kv + g) * R + row0;
    for (int e = tid; e < n_rows * n_split; e += kThreads)
        wts[e] = __ldcg(ws.lse_part + prow0 * n_split + e);
    __syncthreads();
    for (int i = tid; i < n_rows; i += kThreads) {
        float *w = wts + i * n_split;
        float M = -INFINITY;
        for (int s2 = 0; s2 < n_split; ++s2) M = fmaxf(M, w[s2]);
        float sum = 0.f;
        if (M != -INFINITY)
            for (int s2 = 0; s2 < n_split; ++s2) sum += w[s2] == -INFINITY ? 0.f : exp2f(w[s2] - M);
        const float lt = sum > 0.f ? M + log2f(sum) : -INFINITY;
        for (int s2 = 0; s2 < n_split; ++s2)
            w[s2] = (sum > 0.f && w[s2] != -INFINITY) ? exp2f(w[s2] - lt) : 0.f;
        const int rq = row0 + i;
        const int64_t orow = (b * n_nodes + rq / G) * H_q + g * G + rq % G;
        if (lse) lse[orow] = lt * kLn2;
    }
    __syncthreads();
    constexpr int D4 = D / 4;
    for (int e = tid; e < n_rows * D4; e += kThreads) {
        const int i = e / D4, d4 = e - i * D4;
        const float *w = wts + i * n_split;
        const float4 *op = reinterpret_cast<const float4 *>(ws.o_part + (prow0 + i) * n_split * D) + d4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < n_split; ++s2) {
            const float4 v = __ldcg(op + (int64_t)s2 * D4);
            acc.x += w[s2] * v.x;
            acc.y += w[s2] * v.y;
            acc.z += w[s2] * v.z;
            acc.w += w[s2] * v.w;
        }
        const int rq = row0 + i;
        const int64_t orow = (b * n_nodes + rq / G) * H_q + g * G + rq % G;
        reinterpret_cast<float4 *>(out + orow * D)[d4] = acc;
    }
    if (tid == 0) ws.counters[cidx] = 0;  // ready for the next call
}

template <int D>
wmtp_status launch_tree(const uint16_t *q, int32_t B, int32_t H_q, int32_t H_kv,
                        const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                        const int32_t *seq_lens, const int32_t *ring_base, int32_t n_sink,
                        int32_t window, int32_t depth, int32_t tree_k, float scale, float *out,
                        float *lse, void *workspace, int32_t n_split, cudaStream_t stream) {
    using C = TCfg<D>;
    const int G = H_q / H_kv;
    const int n_nodes = tree_k * depth;
    const int R = n_nodes * G;
    const int n_rb = (R + kRowsPerCta - 1) / kRowsPerCta;
    static int opted_in[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WMTP_ECUDA;
    if (!opted_in[dev]) {
        if (cudaFuncSetAttribute(tree_decode_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return WMTP_ECUDA;
        opted_in[dev] = 1;
    }
    TreeWs ws{nullptr, nullptr, nullptr};
    if (n_split > 1) {
        uint8_t *p = static_cast<uint8_t *>(workspace);
        ws.counters = reinterpret_cast<int32_t *>(p);
        p += align256t((size_t)B * H_kv * n_rb * 4);
        ws.lse_part = reinterpret_cast<float *>(p);
        p += align256t((size_t)B * H_kv * R * n_split * 4);
        ws.o_part = reinterpret_cast<float *>(p);
    }
    PdlLaunch launch(dim3((unsigned)n_split, (unsigned)(H_kv * n_rb), (unsigned)B), dim3(kThreads),
                     C::kSmemBytes, stream);
    const cudaError_t err = cudaLaunchKernelEx(
        &launch.cfg, tree_decode_kernel<D>, reinterpret_cast<const __nv_bfloat16 *>(q), H_q, H_kv,
        G, n_nodes, reinterpret_cast<const __nv_bfloat16 *>(k_pool),
        reinterpret_cast<const __nv_bfloat16 *>(v_pool), num_slots, seq_lens, ring_base, n_sink,
        window, depth, tree_k, scale * 1.4426950408889634f, out, lse, ws, n_split, n_rb);
    return err == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

}  // namespace

cudaError_t read_tree_error(int32_t *code, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(code, g_tree_error, sizeof(int32_t));
    if (err != cudaSuccess || !clear) return err;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_tree_error, &zero, sizeof(int32_t));
}

}  // namespace wmtp

using namespace wmtp;

extern "C" {

size_t wmtp_tree_workspace_bytes(int32_t B, int32_t H_q, int32_t H_kv, int32_t D, int32_t depth,
                                 int32_t tree_k, int32_t n_split) {
    if (B < 0 || H_kv < 1 || H_q < H_kv || D < 1 || depth < 1 || tree_k < 1 || n_split < 1) return 0;
    const int64_t R = (int64_t)tree_k * depth * (H_q / H_kv);
    return tree_tc_workspace_bytes(B, H_kv, R, D, n_split);
}

int32_t wmtp_tree_num_splits(int32_t B, int32_t H_q, int32_t H_kv, int32_t depth, int32_t tree_k,
                             int32_t n_sink, int32_t window) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (B < 1 || H_kv < 1 || H_q < H_kv || depth < 1 || tree_k < 1) return 1;
    const int64_t R = (int64_t)tree_k * depth * (H_q / H_kv);
    const int64_t n_rb = (R + kTcRows - 1) / kTcRows;
    const int64_t per_split = (int64_t)B * H_kv * n_rb;
    const int64_t keys = (int64_t)n_sink + window + (int64_t)tree_k * depth;
    int64_t n = sms / per_split;
    const int64_t by_len = (keys + kTileKeys - 1) / kTileKeys / 4;  // >= four tiles per split
    if (n > by_len) n = by_len;
    if (n < 1) n = 1;
    if (n > kMaxTreeSplits) n = kMaxTreeSplits;
    return (int32_t)n;
}

wmtp_status wmtp_tree_draft_attn(const uint16_t *q, int32_t B, int32_t H_q, int32_t H_kv,
                                 int32_t D, const uint16_t *k_pool, const uint16_t *v_pool,
                                 int64_t num_slots, const int32_t *seq_lens,
                                 const int32_t *ring_base, int32_t n_sink, int32_t window,
                                 int32_t depth, int32_t tree_k, float scale, float *out,
                                 float *lse, void *workspace, size_t workspace_bytes,
                                 int32_t n_split, void *stream) {
    if (B < 0 || H_q < 1 || H_kv < 1 || (H_q % H_kv) != 0) return WMTP_EINVAL;
    if (D != 128 && D != 256) return WMTP_EINVAL;
    if (n_sink < 0 || window < 1 || depth < 1 || tree_k < 1) return WMTP_EINVAL;
    if (n_split < 1 || n_split > kMaxTreeSplits || num_slots < 0) return WMTP_EINVAL;
    if (depth > 255) return WMTP_EINVAL;
    const int64_t R = (int64_t)tree_k * depth * (H_q / H_kv);
    const int64_t n_rb = (R + kTcRows - 1) / kTcRows;
    if (R > (1 << 20) || (int64_t)H_kv * n_rb > 65535 || B > 65535) return WMTP_EINVAL;
    if (B == 0) return WMTP_OK;
    if (!q || !k_pool || !v_pool || !seq_lens || !ring_base || !out) return WMTP_EINVAL;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return WMTP_EINVAL;
    if (n_split > 1) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return WMTP_EINVAL;
        if (workspace_bytes < tree_tc_workspace_bytes(B, H_kv, R, D, n_split)) return WMTP_ECAPACITY;
    }
    return tree_tc_launch(q, B, H_q, H_kv, D, k_pool, v_pool, num_slots, seq_lens, ring_base,
                          n_sink, window, depth, tree_k, scale, out, lse, workspace, n_split,
                          as_stream(stream));
}

}  // extern "C"
