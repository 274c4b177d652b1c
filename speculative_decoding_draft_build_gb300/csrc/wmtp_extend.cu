// wmtp_extend.cu -- draft-extend attention that serves all of a request's
// new tokens from one read of its keys, for sm_103a.
//
// Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
// Million-Token Context" (arXiv 2607.21535), §4 Mechanism and App. A: draft
// step t of a request with committed length S sees keep(S + t + 1).  The
// draft forward over the n tokens the request accepted computes all n steps
// at once; their key sets differ only in their last few positions, so the
// union of the n sets is one table row (wmtp_build_extend_indices) and each
// token masks the union entries outside its own set.
//
// Kernel design (one CTA = one chunk of one request's union row for one KV
// head, all of its tokens):
//   * eight warps gather each 64-key tile once (each warp 8 keys' K and V
//     rows with 16-byte cp.async into a padded tile, slot numbers fetched
//     tiles ahead into a shared-memory ring), then every warp computes one
//     token over the whole tile: warp t owns token t.  The K/V bytes of a
//     request are read from memory once instead of once per token.
//   * per token the math is the decode kernel's: QK^T on mma.sync bf16 with
//     keys as M and the GQA group's query heads as N, online softmax in base
//     2, P split into bf16 head + tail and transposed with movmatrix into the
//     PV B operand, O^T accumulated in fp32 registers.
//   * splits of a (request, KV head) merge through the workspace: each split
//     writes its normalised partial per (token, head), takes a ticket, and
//     the last CTA merges every row in split order (no CTA waits on another).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"

namespace wmtp {
namespace {

__device__ int32_t g_extend_error = 0;

__device__ __forceinline__ void latch(int32_t code) { atomicCAS(&g_extend_error, 0, code); }

constexpr int kWarps = 8;                     // one token per warp
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 64;                     // keys per tile
constexpr int kKeysPerWarp = kTile / kWarps;  // keys each warp gathers
constexpr int kStages = 3;
constexpr int kRingTiles = 2 * kStages;
constexpr int kMaxGroup = 8;
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct XCfg {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kPitch = kRowBytes + 16;  // conflict-free ldmatrix
    static constexpr int kTileBytes = kTile * kPitch;
    static constexpr int kStageBytes = 2 * kTileBytes;  // K rows, then V rows
    static constexpr int kTilesBytes = kStages * kStageBytes;
    static constexpr int kRingOffset = kTilesBytes;                         // int32 [ring tiles][kTile]
    static constexpr int kMaskOffset = kRingOffset + kRingTiles * kTile * 4;  // uint8 [stages][warps]
    static constexpr int kFlagOffset = kMaskOffset + kStages * kWarps;
    static constexpr int kSmemBytes = kFlagOffset + 16;
    // merge weights [tokens * group][splits] reuse the tile area
    static_assert(kMaxExtendTokens * kMaxGroup * kMaxExtendSplits * 4 <= kTilesBytes, "merge scratch");
};

// Workspace views (the split-order layout of wmtp_draft_decode_attn):
// counters [B * H_kv] (one per request and KV head), lse_part [rows][n_split]
// (base 2), o_part [rows][n_split][D]; rows = (b * n_q + t) * H_q + h.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) extend_kernel(
    const __nv_bfloat16 *__restrict__ q, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t G,
    const __nv_bfloat16 *__restrict__ k_pool, const __nv_bfloat16 *__restrict__ v_pool, int64_t num_slots,
    const int32_t *__restrict__ table, int64_t table_stride, const int32_t *__restrict__ lens,
    const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ n_new, int32_t n_sink, int32_t window,
    int32_t windowed, float scale_log2, float *__restrict__ out, float *__restrict__ lse,
    int32_t *__restrict__ counters, float *__restrict__ lse_part, float *__restrict__ o_part, int32_t n_split) {
    using C = XCfg<D>;
    constexpr int S = kStages;
    constexpr int R = kRingTiles;
    constexpr int KD = D / 16;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *masks = smem + C::kMaskOffset;
    volatile int32_t *flags = reinterpret_cast<volatile int32_t *>(smem + C::kFlagOffset);

    griddep_launch_dependents();
    griddep_wait();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int r = lane >> 2;  // MMA group: key row (QK) / output dim row (PV)
    const int c = lane & 3;   // query-head pair 2c, 2c+1
    const int tk = warp;      // this warp's token

    // Request geometry: union row length, committed length, tokens.
    int64_t L = lens[b];
    if (L < 0 || L > table_stride) {
        if (threadIdx.x == 0 && split == 0 && g == 0) latch(WMTP_DEV_LEN_RANGE);
        L = L < 0 ? 0 : table_stride;
    }
    int32_t nn = n_new[b];
    nn = nn < 0 ? 0 : (nn > n_q ? n_q : nn);
    const int64_t S_b = seq_lens[b];
    // union entry e -> position: e below n_sink (or a non-windowed union),
    // else lo_u + e - n_sink
    const int64_t kv_u = S_b + nn, w_u = (int64_t)window + (nn > 0 ? nn - 1 : 0);
    const bool win_u = windowed && kv_u > (int64_t)n_sink + w_u;
    const int64_t lo_u = kv_u - w_u;
    // this warp's token sees positions below kv_t and, when windowed, sinks
    // or positions from lo_t
    const int64_t kv_t = S_b + tk + 1;
    const bool win_t = windowed && kv_t > (int64_t)n_sink + window;
    const int64_t lo_t = kv_t - window;
    const bool active = tk < nn;

    // Query fragments of this warp's token (B operand of QK^T).
    uint32_t qf[KD][2];
    {
        const bool live = active && r < G;
        const __nv_bfloat16 *qrow = q + ((b * n_q + (active ? tk : 0)) * H_q + (int64_t)g * G + (live ? r : 0)) * D;
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            qf[kd][0] = live ? __ldg(reinterpret_cast<const uint32_t *>(qrow + kd * 16 + 2 * c)) : 0u;
            qf[kd][1] = live ? __ldg(reinterpret_cast<const uint32_t *>(qrow + kd * 16 + 2 * c + 8)) : 0u;
        }
    }

    // Chunk of this split (whole tiles), as in the decode kernel.
    const int64_t ch = (L + n_split - 1) / n_split;
    const int64_t chunk = (ch + kTile - 1) / kTile * kTile;
    const int64_t start = (int64_t)split * chunk;
    const int64_t cnt = L - start < 0 ? 0 : (L - start < chunk ? L - start : chunk);
    const int n_tiles = (int)((cnt + kTile - 1) / kTile);
    const int32_t *__restrict__ trow = table + b * table_stride + start;

    const uint64_t policy = l2_policy_evict_first();
    const uint8_t *kbase = reinterpret_cast<const uint8_t *>(k_pool) + (size_t)g * C::kRowBytes;
    const uint8_t *vbase = reinterpret_cast<const uint8_t *>(v_pool) + (size_t)g * C::kRowBytes;
    const size_t slot_bytes = (size_t)H_kv * C::kRowBytes;
    const int32_t *ring = reinterpret_cast<const int32_t *>(smem + C::kRingOffset);
    const uint32_t ring_addr = smem_addr(ring);
    const uint32_t tiles_addr = smem_addr(smem);

    // Slot numbers of tile t (this warp's 8 keys) into the ring.
    auto fetch_slots = [&](int t) {
        if (lane < kKeysPerWarp) {
            const int key = warp * kKeysPerWarp + lane;
            const int64_t k = (int64_t)t * kTile + key;
            const bool in = k < cnt;
            cp_async_4(ring_addr + ((t % R) * kTile + key) * 4,
                       in ? static_cast<const void *>(trow + k) : static_cast<const void *>(table), in ? 4u : 0u);
        }
    };
    // K/V gathers of tile t (stage t % S) for this warp's 8 keys.
    auto issue = [&](int t) {
        const int st = t % S;
        const int key0 = warp * kKeysPerWarp;
        const int32_t my_slot = lane < kKeysPerWarp ? ring[(t % R) * kTile + key0 + lane] : 0;
        const int64_t k = (int64_t)t * kTile + key0 + lane;
        const bool in = lane < kKeysPerWarp && k < cnt;
        const bool ok = in && my_slot >= 0 && my_slot < num_slots;
        if (in && !ok) latch(WMTP_DEV_SLOT_RANGE);
        const uint32_t vm = __ballot_sync(0xffffffffu, ok) & 0xffu;
        if (lane == 0) masks[st * kWarps + warp] = (uint8_t)vm;
        const uint32_t kdst = tiles_addr + st * C::kStageBytes;
        const uint32_t vdst = kdst + C::kTileBytes;
        constexpr int kLanesPerRow = C::kRowBytes / 16;  // 32 (D=256) or 16 (D=128)
        constexpr int kRowsPerInst = 32 / kLanesPerRow;
        const int sub = lane / kLanesPerRow;
        const int col = (lane % kLanesPerRow) * 16;
#pragma unroll
        for (int r0 = 0; r0 < kKeysPerWarp; r0 += kRowsPerInst) {
            const int kk = r0 + sub;
            const int32_t slot = __shfl_sync(0xffffffffu, my_slot, kk);
            const bool kv = (vm >> kk) & 1u;
            const size_t off = kv ? (size_t)slot * slot_bytes + col : 0;
            const int row = key0 + kk;
            cp_async_16(kdst + row * C::kPitch + col, kbase + off, kv ? 16u : 0u, policy);
            cp_async_16(vdst + row * C::kPitch + col, vbase + off, kv ? 16u : 0u, policy);
        }
    };

    // Prologue: slots of the first 2S-1 tiles, then K/V of the first S-1.
    for (int t = 0; t < 2 * S - 1 && t < n_tiles; ++t) fetch_slots(t);
    cp_async_commit();
    cp_async_wait<0>();
    __syncwarp();
#pragma unroll
    for (int t = 0; t < S - 1; ++t) {
        if (t < n_tiles) issue(t);
        cp_async_commit();
    }

    float o[KD][4];
#pragma unroll
    for (int dt = 0; dt < KD; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max, heads 2c and 2c+1 (base 2)
    float l0 = 0.f, l1 = 0.f;              // this thread's share of the running sums

    const uint32_t k_off = (uint32_t)((lane & 15) * C::kPitch + (lane >> 4) * 16);
    const uint32_t v_off = (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * C::kPitch + ((lane >> 3) & 1) * 16);

    for (int it = 0; it < n_tiles; ++it) {
        // Groups committed so far: slots, K/V of tiles 0..S-2, one per
        // iteration; all but the newest S-2 done makes tile `it` resident
        // for this thread; the barrier makes it resident for every warp and
        // frees the stage of tile it-1 for the next gathers.
        cp_async_wait<S - 2>();
        __syncthreads();
        if (it + S - 1 < n_tiles) issue(it + S - 1);
        if (it + 2 * S - 1 < n_tiles) fetch_slots(it + 2 * S - 1);
        cp_async_commit();
        if (!active) continue;
        const int st = it % S;
        const int64_t e0 = start + (int64_t)it * kTile;
        // visibility of keys mt*16 + r and mt*16 + r + 8 for this token
        bool vis[4][2];
        bool any = false;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int key = mt * 16 + r + hh * 8;
                const bool valid = (masks[st * kWarps + (key >> 3)] >> (key & 7)) & 1u;
                const int64_t e = e0 + key;
                const int64_t pos = (win_u && e >= n_sink) ? lo_u + (e - n_sink) : e;
                vis[mt][hh] = valid && pos < kv_t && (!win_t || pos < n_sink || pos >= lo_t);
                any |= vis[mt][hh];
            }
        }
        if (!__any_sync(0xffffffffu, any)) continue;
        const uint32_t kaddr = tiles_addr + st * C::kStageBytes + k_off;
        const uint32_t vaddr = tiles_addr + st * C::kStageBytes + C::kTileBytes + v_off;
        float sacc[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) sacc[mt][0] = sacc[mt][1] = sacc[mt][2] = sacc[mt][3] = 0.f;
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kaddr + mt * 16 * C::kPitch + kd * 32, a0, a1, a2, a3);
                mma_bf16_16816(sacc[mt], a0, a1, a2, a3, qf[kd][0], qf[kd][1]);
            }
        }
        // sacc[mt][0]: key mt*16+r, head 2c; [1]: head 2c+1; [2], [3]: key +8
        float x[4][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            x[mt][0] = vis[mt][0] ? sacc[mt][0] * scale_log2 : -INFINITY;
            x[mt][1] = vis[mt][0] ? sacc[mt][1] * scale_log2 : -INFINITY;
            x[mt][2] = vis[mt][1] ? sacc[mt][2] * scale_log2 : -INFINITY;
            x[mt][3] = vis[mt][1] ? sacc[mt][3] * scale_log2 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(x[mt][0], x[mt][2]));
            mx1 = fmaxf(mx1, fmaxf(x[mt][1], x[mt][3]));
        }
#pragma unroll
        for (int sh = 4; sh < 32; sh <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: a key is visible
        const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            x[mt][0] = exp2f(x[mt][0] - mn0);
            x[mt][1] = exp2f(x[mt][1] - mn1);
            x[mt][2] = exp2f(x[mt][2] - mn0);
            x[mt][3] = exp2f(x[mt][3] - mn1);
            ps0 += x[mt][0] + x[mt][2];
            ps1 += x[mt][1] + x[mt][3];
        }
        l0 = l0 * al0 + ps0;
        l1 = l1 * al1 + ps1;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // a running max moved
#pragma unroll
            for (int dt = 0; dt < KD; ++dt) {
                o[dt][0] *= al0;
                o[dt][1] *= al1;
                o[dt][2] *= al0;
                o[dt][3] *= al1;
            }
        }
        // PV over the four 16-key groups: P^T (bf16 head + tail, movmatrix)
        // as the B operand, V^T through ldmatrix.trans as A.
#pragma unroll
        for (int mt = 0; mt < 4; ++mt) {
            const uint32_t h01 = pack_bf16x2(x[mt][0], x[mt][1]), h23 = pack_bf16x2(x[mt][2], x[mt][3]);
            const uint32_t t01 = pack_bf16x2(x[mt][0] - bf16_lo_to_f32(h01), x[mt][1] - bf16_hi_to_f32(h01));
            const uint32_t t23 = pack_bf16x2(x[mt][2] - bf16_lo_to_f32(h23), x[mt][3] - bf16_hi_to_f32(h23));
            const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
            const uint32_t pl0 = movmatrix_trans(t01), pl1 = movmatrix_trans(t23);
#pragma unroll
            for (int dt = 0; dt < KD; ++dt) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(vaddr + mt * 16 * C::kPitch + dt * 32, a0, a1, a2, a3);
                mma_bf16_16816(o[dt], a0, a1, a2, a3, ph0, ph1);
                mma_bf16_16816(o[dt], a0, a1, a2, a3, pl0, pl1);
            }
        }
    }
    cp_async_wait<0>();

    // Row sums: add the shares of the 8 lanes that hold the same heads.
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }

    // ------------------------------------------- this split's rows (per warp)
    // Warp tk holds token tk's heads 2c, 2c+1 of the group; accumulator rows
    // r and r + 8 of group dt are dimensions 16dt + r and 16dt + r + 8.
    const int64_t row_t = (b * n_q + tk) * H_q + (int64_t)g * G;  // first head of the group
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    const float ls0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY, ls1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
    if (tk < n_q) {
        const int h0 = 2 * c, h1 = 2 * c + 1;
        float *dst0, *dst1;
        if (n_split == 1) {
            dst0 = out + (row_t + h0) * D;
            dst1 = out + (row_t + h1) * D;
        } else {
            dst0 = o_part + ((row_t + h0) * n_split + split) * D;
            dst1 = o_part + ((row_t + h1) * n_split + split) * D;
        }
#pragma unroll
        for (int dt = 0; dt < KD; ++dt) {
            if (h0 < G) {
                dst0[dt * 16 + r] = o[dt][0] * inv0;
                dst0[dt * 16 + r + 8] = o[dt][2] * inv0;
            }
            if (h1 < G) {
                dst1[dt * 16 + r] = o[dt][1] * inv1;
                dst1[dt * 16 + r + 8] = o[dt][3] * inv1;
            }
        }
        if (r == 0) {
            if (n_split == 1) {
                if (lse && h0 < G) lse[row_t + h0] = ls0 * kLn2;
                if (lse && h1 < G) lse[row_t + h1] = ls1 * kLn2;
            } else {
                if (h0 < G) lse_part[(row_t + h0) * n_split + split] = ls0;
                if (h1 < G) lse_part[(row_t + h1) * n_split + split] = ls1;
            }
        }
    }
    if (n_split == 1) return;

    // ------------------------------------------ ticket; the last CTA merges
    __threadfence();
    __syncthreads();
    int32_t *ctr = counters + b * H_kv + g;
    if (threadIdx.x == 0) flags[0] = (atomicAdd(ctr, 1) == n_split - 1);
    __syncthreads();
    if (!flags[0]) return;
    __threadfence();

    // Merge rows (t, h), t < n_q, h < G, in split order: lse = log2 sum_s
    // 2^lse_s, weights 2^(lse_s - lse) (the tile area holds the weights).
    const int rows = n_q * G;
    float *wts = reinterpret_cast<float *>(smem);  // [rows][n_split]
    const int tid = threadIdx.x;
    auto row_q = [&](int rr) { return (b * n_q + rr / G) * H_q + (int64_t)g * G + rr % G; };
    for (int e = tid; e < rows * n_split; e += kThreads) {
        const int rr = e / n_split, s2 = e - rr * n_split;
        wts[e] = __ldcg(lse_part + row_q(rr) * n_split + s2);
    }
    __syncthreads();
    for (int rr = warp; rr < rows; rr += kWarps) {
        float M = -INFINITY;
        for (int s2 = lane; s2 < n_split; s2 += 32) M = fmaxf(M, wts[rr * n_split + s2]);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
        float sum = 0.f;
        if (M != -INFINITY) {
            for (int s2 = lane; s2 < n_split; s2 += 32) {
                const float xv = wts[rr * n_split + s2];
                sum += xv == -INFINITY ? 0.f : exp2f(xv - M);
            }
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
        const float lse_tot = sum > 0.f ? M + log2f(sum) : -INFINITY;
        __syncwarp();
        for (int s2 = lane; s2 < n_split; s2 += 32) {
            const float xv = wts[rr * n_split + s2];
            wts[rr * n_split + s2] = (sum > 0.f && xv != -INFINITY) ? exp2f(xv - lse_tot) : 0.f;
        }
        if (lane == 0 && lse) lse[row_q(rr)] = lse_tot * kLn2;
    }
    __syncthreads();
    constexpr int D4 = D / 4;
    constexpr int kUnroll = 8;
    for (int e = tid; e < rows * D4; e += kThreads) {
        const int rr = e / D4, d4 = e - rr * D4;
        const int64_t rq = row_q(rr);
        const float4 *op = reinterpret_cast<const float4 *>(o_part + rq * n_split * D) + d4;
        const float *wh = wts + rr * n_split;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int s2 = 0;
        for (; s2 + kUnroll <= n_split; s2 += kUnroll) {
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) v[u] = __ldcg(op + (int64_t)(s2 + u) * D4);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float w = wh[s2 + u];
                acc.x += w * v[u].x;
                acc.y += w * v[u].y;
                acc.z += w * v[u].z;
                acc.w += w * v[u].w;
            }
        }
        for (; s2 < n_split; ++s2) {
            const float4 v = __ldcg(op + (int64_t)s2 * D4);
            const float w = wh[s2];
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        reinterpret_cast<float4 *>(out + rq * D)[d4] = acc;
    }
    if (tid == 0) *ctr = 0;  // ready for the next call
}

template <int D>
bool prepare_extend(int dev) {
    static int8_t done[64] = {};
    if (dev < 0 || dev >= 64) return false;
    if (done[dev]) return done[dev] > 0;
    const bool ok = cudaFuncSetAttribute(extend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         XCfg<D>::kSmemBytes) == cudaSuccess;
    cudaGetLastError();
    done[dev] = ok ? 1 : -1;
    return ok;
}

}  // namespace

cudaError_t read_extend_error(int32_t *code, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(code, g_extend_error, sizeof(int32_t));
    if (err != cudaSuccess || !clear) return err;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_extend_error, &zero, sizeof(int32_t));
}

wmtp_status extend_multi_launch(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t D,
                                const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                                const int32_t *table, int64_t table_stride, const int32_t *lens,
                                const int32_t *seq_lens, const int32_t *n_new, int32_t n_sink, int32_t window,
                                int32_t windowed, float scale, float *out, float *lse, int32_t *counters,
                                float *lse_part, float *o_part, int32_t n_split, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WMTP_ECUDA;
    if (!(D == 256 ? prepare_extend<256>(dev) : prepare_extend<128>(dev))) return WMTP_ECUDA;
    const float scale_log2 = scale * 1.4426950408889634f;
    PdlLaunch launch(dim3((unsigned)n_split, (unsigned)H_kv, (unsigned)B), dim3(kThreads),
                     D == 256 ? XCfg<256>::kSmemBytes : XCfg<128>::kSmemBytes, stream);
    const auto kern = D == 256 ? extend_kernel<256> : extend_kernel<128>;
    const cudaError_t err = cudaLaunchKernelEx(
        &launch.cfg, kern, reinterpret_cast<const __nv_bfloat16 *>(q), n_q, H_q, H_kv, H_q / H_kv,
        reinterpret_cast<const __nv_bfloat16 *>(k_pool), reinterpret_cast<const __nv_bfloat16 *>(v_pool),
        num_slots, table, table_stride, lens, seq_lens, n_new, n_sink, window, windowed, scale_log2, out, lse,
        counters, lse_part, o_part, n_split);
    return err == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

}  // namespace wmtp

using namespace wmtp;

extern "C" {

int32_t wmtp_extend_num_splits(int32_t B, int32_t n_q, int32_t H_kv, int64_t max_len) {
    if (n_q >= 2 && n_q <= kMaxExtendTokens) {
        int32_t n = wmtp_attn_num_splits(B, 1, H_kv, max_len);
        n = n > kMaxExtendSplits ? kMaxExtendSplits : n;
        if (max_len >= (int64_t)kExtendMinKeysPerSplit * n) return n;
    }
    return wmtp_attn_num_splits(B, n_q, H_kv, max_len);
}

}  // extern "C"
