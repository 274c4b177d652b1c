// wmtp_attn.cu -- split-KV flash-decode draft attention for sm_103a.
//
// Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
// Million-Token Context" (arXiv 2607.21535), §4 Mechanism: the draft's
// decode attention reads exactly the keys its (reduced) block table lists,
// with no further mask.  The split-KV partition and the log-sum-exp merge are
// textbook flash-decoding: exact in exact arithmetic, so the result does not
// depend on how the row is split.
//
// Kernel design (one CTA = one chunk of one table row for one KV head):
//   * four warps; each warp owns 16 keys of every 64-key tile and runs its
//     own three-stage copy pipeline for them.  The chunk's slot numbers are
//     fetched from the table into a per-warp shared-memory ring with cp.async
//     five tiles ahead; each key's K row and V row (D bf16) is then gathered
//     with 16-byte cp.async copies -- one 512-byte row per warp instruction,
//     fully coalesced -- into a padded shared-memory tile.  Keys past the
//     chunk end (or with a bad slot) are zero-filled by the copy itself
//     (source size 0) and masked.  Warps never wait for each other inside
//     the loop, and no issue ever waits on a global load.
//   * QK^T runs on the tensor cores with the keys as the M dimension and the
//     (up to 8) query heads of the GQA group as N, so one K/V read serves the
//     whole group and no MMA rows are padding.  The weights are split into
//     bf16 head + tail and transposed in registers (movmatrix) into the B
//     operand of the PV product, which accumulates O^T (D x 8) in fp32
//     registers.  Online softmax in base 2, max/sum across lanes with warp
//     shuffles; the accumulator is rescaled only when a running max moves.
//   * at the end the four warps combine through shared memory (per-head
//     factors computed once).  The splits of a (row, KV head) then merge in
//     one of four ways:
//       - up to 16 splits run as one thread-block cluster and merge through
//         distributed shared memory, each CTA producing a slice of the
//         output;
//       - up to 8 such clusters (128 splits) merge in two levels: each
//         cluster merges as above into a per-cluster partial of its slice,
//         takes a ticket for that slice, and the last cluster's CTA merges
//         the slice over the clusters in cluster order;
//       - without a cluster plan, when the whole grid is resident at once,
//         every split writes its partial, takes an arrival ticket and merges
//         its own slice of the output once all have arrived (slice merge);
//       - otherwise every split writes its partial to the workspace, takes a
//         ticket, and the last CTA merges all splits in split order.
//     Only the slice merge waits on other CTAs, and only for a bounded time
//     (the last CTA to arrive merges whatever the others left).
//   * every kernel is launched with programmatic stream serialization and
//     waits on its predecessor with griddepcontrol.wait before touching
//     global memory, so consecutive launches overlap only their start-up;
//     chained draft steps (the _overlap entry points) instead copy the keys
//     their predecessor cannot be writing before that wait, and release
//     their own dependents only after it.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <type_traits>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"

namespace wmtp {
namespace {

__device__ int32_t g_attn_error = 0;

__device__ __forceinline__ void latch(int32_t code) { atomicCAS(&g_attn_error, 0, code); }

constexpr int kConsumerWarps = 4;
constexpr int kKeysPerWarp = 16;
constexpr int kTileKeys = kConsumerWarps * kKeysPerWarp;  // 64 keys per tile
constexpr int kThreads = kConsumerWarps * 32;
constexpr int kMaxGroup = 8;  // query heads per KV head handled by one CTA
constexpr int kMaxSplits = 1024;
constexpr int kMaxClusterMerge = 16;  // splits merged through a cluster (non-portable size)
constexpr int kMaxClusters = 8;       // clusters merged by the second level
constexpr int kMaxNew = 4;            // rows one request appends in a fused call (one per warp)
constexpr uint64_t kSlicePollNs = 50000;  // a slice-merge wait gives up after 50 us (results stay exact)
constexpr float kLn2 = 0.69314718055994530942f;
// Warp-specialised instances (long rows): one producer warp issues every
// copy, the four consumer warps only compute; waits are time-bounded.
constexpr int kWsProducers = 4;  // one producer warp per consumer warp (one of each per scheduler)
constexpr int kWsThreads = kThreads + 32 * kWsProducers;
constexpr int kWsMinKeysPerSplit = 4 * kTileKeys;  // rows with at least four key tiles per split
constexpr uint64_t kWsWaitNs = 2000000000ull;

// The consumer warps' CTA barrier (named barrier 1, 128 threads): in a
// warp-specialised CTA the producer warp has left by then.
__device__ __forceinline__ void sync_consumers() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The same barrier, returning how many of the consumer threads passed p.
__device__ __forceinline__ int sync_consumers_count(bool p) {
    int n;
    asm volatile(
        "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.popc.u32 %0, 1, 128, q;\n\t}"
        : "=r"(n)
        : "r"((uint32_t)p)
        : "memory");
    return n;
}

#ifndef WMTP_FP8_STAGES
#define WMTP_FP8_STAGES 6
#endif

template <int D, bool kFp8 = false, bool kSwzTiles = false>
struct Cfg {
    static constexpr int kRowBytes = D * (kFp8 ? 1 : 2);  // one K (or V) row of one head
    // Ring instances (bf16): 16 rows per warp as D/64 blocks of 16 x 128
    // bytes in the 128-byte-swizzled layout a TMA box writes (16-byte chunk c
    // of row r at ((c ^ r % 8) << 4)), conflict-free for ldmatrix, so that a
    // warp's keys in consecutive ring slots arrive as TMA boxes.  Table
    // instances: rows padded by 16 bytes (every key a row copy: a random
    // page table has no runs, and the padded layout measured faster there).
    static constexpr bool kSwz = kSwzTiles && !kFp8;
    static constexpr int kPitch = kSwz ? kRowBytes : kRowBytes + 16;
    static constexpr int kBlockBytes = kKeysPerWarp * 128;  // one 64-dimension block of a warp tile
    // fp8 rows are half as long: more stages keep as many bytes in flight
    static constexpr int kStages = kFp8 ? WMTP_FP8_STAGES : 3;
    static constexpr int kWarpTile = kKeysPerWarp * kPitch;     // 16 rows of K (or V)
    static constexpr int kWarpStage = 2 * kWarpTile;            // K rows then V rows
    static constexpr int kWarpBytes = kStages * kWarpStage;     // one warp's pipeline
    static constexpr int kTilesBytes = kConsumerWarps * kWarpBytes;
    static constexpr int kOPitch = D + 4;                       // fp32 combine rows
    static constexpr int kCombineBytes =
        kConsumerWarps * kMaxGroup * kOPitch * 4 + 2 * kConsumerWarps * kMaxGroup * 4;
    static constexpr int kPartBytes = kMaxGroup * D * 4 + kMaxGroup * 4;  // cluster merge
    static constexpr int kMergeBytes = kMaxGroup * kMaxSplits * 4;        // ticket merge
    static_assert(kCombineBytes + kPartBytes + kMergeBytes <= kTilesBytes, "merge areas must fit");
    static constexpr int kRingTiles = 2 * kStages;   // slot tiles held per warp
    static constexpr int kRingOffset = kTilesBytes;  // int32 [warps][ring tiles][16]
    static constexpr int kMaskOffset = kRingOffset + kConsumerWarps * kRingTiles * kKeysPerWarp * 4;
    static constexpr int kFlagOffset = kMaskOffset + kConsumerWarps * kStages * 4;
    // warp-specialised instances: a full and an empty mbarrier per stage
    static constexpr int kBarOffset = (kFlagOffset + 16 + 7) / 8 * 8;
    // swizzled tiles: one TMA mbarrier per warp and stage
    static constexpr int kTmaBarOffset = kBarOffset + 2 * kStages * 8;
    // + slack to align the base of the swizzled tiles to 1024 bytes
    static constexpr int kSmemBytes = kTmaBarOffset + kConsumerWarps * kStages * 8 + (kSwz ? 1024 : 0);
};

// Workspace: a counter region of kMaxClusterMerge int32 per (row, KV head),
// then the partials.  Split-order merge: lse_part [B*n_q*H_q][n_split] (base
// 2) and o_part [B*n_q*H_q][n_split][D].  Two-level merge: o_part holds the
// per-cluster outputs [B*n_q*H_kv][clusters][G*D] and lse_part the matching
// per-element lse [B*n_q*H_kv][clusters][G*D/4].  Every path returns the
// counters it used to zero.
struct WorkspaceView {
    int32_t *counters;
    float *lse_part;
    float *o_part;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// int32 counters per (row, KV head): at least one cluster's worth, or the
// slice merge's arrival and departure counts plus one claim word per split.
inline int counter_stride(int n_split) {
    const int need = (2 + n_split + 15) / 16 * 16;
    return need > kMaxClusterMerge ? need : kMaxClusterMerge;
}
inline size_t counter_bytes(int64_t rows_kv, int n_split) {
    return align256((size_t)rows_kv * counter_stride(n_split) * 4);
}

// Bytes for the split-order merge; the two-level merge (at most n_split / 2
// clusters, each holding rows_q * D outputs and rows_q * D / 4 lse values)
// never needs more.
inline size_t workspace_bytes(int64_t rows_q, int64_t rows_kv, int D, int n_split) {
    if (n_split <= 1) return 0;
    const size_t split_order = counter_bytes(rows_kv, n_split) + align256((size_t)rows_q * n_split * 4) +
                               (size_t)rows_q * n_split * D * 4;
    const int64_t m = n_split / 2 < kMaxClusters ? n_split / 2 : kMaxClusters;
    const size_t two_level =
        counter_bytes(rows_kv, n_split) + align256((size_t)rows_q * m * D * 4) + (size_t)rows_q * m * D;
    return split_order > two_level ? split_order : two_level;
}

// The step's own K/V rows, appended to the pool by the same launch:
// k_new / v_new [B][n_new][H_kv][D] bf16, slots [B][n_new].  n_new == 0: no
// append.  Gathers of a key whose slot is one of its request's appended
// slots read the new row itself, so no CTA reads a pool slot that this
// launch writes.
// Chained steps (chain != 0: the overlapped bf16 table and ring steps)
// release their dependents only after their own wait.  With hold >= 0 the
// table, lengths, slots and the K/V rows of entries below L - hold are read
// before the preceding kernel has completed (copied while it finishes); q,
// the new rows and the last `hold` entries of each row only after it.
struct AppendView {
    const __nv_bfloat16 *k_new;
    const __nv_bfloat16 *v_new;
    const int32_t *slots;
    __nv_bfloat16 *k_pool;
    __nv_bfloat16 *v_pool;
    int32_t n_new;
    int32_t chain;
    int32_t hold;
};
// Draft-extend pass: the n_q rows of request b are its new tokens at
// positions S..S+n-1 (n = n_new[b]; rows t >= n are empty), all reading the
// union table of wmtp_build_extend_indices; token t sees only the keys of
// its own keep set (positions below S + t + 1, and, when windowed, sinks or
// positions from S + t + 1 - W).  seq_lens == nullptr: not an extend pass.
struct ExtendView {
    const int32_t *seq_lens;
    const int32_t *n_new;
    int32_t n_sink;
    int32_t window;
    int32_t windowed;
};
// fp8 KV: the pools hold E4M3 codes; key/value element = code * scale of
// its KV head (k_scale / v_scale [H_kv] fp32).  k_scale folds into the
// softmax scale, v_scale into the output.  k_scale == nullptr: bf16 pools.
struct Fp8View {
    const float *k_scale;
    const float *v_scale;
};
// The fp8 path feeds P to the tensor cores in fp16, scaled by 2^15 so that
// weights down to 2^-29 keep full fp16 precision (P <= 1 after the running
// max); the scale is divided out with the output normalisation.
constexpr float kPScaleF16 = 32768.f;
// Implicit-table ring attention: no table is read.  Draft step `step` of
// request b (committed length S = seq_lens[b]) sees kv_len = S + step + 1
// positions; the kept entries (sinks, then the W most recent when kv_len >
// n_sink + W) are mapped to ring slots in the kernel by the ring rule of
// ring_base[b].  With the fused append, the new row is position S + step.
// seq_lens == nullptr: not a ring launch.
struct RingView {
    const int32_t *seq_lens;
    const int32_t *ring_base;
    int32_t n_sink;
    int32_t window;
    int32_t depth;
    int32_t tree_k;
    int32_t step;
};

inline WorkspaceView carve(void *ws, int64_t rows_q, int64_t rows_kv, int n_split) {
    uint8_t *p = static_cast<uint8_t *>(ws);
    WorkspaceView v;
    v.counters = reinterpret_cast<int32_t *>(p);
    p += counter_bytes(rows_kv, n_split);
    v.lse_part = reinterpret_cast<float *>(p);
    p += align256((size_t)rows_q * n_split * 4);
    v.o_part = reinterpret_cast<float *>(p);
    return v;
}

inline WorkspaceView carve_two_level(void *ws, int64_t rows_q, int64_t rows_kv, int D, int n_split, int clusters) {
    uint8_t *p = static_cast<uint8_t *>(ws);
    WorkspaceView v;
    v.counters = reinterpret_cast<int32_t *>(p);
    p += counter_bytes(rows_kv, n_split);
    v.o_part = reinterpret_cast<float *>(p);
    p += align256((size_t)rows_q * clusters * D * 4);
    v.lse_part = reinterpret_cast<float *>(p);
    return v;
}

template <int D, bool kAppend, bool kExtend, bool kFp8, bool kRing = false, bool kWs = false,
          bool kChain = false>
__global__ void __launch_bounds__(kWs ? kWsThreads : kThreads, 1) split_decode_kernel(
    const __nv_bfloat16 *__restrict__ q, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t G,
    const void *__restrict__ k_pool, const void *__restrict__ v_pool,
    int64_t num_slots, const int32_t *__restrict__ table, int64_t table_stride,
    const int32_t *__restrict__ lens, float scale_log2, float *__restrict__ out,
    float *__restrict__ lse, WorkspaceView ws, int32_t n_split, int32_t csz, int32_t slice_stride,
    AppendView ap, ExtendView ev, Fp8View fv, RingView rv, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, int32_t tma_ok) {
    static_assert(!(kFp8 && (kAppend || kExtend)), "the fp8 path appends with its own kernel");
    static_assert(!(kRing && (kExtend || kFp8)), "ring launches are bf16 decode steps");
    static_assert(!kChain || (kAppend && !kExtend && !kFp8 && !kWs), "chained launches are fused bf16 steps");
    using C = Cfg<D, kFp8, kRing>;
    constexpr int S = C::kStages;
    constexpr int R = C::kRingTiles;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = C::kSwz ? reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))
                            : smem_raw;
    uint32_t *masks = reinterpret_cast<uint32_t *>(smem + C::kMaskOffset);
    uint64_t *tma_bars = reinterpret_cast<uint64_t *>(smem + C::kTmaBarOffset);  // [warp][stage]
    volatile int32_t *flags = reinterpret_cast<volatile int32_t *>(smem + C::kFlagOffset);
    uint64_t *ws_bars = reinterpret_cast<uint64_t *>(smem + C::kBarOffset);  // [S] full, then [S] empty

    if constexpr (!kChain) griddep_launch_dependents();
    if constexpr (C::kSwz) {
        // one arrival per use: the issuing lane's (with the TMA byte count
        // when the warp's keys arrive as boxes)
        if (threadIdx.x == 0) {
            for (int i = 0; i < kConsumerWarps * S; ++i) mbar_init(smem_addr(tma_bars + i), 1);
            fence_mbar_init();
        }
        __syncthreads();
    }
    if constexpr (kWs) {
        // full: per producer warp, 32 copy-completion arrivals of its lanes
        // and one after its key mask is stored; empty: one per consumer warp
        if (threadIdx.x == 0) {
            for (int i = 0; i < S; ++i) {
                mbar_init(smem_addr(ws_bars + i), kWsProducers * 33);
                mbar_init(smem_addr(ws_bars + S + i), kConsumerWarps);
            }
            flags[3] = 0;
            fence_mbar_init();
        }
        __syncthreads();  // all warps, before the roles split
    }

    // A chained launch releases its dependents only after its own wait, so
    // a dependent that reads early overlaps with this kernel alone.
    const bool early = kChain && ap.hold >= 0;
    if (!early) {
        griddep_wait();
        if constexpr (kChain) griddep_launch_dependents();
    }

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int g = blockIdx.y;
    const int64_t bt = blockIdx.z;  // request * n_q + query token
    const int64_t b = bt / n_q;
    const int r = lane >> 2;  // MMA group: key row (QK) / output dim row (PV)
    const int c = lane & 3;   // thread in group: query-head pair 2c, 2c+1
    constexpr int KD = D / 16;
    // Ring launch: the request's length and ring base, loaded before q so
    // that both loads are in flight together.
    int32_t r_S = 0, r_base32 = 0;
    if constexpr (kRing) {
        r_S = __ldg(rv.seq_lens + b);
        r_base32 = __ldg(rv.ring_base + b);
    }

    // Query fragments (B operand of QK^T), loaded first so that their latency
    // overlaps the table fetch.  fp8 path: fp16 fragments, with the head
    // dimension in the order the E4M3 key fragments come in (k index 2c+e of
    // step kd is dimension 16kd + 4c + e, k index 2c+8+e is 16kd + 4c+2+e).
    uint32_t qf[KD][2];
    auto load_q = [&]() {
        const bool live = r < G;
        const __nv_bfloat16 *qrow = q + (bt * H_q + (int64_t)g * G + (live ? r : 0)) * D;
#pragma unroll
        for (int kd = 0; kd < KD; ++kd) {
            if constexpr (kFp8) {
                const uint32_t *q2 = reinterpret_cast<const uint32_t *>(qrow + kd * 16 + 4 * c);
                const uint32_t w0 = live ? __ldg(q2) : 0u, w1 = live ? __ldg(q2 + 1) : 0u;
                qf[kd][0] = pack_f16x2(bf16_lo_to_f32(w0), bf16_hi_to_f32(w0));
                qf[kd][1] = pack_f16x2(bf16_lo_to_f32(w1), bf16_hi_to_f32(w1));
            } else {
                qf[kd][0] = live ? __ldg(reinterpret_cast<const uint32_t *>(qrow + kd * 16 + 2 * c)) : 0u;
                qf[kd][1] = live ? __ldg(reinterpret_cast<const uint32_t *>(qrow + kd * 16 + 2 * c + 8)) : 0u;
            }
        }
    };
    if (!early) load_q();
    float sl2 = scale_log2;  // softmax scale in base 2 (times k_scale for fp8 keys)
    float out_scale = 1.f;   // v_scale / P scale for fp8 values
    if constexpr (kFp8) {
        sl2 *= __ldg(fv.k_scale + g);
        out_scale = __ldg(fv.v_scale + g) * (1.f / kPScaleF16);
    }

    // Ring launch: this step's kv length, its keep rule and the ring.
    int64_t r_kv = 0, r_lo = 0, r_base = 0;
    bool r_win = false;
    if constexpr (kRing) {
        if (r_S < 0 && threadIdx.x == 0 && split == 0 && g == 0) latch(WMTP_DEV_LEN_RANGE);
        r_kv = r_S < 0 ? 0 : (int64_t)r_S + rv.step + 1;
        r_win = r_kv > (int64_t)rv.n_sink + rv.window;
        r_lo = r_kv - rv.window;
        r_base = r_base32;
    }
    const uint32_t r_mod = kRing ? (uint32_t)(rv.window + rv.depth * rv.tree_k) : 1u;
    // ring rule on branch 0 in 32-bit arithmetic (positions, ring sizes and
    // slots are below 2^31: checked on the host)
    auto ring_slot32 = [&](int64_t pos) -> int32_t {
        return pos < rv.n_sink ? (int32_t)(r_base + pos)
                               : (int32_t)r_base + rv.n_sink + (int32_t)((uint32_t)(pos - rv.n_sink) % r_mod);
    };
    // Slots this request appends in this launch (-1: none).  A ring launch
    // needs none before the loop: its new row is always the last kept entry
    // (position S + step), and the writer maps it after the loop.
    int32_t nslot[kMaxNew];
#pragma unroll
    for (int i = 0; i < kMaxNew; ++i)
        nslot[i] = (!kRing && kAppend && i < ap.n_new) ? __ldg(ap.slots + b * ap.n_new + i) : -1;

    // Chunk of this split: a multiple of the key tile, fixed by L and n_split.
    // The slot fetch starts for the chunk of a full row (L = table_stride)
    // while the length is still loading, and is redone only if the real
    // chunk differs.
    const int32_t L_in = kRing ? (int32_t)(r_kv <= 0 ? 0 : (r_win ? (int64_t)rv.n_sink + rv.window : r_kv))
                               : lens[b];
    auto chunk_of = [&](int64_t len) {
        const int64_t ch = (len + n_split - 1) / n_split;
        return (ch + kTileKeys - 1) / kTileKeys * kTileKeys;
    };
    const uint64_t policy = l2_policy_evict_first();
    const uint8_t *kbase = reinterpret_cast<const uint8_t *>(k_pool) + (size_t)g * C::kRowBytes;
    const uint8_t *vbase = reinterpret_cast<const uint8_t *>(v_pool) + (size_t)g * C::kRowBytes;
    const size_t slot_bytes = (size_t)H_kv * C::kRowBytes;
    const uint32_t wsm_addr = smem_addr(smem + warp * C::kWarpBytes);

    // Slot numbers travel through a per-warp shared-memory ring, fetched with
    // cp.async 2S-1 tiles ahead inside the same commit groups as the K/V
    // rows, so issuing a tile's gathers never waits on a global load.
    const int32_t *ring = reinterpret_cast<const int32_t *>(smem + C::kRingOffset) + warp * R * kKeysPerWarp;
    const uint32_t ring_addr = smem_addr(ring);
    auto fetch_slots_from = [&](int t, const int32_t *row, int64_t n) {
        if (!kRing && lane < kKeysPerWarp) {
            const int64_t k = (int64_t)t * kTileKeys + warp * kKeysPerWarp + lane;
            const bool in = k < n;
            cp_async_4(ring_addr + ((t % R) * kKeysPerWarp + lane) * 4,
                       in ? static_cast<const void *>(row + k) : static_cast<const void *>(table),
                       in ? 4u : 0u);
        }
    };
    const int64_t chunk_g = chunk_of(table_stride);
    const int64_t start_g = (int64_t)split * chunk_g;
    const int64_t cnt_g = table_stride - start_g < 0 ? 0 : (table_stride - start_g < chunk_g ? table_stride - start_g : chunk_g);
    const int n_tiles_g = (int)((cnt_g + kTileKeys - 1) / kTileKeys);
    if constexpr (!kWs) {
        for (int t = 0; t < 2 * S - 1 && t < n_tiles_g; ++t) fetch_slots_from(t, table + b * table_stride + start_g, cnt_g);
        cp_async_commit();
    }

    int64_t L = L_in;
    if (L < 0 || L > table_stride) {
        if (threadIdx.x == 0 && split == 0 && g == 0) latch(WMTP_DEV_LEN_RANGE);
        L = L < 0 ? 0 : table_stride;
    }
    // Extend pass: position of union entry e is e below n_sink (or when the
    // union is not windowed), else lo_u + e - n_sink; this row's token sees
    // positions below kv_t and, if windowed, only sinks or from lo_t.
    int64_t x_lo_u = 0, x_kv_t = 0, x_lo_t = 0;
    bool x_win_u = false, x_win_t = false;
    if constexpr (kExtend) {
        const int t = (int)(bt % n_q);
        int32_t nn = ev.n_new[b];
        nn = nn < 0 ? 0 : nn;
        const int64_t S = ev.seq_lens[b];
        if (t >= nn) L = 0;
        const int64_t kv_u = S + nn, w_u = (int64_t)ev.window + (nn > 0 ? nn - 1 : 0);
        x_win_u = ev.windowed && kv_u > (int64_t)ev.n_sink + w_u;
        x_lo_u = kv_u - w_u;
        x_kv_t = S + t + 1;
        x_win_t = ev.windowed && x_kv_t > (int64_t)ev.n_sink + ev.window;
        x_lo_t = x_kv_t - ev.window;
    }
    const int64_t chunk = chunk_of(L);
    const int64_t start = (int64_t)split * chunk;
    const int64_t cnt = L - start < 0 ? 0 : (L - start < chunk ? L - start : chunk);
    const int n_tiles = (int)((cnt + kTileKeys - 1) / kTileKeys);
    const int32_t *__restrict__ trow = table + b * table_stride + start;
    auto fetch_slots = [&](int t) { fetch_slots_from(t, trow, cnt); };
    if (!kWs && chunk != chunk_g) {  // a shorter row: fetch its own chunk
        cp_async_wait<0>();
        __syncwarp();
        for (int t = 0; t < 2 * S - 1 && t < n_tiles; ++t) fetch_slots(t);
        cp_async_commit();
    }

    // Issue the K/V gathers of tile t (stage t % S); its slots are in the ring.
    // Pass 0: every key.  A chained launch that reads early issues its
    // first tiles in two passes: 1 before its wait (every key not held) and
    // 2 after it (the held keys: the last `hold` entries of the row and keys
    // read from the new rows; `issued` is set if there were any).
    const uint8_t *knew = reinterpret_cast<const uint8_t *>(ap.k_new) +
                          ((size_t)b * ap.n_new * H_kv + g) * C::kRowBytes;
    const uint8_t *vnew = reinterpret_cast<const uint8_t *>(ap.v_new) +
                          ((size_t)b * ap.n_new * H_kv + g) * C::kRowBytes;
    auto issue_p = [&](int t, auto phase_c, bool &issued) {
        constexpr int P = decltype(phase_c)::value;
        const int st = t % S;
        const int64_t k = (int64_t)t * kTileKeys + warp * kKeysPerWarp + (lane & 15);
        int32_t my_slot = 0;
        if constexpr (kRing) {
            const int64_t e = start + k;
            const int64_t pos = (r_win && e >= rv.n_sink) ? r_lo + (e - rv.n_sink) : e;
            if (lane < kKeysPerWarp && k < cnt) my_slot = ring_slot32(pos);
        } else {
            my_slot = lane < kKeysPerWarp ? ring[(t % R) * kKeysPerWarp + lane] : 0;
        }
        const bool in = lane < kKeysPerWarp && k < cnt;
        bool ok = in && my_slot >= 0 && my_slot < num_slots;
        if (P != 2 && in && !ok) latch(WMTP_DEV_SLOT_RANGE);
        if constexpr (kExtend) {
            const int64_t e = start + k;
            const int64_t pos = (x_win_u && e >= ev.n_sink) ? x_lo_u + (e - ev.n_sink) : e;
            ok = ok && pos < x_kv_t && (!x_win_t || pos < ev.n_sink || pos >= x_lo_t);
        }
        // A key whose slot this launch appends is marked -2 - i (row i of
        // the new rows); its vm bit stays set.
        int32_t src_slot = my_slot;
        if constexpr (kAppend && kRing) {
            if (ok && start + k == L - 1) src_slot = -2;
        } else if constexpr (kAppend) {
#pragma unroll
            for (int i = kMaxNew - 1; i >= 0; --i)
                if (ok && my_slot == nslot[i]) src_slot = -2 - i;
        }
        uint32_t held = 0;  // keys of the second pass
        if constexpr (P != 0) {
            held = __ballot_sync(0xffffffffu, ok && (start + k >= L - ap.hold || src_slot < -1)) & 0xffffu;
            if (P == 2 && held == 0) return;
            issued = true;
        }
        const uint32_t vm = __ballot_sync(0xffffffffu, ok) & 0xffffu;
        if (P != 2 && lane == 0) masks[warp * S + st] = vm;
        const uint32_t kdst = wsm_addr + st * C::kWarpStage;
        const uint32_t vdst = kdst + C::kWarpTile;
        if constexpr (C::kSwz && P != 2) {
            // 16 valid keys in 16 consecutive pool slots (a ring window, an
            // identity page table), none of them appended by this launch:
            // the warp's K and V rows come in as D/64 TMA boxes each (64
            // dims x 1 head x 16 slots, 128-byte swizzle).  The stage's TMA
            // barrier completes one phase per use either way.
            const uint32_t tbar = smem_addr(tma_bars + warp * S + st);
            const int32_t s0 = __shfl_sync(0xffffffffu, src_slot, 0);
            const bool whole = tma_ok && vm == 0xffffu && held == 0 && s0 >= 0 &&
                               __all_sync(0xffffffffu, lane >= kKeysPerWarp || src_slot == s0 + lane);
            if (whole) {
                fence_proxy_async_smem();  // this warp's reads of the stage's previous rows come first
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_expect_tx(tbar, 2u * kKeysPerWarp * C::kRowBytes);
#pragma unroll
                    for (int db = 0; db < D / 64; ++db) {
                        tma_load_3d(kdst + db * C::kBlockBytes, &tm_k, db * 64, g, s0, tbar);
                        tma_load_3d(vdst + db * C::kBlockBytes, &tm_v, db * 64, g, s0, tbar);
                    }
                }
                return;
            }
            if (lane == 0) mbar_arrive(tbar);
        }
        constexpr int kLanesPerRow = C::kRowBytes / 16;  // 32 (D=256) or 16 (D=128)
        constexpr int kRowsPerInst = 32 / kLanesPerRow;
        const int sub = lane / kLanesPerRow;
        const int col = (lane % kLanesPerRow) * 16;
#pragma unroll
        for (int r0 = 0; r0 < kKeysPerWarp; r0 += kRowsPerInst) {
            const int key = r0 + sub;
            const int32_t slot = __shfl_sync(0xffffffffu, src_slot, key);
            const bool kv = (vm >> key) & 1u;
            const uint8_t *ksrc, *vsrc;
            if (kAppend && slot < -1) {
                ksrc = knew + (size_t)(-2 - slot) * slot_bytes + col;
                vsrc = vnew + (size_t)(-2 - slot) * slot_bytes + col;
            } else {
                const size_t off = kv ? (size_t)slot * slot_bytes + col : 0;
                ksrc = kbase + off;
                vsrc = vbase + off;
            }
            // swizzled: chunk c of row `key` in block c / 8 at ((c % 8) ^ (key % 8)) * 16
            const int chunk = col >> 4;
            const uint32_t dofs = C::kSwz ? (uint32_t)((chunk >> 3) * C::kBlockBytes + key * 128 + (((chunk & 7) ^ (key & 7)) << 4))
                                          : (uint32_t)(key * C::kPitch + col);
            if constexpr (P == 0) {
                cp_async_16(kdst + dofs, ksrc, kv ? 16u : 0u, policy);
                cp_async_16(vdst + dofs, vsrc, kv ? 16u : 0u, policy);
            } else {
                const bool hr = (held >> key) & 1u;
                if (P == 1 ? !hr : hr) {
                    cp_async_16(kdst + dofs, ksrc, kv ? 16u : 0u, policy);
                    cp_async_16(vdst + dofs, vsrc, kv ? 16u : 0u, policy);
                }
            }
        }
    };
    auto issue = [&](int t) {
        bool unused = false;
        issue_p(t, std::integral_constant<int, 0>{}, unused);
    };

    // Append: the first split of each (request, KV head) writes the new rows
    // of head g to the pool (read by later launches only).  Warp i loads row
    // i into registers here and stores it after the main loop, so the load
    // latency never sits on its path.
    constexpr int kNewPerLane = (C::kRowBytes + 32 * 16 - 1) / (32 * 16);  // 16-byte pieces
    const bool writer = kAppend && split == 0 && (bt % n_q) == 0 && warp < ap.n_new;
    int4 new_k[kNewPerLane], new_v[kNewPerLane];
    auto load_new = [&]() {
#pragma unroll
        for (int u = 0; u < kNewPerLane; ++u) {
            const int off = (u * 32 + lane) * 16;
            if (off < C::kRowBytes) {
                new_k[u] = *reinterpret_cast<const int4 *>(knew + (size_t)warp * slot_bytes + off);
                new_v[u] = *reinterpret_cast<const int4 *>(vnew + (size_t)warp * slot_bytes + off);
            }
        }
    };
    if (writer && !early) load_new();

    if constexpr (kWs) {
        if (warp >= kConsumerWarps) {
            // --------------------------------------------- producer warps
            // Producer warp p copies, for every tile, the 16 keys that
            // consumer warp p computes (lane l < 16: key 16p + l), with the
            // slot (table entry loaded three tiles ahead, or the ring rule),
            // validity and append substitution of the other instances'
            // gathers.  The stage's full barrier completes when every
            // producer's copies have landed and its key mask is stored.
            const int pw = warp - kConsumerWarps;
            auto slot_at = [&](int t) -> int32_t {
                const int64_t k = (int64_t)t * kTileKeys + pw * kKeysPerWarp + lane;
                return (!kRing && lane < kKeysPerWarp && k < cnt) ? __ldg(trow + k) : 0;
            };
            int32_t p0 = slot_at(0), p1 = slot_at(1), p2 = slot_at(2);
            constexpr int kLanesPerRow = C::kRowBytes / 16;
            constexpr int kRowsPerInst = 32 / kLanesPerRow;
            const int sub = lane / kLanesPerRow;
            const int col = (lane % kLanesPerRow) * 16;
            const uint32_t wsm = smem_addr(smem + pw * C::kWarpBytes);
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % S;
                const int32_t p3 = slot_at(t + 3);
                if (t >= S && !__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(ws_bars + S + st),
                                                                          ((t / S) - 1) & 1, kWsWaitNs))) {
                    if (lane == 0) {
                        latch(WMTP_DEV_WAIT_TIMEOUT);
                        flags[3] = 1;
                    }
                    break;
                }
                const int64_t k = (int64_t)t * kTileKeys + pw * kKeysPerWarp + (lane & 15);
                int32_t my_slot = p0;
                if constexpr (kRing) {
                    const int64_t e = start + k;
                    const int64_t pos = (r_win && e >= rv.n_sink) ? r_lo + (e - rv.n_sink) : e;
                    my_slot = (lane < kKeysPerWarp && k < cnt) ? ring_slot32(pos) : 0;
                }
                const bool in = lane < kKeysPerWarp && k < cnt;
                const bool ok = in && my_slot >= 0 && my_slot < num_slots;
                if (in && !ok) latch(WMTP_DEV_SLOT_RANGE);
                int32_t src_slot = my_slot;
                if constexpr (kAppend && kRing) {
                    if (ok && start + k == L - 1) src_slot = -2;
                } else if constexpr (kAppend) {
#pragma unroll
                    for (int i = kMaxNew - 1; i >= 0; --i)
                        if (ok && my_slot == nslot[i]) src_slot = -2 - i;
                }
                const uint32_t vm = __ballot_sync(0xffffffffu, ok) & 0xffffu;
                if (lane == 0) masks[pw * S + st] = vm;
                const uint32_t kdst0 = wsm + st * C::kWarpStage;
#pragma unroll
                for (int r0 = 0; r0 < kKeysPerWarp; r0 += kRowsPerInst) {
                    const int key = r0 + sub;
                    const int32_t slot = __shfl_sync(0xffffffffu, src_slot, key);
                    const bool kv = (vm >> key) & 1u;
                    const uint8_t *ksrc, *vsrc;
                    if (kAppend && slot < -1) {
                        ksrc = knew + (size_t)(-2 - slot) * slot_bytes + col;
                        vsrc = vnew + (size_t)(-2 - slot) * slot_bytes + col;
                    } else {
                        const size_t off = kv ? (size_t)slot * slot_bytes + col : 0;
                        ksrc = kbase + off;
                        vsrc = vbase + off;
                    }
                    cp_async_16(kdst0 + key * C::kPitch + col, ksrc, kv ? 16u : 0u, policy);
                    cp_async_16(kdst0 + C::kWarpTile + key * C::kPitch + col, vsrc, kv ? 16u : 0u, policy);
                }
                cp_async_mbar_arrive(smem_addr(ws_bars + st));
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(ws_bars + st));
                p0 = p1;
                p1 = p2;
                p2 = p3;
            }
            cp_async_wait<0>();
            return;
        }
    } else {
        // Prologue: slots of the first 2S-1 tiles (fetched above), then K/V
        // of the first S-1.
        cp_async_wait<0>();
        __syncwarp();
#pragma unroll
        for (int t = 0; t < S - 1; ++t) {
            if (t < n_tiles) {
                if constexpr (kChain) {
                    bool unused = false;
                    if (early)
                        issue_p(t, std::integral_constant<int, 1>{}, unused);
                    else
                        issue(t);
                } else {
                    issue(t);
                }
            }
            cp_async_commit();
        }
        if (early) {
            // the preceding kernel has completed: q, the new rows and the
            // held keys (in a group of their own, complete before tile 0)
            griddep_wait();
            griddep_launch_dependents();
            load_q();
            if (writer) load_new();
            bool any = false;
#pragma unroll
            for (int t = 0; t < S - 1; ++t)
                if (t < n_tiles) issue_p(t, std::integral_constant<int, 2>{}, any);
            cp_async_commit();
            if (any) cp_async_wait<0>();
        }
    }


    // -------------------------------------------------------------- compute
    float o[KD][4];
#pragma unroll
    for (int dt = 0; dt < KD; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max, rows 2c and 2c+1 (base 2)
    float l0 = 0.f, l1 = 0.f;              // this thread's share of the running sums

    const uint32_t k_off = (uint32_t)((lane & 15) * C::kPitch + (lane >> 4) * 16);
    const uint32_t v_off = (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * C::kPitch + ((lane >> 3) & 1) * 16);
    // swizzled tiles: this lane's ldmatrix row address for the 16-dimension
    // step kd lies in block kd / 4 at an in-block offset that repeats every
    // four steps
    uint32_t kso[4], vso[4];
    if constexpr (C::kSwz) {
        const int kr = lane & 15, ks = lane >> 4;
        const int vr = (lane & 7) + ((lane >> 4) << 3), vs = (lane >> 3) & 1;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            kso[i] = (uint32_t)(kr * 128 + (((2 * i + ks) ^ (kr & 7)) << 4));
            vso[i] = (uint32_t)(vr * 128 + (((2 * i + vs) ^ (vr & 7)) << 4));
        }
    }

    for (int it = 0; it < n_tiles; ++it) {
        if constexpr (kWs) {
            // the producer warp's copies of tile `it` have landed
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(ws_bars + it % S), (it / S) & 1, kWsWaitNs))) {
                if (lane == 0) {
                    latch(WMTP_DEV_WAIT_TIMEOUT);
                    flags[3] = 1;
                }
                break;
            }
        } else {
            // Groups committed so far: slots, K/V of tiles 0..S-2, then one
            // group per iteration; waiting for all but the newest S-1 makes
            // tile `it` (and the slots of tile it+S) resident.
            if (it + S - 1 < n_tiles) issue(it + S - 1);
            if (it + 2 * S - 1 < n_tiles) fetch_slots(it + 2 * S - 1);
            cp_async_commit();
            cp_async_wait<S - 1>();
            if constexpr (C::kSwz) {
                // the stage's TMA boxes (if its keys came that way) have landed
                if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(tma_bars + warp * S + it % S), (it / S) & 1,
                                                                kWsWaitNs))) {
                    if (lane == 0) latch(WMTP_DEV_WAIT_TIMEOUT);
                    break;
                }
            }
        }
        __syncwarp();
        const int st = it % S;
        const uint32_t wm = masks[warp * S + st];
        if (wm) {
            const uint32_t kaddr = wsm_addr + st * C::kWarpStage + k_off;
            const uint32_t vaddr = wsm_addr + st * C::kWarpStage + C::kWarpTile + (kFp8 ? k_off : v_off);
            const uint32_t kbase_s = wsm_addr + st * C::kWarpStage;   // swizzled tiles
            const uint32_t vbase_s = kbase_s + C::kWarpTile;
            // Four independent accumulation chains over the head dimension.
            float sacc[4][4] = {};
            if constexpr (kFp8) {
                // One ldmatrix brings 32 dimensions of 16 keys: register j
                // holds 4 codes (dimensions 4c..4c+3 of a 16-byte half) of
                // key r (j = 0, 2) or r + 8 (j = 1, 3), widened to two fp16
                // pairs for two k16 MMAs.
#pragma unroll
                for (int kc = 0; kc < D / 32; ++kc) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(kaddr + kc * 32, a0, a1, a2, a3);
                    mma_f16_16816(sacc[(2 * kc) & 3], e4m3x2_to_f16x2(a0), e4m3x2_to_f16x2(a1),
                                  e4m3x2_to_f16x2(a0 >> 16), e4m3x2_to_f16x2(a1 >> 16),
                                  qf[2 * kc][0], qf[2 * kc][1]);
                    mma_f16_16816(sacc[(2 * kc + 1) & 3], e4m3x2_to_f16x2(a2), e4m3x2_to_f16x2(a3),
                                  e4m3x2_to_f16x2(a2 >> 16), e4m3x2_to_f16x2(a3 >> 16),
                                  qf[2 * kc + 1][0], qf[2 * kc + 1][1]);
                }
            } else {
#pragma unroll
                for (int kd = 0; kd < KD; ++kd) {
                    uint32_t a0, a1, a2, a3;
                    if constexpr (C::kSwz)
                        ldsm_x4(kbase_s + (kd >> 2) * C::kBlockBytes + kso[kd & 3], a0, a1, a2, a3);
                    else
                        ldsm_x4(kaddr + kd * 32, a0, a1, a2, a3);
                    mma_bf16_16816(sacc[kd & 3], a0, a1, a2, a3, qf[kd][0], qf[kd][1]);
                }
            }
            float sc[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[i] = (sacc[0][i] + sacc[1][i]) + (sacc[2][i] + sacc[3][i]);
            // sc[0]: key r, head 2c; sc[1]: key r, head 2c+1; sc[2], sc[3]: key r+8.
            const bool ok_lo = (wm >> r) & 1u, ok_hi = (wm >> (r + 8)) & 1u;
            const float x0 = ok_lo ? sc[0] * sl2 : -INFINITY;
            const float x1 = ok_lo ? sc[1] * sl2 : -INFINITY;
            const float x2 = ok_hi ? sc[2] * sl2 : -INFINITY;
            const float x3 = ok_hi ? sc[3] * sl2 : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int sh = 4; sh < 32; sh <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);  // finite: wm != 0
            const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
            const float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1);
            const float p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);
            l0 = l0 * al0 + (p0 + p2);
            l1 = l1 * al1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {  // a running max moved
#pragma unroll
                for (int dt = 0; dt < KD; ++dt) {
                    o[dt][0] *= al0;
                    o[dt][1] *= al1;
                    o[dt][2] *= al0;
                    o[dt][3] *= al1;
                }
            }
            if constexpr (kFp8) {
                // P^T in fp16 (11 significant bits, scaled by 2^15) as the B
                // operand.  V^T comes from plain ldmatrix rows of codes: the
                // fp16 pairs of key r hold dimensions (4c, 4c+1) and
                // (4c+2, 4c+3), and movmatrix turns each 8x8 block into the
                // A fragment with M row r standing for dimension
                // 4(r/2) + r%2 (rows r) and that + 2 (rows r + 8) of its
                // 16-dimension group.
                const uint32_t ph0 = movmatrix_trans(pack_f16x2(p0 * kPScaleF16, p1 * kPScaleF16));
                const uint32_t ph1 = movmatrix_trans(pack_f16x2(p2 * kPScaleF16, p3 * kPScaleF16));
#pragma unroll
                for (int kc = 0; kc < D / 32; ++kc) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(vaddr + kc * 32, a0, a1, a2, a3);
                    mma_f16_16816(o[2 * kc], movmatrix_trans(e4m3x2_to_f16x2(a0)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a0 >> 16)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a1)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a1 >> 16)), ph0, ph1);
                    mma_f16_16816(o[2 * kc + 1], movmatrix_trans(e4m3x2_to_f16x2(a2)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a2 >> 16)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a3)),
                                  movmatrix_trans(e4m3x2_to_f16x2(a3 >> 16)), ph0, ph1);
                }
            } else {
                // P^T as the B operand: keys 2c,2c+1 (and +8) for query head
                // r.  P is split into a bf16 head and a bf16 tail (p = hi + lo
                // to about 16 significant bits) so that rounding the weights
                // to bf16 does not cost accuracy; both halves share the same V
                // fragment.
                const uint32_t h01 = pack_bf16x2(p0, p1), h23 = pack_bf16x2(p2, p3);
                const uint32_t t01 = pack_bf16x2(p0 - bf16_lo_to_f32(h01), p1 - bf16_hi_to_f32(h01));
                const uint32_t t23 = pack_bf16x2(p2 - bf16_lo_to_f32(h23), p3 - bf16_hi_to_f32(h23));
                const uint32_t ph0 = movmatrix_trans(h01), ph1 = movmatrix_trans(h23);
                const uint32_t pl0 = movmatrix_trans(t01), pl1 = movmatrix_trans(t23);
#pragma unroll
                for (int dt = 0; dt < KD; ++dt) {
                    uint32_t a0, a1, a2, a3;
                    if constexpr (C::kSwz)
                        ldsm_x4_trans(vbase_s + (dt >> 2) * C::kBlockBytes + vso[dt & 3], a0, a1, a2, a3);
                    else
                        ldsm_x4_trans(vaddr + dt * 32, a0, a1, a2, a3);
                    mma_bf16_16816(o[dt], a0, a1, a2, a3, ph0, ph1);
                    mma_bf16_16816(o[dt], a0, a1, a2, a3, pl0, pl1);
                }
            }
        }
        __syncwarp();
        if constexpr (kWs) {
            if (lane == 0) mbar_arrive(smem_addr(ws_bars + S + st));  // stage st is free again
        }
    }
    cp_async_wait<0>();

    if (writer) {
        int32_t sl = nslot[0];
#pragma unroll
        for (int i = 1; i < kMaxNew; ++i)
            if (warp == i) sl = nslot[i];
        if constexpr (kRing) sl = r_kv > 0 ? ring_slot32(r_kv - 1) : -1;
        if (sl < 0 || sl >= num_slots) {
            if (lane == 0) latch(WMTP_DEV_SLOT_RANGE);
        } else {
            uint8_t *kd = reinterpret_cast<uint8_t *>(ap.k_pool) + (size_t)sl * slot_bytes + (size_t)g * C::kRowBytes;
            uint8_t *vd = reinterpret_cast<uint8_t *>(ap.v_pool) + (size_t)sl * slot_bytes + (size_t)g * C::kRowBytes;
#pragma unroll
            for (int u = 0; u < kNewPerLane; ++u) {
                const int off = (u * 32 + lane) * 16;
                if (off < C::kRowBytes) {
                    *reinterpret_cast<int4 *>(kd + off) = new_k[u];
                    *reinterpret_cast<int4 *>(vd + off) = new_v[u];
                }
            }
        }
    }

    // Row sums: add the shares of the 8 lanes that hold the same query heads.
#pragma unroll
    for (int sh = 4; sh < 32; sh <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
        l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
    }

    // ---------------------------------------------- combine the four warps
    sync_consumers();  // every warp is done with its tiles
    float *ow = reinterpret_cast<float *>(smem);                       // [warp][head][kOPitch]
    float *mw = ow + kConsumerWarps * kMaxGroup * C::kOPitch;          // [warp][head]
    float *lw = mw + kConsumerWarps * kMaxGroup;                       // [warp][head]
    float *part_o = lw + kConsumerWarps * kMaxGroup;                   // [head][D] (cluster)
    float *part_lse = part_o + kMaxGroup * D;                          // [head]
    float *wts = part_lse + kMaxGroup;                                 // scratch for merges
    {
        float *o_lo = ow + (warp * kMaxGroup + 2 * c) * C::kOPitch;
        float *o_hi = o_lo + C::kOPitch;
        // accumulator rows r and r + 8 of group dt: dimensions 16dt + r and
        // 16dt + r + 8 (bf16), or 16dt + 4(r/2) + r%2 and that + 2 (fp8)
        const int d_a = kFp8 ? 4 * (r >> 1) + (r & 1) : r;
        const int d_b = kFp8 ? d_a + 2 : r + 8;
#pragma unroll
        for (int dt = 0; dt < KD; ++dt) {
            o_lo[dt * 16 + d_a] = o[dt][0];
            o_hi[dt * 16 + d_a] = o[dt][1];
            o_lo[dt * 16 + d_b] = o[dt][2];
            o_hi[dt * 16 + d_b] = o[dt][3];
        }
        if (r == 0) {
            mw[warp * kMaxGroup + 2 * c] = m0;
            mw[warp * kMaxGroup + 2 * c + 1] = m1;
            lw[warp * kMaxGroup + 2 * c] = l0;
            lw[warp * kMaxGroup + 2 * c + 1] = l1;
        }
    }
    sync_consumers();

    const int tid = threadIdx.x;
    const int64_t row_q0 = bt * H_q + (int64_t)g * G;  // first query row of the group
    // Per query head: the CTA max, each warp's factor 2^(m_w - M) / L and the
    // CTA's lse, computed once; then every output element is four FMAs.
    float *fac = wts;                                    // [head][warp]
    float *cta_lse = fac + kMaxGroup * kConsumerWarps;   // [head]
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mw[w * kMaxGroup + h]);
        float f[kConsumerWarps], Ls = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            f[w] = M == -INFINITY ? 0.f : exp2f(mw[w * kMaxGroup + h] - M);
            Ls += lw[w * kMaxGroup + h] * f[w];
        }
        const float inv = Ls > 0.f ? out_scale / Ls : 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) fac[h * kConsumerWarps + w] = f[w] * inv;
        cta_lse[h] = Ls > 0.f ? M + log2f(Ls) : -INFINITY;
    }
    sync_consumers();
    constexpr int D4 = D / 4;
    for (int e = tid; e < G * D4; e += kThreads) {
        const int h = e / D4, d4 = e - h * D4;
        float4 o_val = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float4 v = *reinterpret_cast<const float4 *>(ow + (w * kMaxGroup + h) * C::kOPitch + 4 * d4);
            const float f = fac[h * kConsumerWarps + w];
            o_val.x += v.x * f;
            o_val.y += v.y * f;
            o_val.z += v.z * f;
            o_val.w += v.w * f;
        }
        const float lse2 = cta_lse[h];
        if (csz) {
            reinterpret_cast<float4 *>(part_o + h * D)[d4] = o_val;
            if (d4 == 0) part_lse[h] = lse2;
        } else if (n_split == 1) {
            reinterpret_cast<float4 *>(out + (row_q0 + h) * D)[d4] = o_val;
            if (lse && d4 == 0) lse[row_q0 + h] = lse2 * kLn2;
        } else {
            reinterpret_cast<float4 *>(ws.o_part + ((row_q0 + h) * n_split + split) * D)[d4] = o_val;
            if (d4 == 0) ws.lse_part[(row_q0 + h) * n_split + split] = lse2;
        }
    }
    if (n_split == 1) return;

    if (csz) {
        // ---------------------------------- merge through distributed smem
        // Each cluster of csz CTAs covers csz consecutive splits of this
        // (row, KV head); CTA `rank` merges a slice of the G x D outputs,
        // reading every peer's partial in split order.  Each CTA arrives on
        // the closing barrier once its remote reads are done and waits on it
        // just before exit, which keeps its shared memory alive until every
        // peer has read it.
        __syncwarp();
        cluster_sync();
        const int rank = (int)cluster_ctarank();
        const int n_cl = n_split / csz;  // clusters of this (row, KV head)
        const int cl = split / csz;
        const int64_t rk = bt * H_kv + g;
        const int total4 = G * D4;
        const int per4 = (total4 + csz - 1) / csz;
        const int lo4 = rank * per4;
        const int hi4 = lo4 + per4 < total4 ? lo4 + per4 : total4;
        const uint32_t po_addr = smem_addr(part_o), pl_addr = smem_addr(part_lse);
        for (int f = lo4 + tid; f < hi4; f += kThreads) {  // one float4 of outputs
            const int h = f / D4;
            float ls[kMaxClusterMerge];
            float4 ov[kMaxClusterMerge];
            // every remote load is issued before any is used
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterMerge; ++s2) {
                if (s2 < csz) {
                    ls[s2] = ld_dsmem_f32(map_to_rank(pl_addr + h * 4, s2));
                    ov[s2] = ld_dsmem_f32x4(map_to_rank(po_addr + f * 16, s2));
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterMerge; ++s2)
                if (s2 < csz) M = fmaxf(M, ls[s2]);
            float sum = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (M != -INFINITY) {
#pragma unroll
                for (int s2 = 0; s2 < kMaxClusterMerge; ++s2) {
                    if (s2 < csz && ls[s2] != -INFINITY) {
                        const float w = exp2f(ls[s2] - M);
                        sum += w;
                        acc.x += w * ov[s2].x;
                        acc.y += w * ov[s2].y;
                        acc.z += w * ov[s2].z;
                        acc.w += w * ov[s2].w;
                    }
                }
            }
            const float inv = sum > 0.f ? 1.f / sum : 0.f;
            const float4 o_cl = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
            const float lse_cl = sum > 0.f ? M + log2f(sum) : -INFINITY;
            if (n_cl == 1) {
                reinterpret_cast<float4 *>(out + (row_q0 + h) * D)[f - h * D4] = o_cl;
                if (lse && f == h * D4) lse[row_q0 + h] = lse_cl * kLn2;
            } else {
                const int64_t idx = (rk * n_cl + cl) * total4 + f;
                reinterpret_cast<float4 *>(ws.o_part)[idx] = o_cl;
                ws.lse_part[idx] = lse_cl;
            }
        }
        cluster_arrive();  // this CTA's reads of its peers are done
        if (n_cl > 1) {
            // -------------------- second level: the last cluster merges the
            // slice over all clusters, in cluster order
            __threadfence();
            sync_consumers();
            int32_t *ctr = ws.counters + rk * kMaxClusterMerge + rank;
            if (tid == 0) flags[0] = (atomicAdd(ctr, 1) == n_cl - 1);
            sync_consumers();
            if (flags[0]) {
                __threadfence();
                const float4 *o2 = reinterpret_cast<const float4 *>(ws.o_part) + rk * n_cl * total4;
                const float *l2 = ws.lse_part + rk * n_cl * total4;
                for (int f = lo4 + tid; f < hi4; f += kThreads) {
                    const int h = f / D4;
                    float ls[kMaxClusters];
                    float4 ov[kMaxClusters];
#pragma unroll
                    for (int c2 = 0; c2 < kMaxClusters; ++c2) {
                        if (c2 < n_cl) {
                            ls[c2] = __ldcg(l2 + (int64_t)c2 * total4 + f);
                            ov[c2] = __ldcg(o2 + (int64_t)c2 * total4 + f);
                        }
                    }
                    float M = -INFINITY;
#pragma unroll
                    for (int c2 = 0; c2 < kMaxClusters; ++c2)
                        if (c2 < n_cl) M = fmaxf(M, ls[c2]);
                    float sum = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != -INFINITY) {
#pragma unroll
                        for (int c2 = 0; c2 < kMaxClusters; ++c2) {
                            if (c2 < n_cl && ls[c2] != -INFINITY) {
                                const float w = exp2f(ls[c2] - M);
                                sum += w;
                                acc.x += w * ov[c2].x;
                                acc.y += w * ov[c2].y;
                                acc.z += w * ov[c2].z;
                                acc.w += w * ov[c2].w;
                            }
                        }
                    }
                    const float inv = sum > 0.f ? 1.f / sum : 0.f;
                    reinterpret_cast<float4 *>(out + (row_q0 + h) * D)[f - h * D4] =
                        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
                    if (lse && f == h * D4)
                        lse[row_q0 + h] = sum > 0.f ? (M + log2f(sum)) * kLn2 : -INFINITY;
                }
                if (tid == 0) *ctr = 0;  // ready for the next call
            }
        }
        cluster_wait();  // peers may still read this CTA's shared memory
        return;
    }

    if (slice_stride) {
        // ------------------------------------------------- slice merge
        // Every split has written its partial.  Each CTA takes an arrival
        // ticket; all but the last wait (time-bounded) until every split has
        // arrived and then merge their own slice of the G x D outputs, so the
        // merge runs on all the launch's SMs at once.  The last to arrive
        // never waits: it merges its own slice and then every slice still
        // unclaimed (one whose CTA gave up waiting), so each slice is merged
        // exactly once (claims are compare-and-swap) whatever the
        // co-residency.  The last CTA to leave returns the counters to zero.
        __threadfence();
        sync_consumers();
        int32_t *ctr = ws.counters + (bt * H_kv + g) * slice_stride;  // arrivals, departures, claims
        if (tid == 0) {
            const bool last = atomicAdd(ctr, 1) == n_split - 1;
            const bool all_in = last || poll_geq_bounded(ctr, n_split, kSlicePollNs);
            if (all_in) __threadfence();
            flags[1] = last;
            flags[2] = all_in && atomicCAS(ctr + 2 + split, 0, 1) == 0;
        }
        sync_consumers();
        const bool last = flags[1] != 0;
        const bool mine = flags[2] != 0;
        const int total4 = G * D4;
        const int per4 = (total4 + n_split - 1) / n_split;
        float *sw = wts;                                    // [heads of the slice][n_split]
        float4 *red = reinterpret_cast<float4 *>(part_o);   // [kThreads]
        int32_t *claim = reinterpret_cast<int32_t *>(ow);   // [n_split]
        // Merges slice s_idx: float4 outputs [lo4, hi4) of this (row, KV
        // head); kThreads / nel threads per output, each summing a strided
        // subset of the splits, then a fixed-order reduction.
        auto slice_merge = [&](int s_idx) {
            const int lo4 = s_idx * per4;
            const int hi4 = lo4 + per4 < total4 ? lo4 + per4 : total4;
            if (lo4 >= hi4) return;
            const int nel = hi4 - lo4;
            const int h0 = lo4 / D4;
            const int nh = (hi4 - 1) / D4 - h0 + 1;
            const int R = kThreads / nel;  // >= 1: the host takes this path only when nel <= kThreads
            const int r = tid / nel, el = tid - (tid / nel) * nel;
            const int f = lo4 + el;
            const int h = f / D4, d4 = f - h * D4;
            const float4 *op = reinterpret_cast<const float4 *>(ws.o_part + (row_q0 + h) * n_split * D) + d4;
            // the first batch of output partials is in flight while the lse
            // values load and the weights are formed
            constexpr int kBatch = 8;
            float4 v[kBatch];
            if (r < R) {
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int s2 = r + u * R;
                    if (s2 < n_split) v[u] = __ldcg(op + (int64_t)s2 * D4);
                }
            }
            for (int e = tid; e < nh * n_split; e += kThreads) {
                const int hh = e / n_split, s2 = e - hh * n_split;
                sw[e] = __ldcg(ws.lse_part + (row_q0 + h0 + hh) * n_split + s2);
            }
            sync_consumers();
            for (int hh = warp; hh < nh; hh += kConsumerWarps) {
                float *x = sw + hh * n_split;
                float M = -INFINITY;
                for (int s2 = lane; s2 < n_split; s2 += 32) M = fmaxf(M, x[s2]);
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
                float sum = 0.f;
                if (M != -INFINITY)
                    for (int s2 = lane; s2 < n_split; s2 += 32) sum += x[s2] == -INFINITY ? 0.f : exp2f(x[s2] - M);
#pragma unroll
                for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
                const float lse_tot = sum > 0.f ? M + log2f(sum) : -INFINITY;
                __syncwarp();
                for (int s2 = lane; s2 < n_split; s2 += 32)
                    x[s2] = (sum > 0.f && x[s2] != -INFINITY) ? exp2f(x[s2] - lse_tot) : 0.f;
                if (lane == 0 && lse && (h0 + hh) * D4 >= lo4) lse[row_q0 + h0 + hh] = lse_tot * kLn2;
            }
            sync_consumers();
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < R) {
                const float *wh = sw + (h - h0) * n_split;
                for (int s0 = r; s0 < n_split; s0 += kBatch * R) {
                    if (s0 != r) {
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int s2 = s0 + u * R;
                            if (s2 < n_split) v[u] = __ldcg(op + (int64_t)s2 * D4);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kBatch; ++u) {
                        const int s2 = s0 + u * R;
                        if (s2 < n_split) {
                            const float w = wh[s2];
                            acc.x += w * v[u].x;
                            acc.y += w * v[u].y;
                            acc.z += w * v[u].z;
                            acc.w += w * v[u].w;
                        }
                    }
                }
            }
            red[tid] = acc;
            sync_consumers();
            if (tid < nel) {
                float4 t = red[tid];
                for (int rr = 1; rr < R; ++rr) {
                    const float4 u = red[rr * nel + tid];
                    t.x += u.x;
                    t.y += u.y;
                    t.z += u.z;
                    t.w += u.w;
                }
                reinterpret_cast<float4 *>(out + (row_q0 + h) * D)[d4] = t;
            }
            sync_consumers();  // sw and red are reused by the next slice
        };
        if (mine) slice_merge(split);
        if (last) {
            // a plain load first: a claimed word (every one, unless a CTA
            // gave up waiting) needs no compare-and-swap
            bool any = false;
            for (int s2 = tid; s2 < n_split; s2 += kThreads) {
                const bool c = s2 != split && ld_acquire_gpu(ctr + 2 + s2) == 0 &&
                               atomicCAS(ctr + 2 + s2, 0, 2) == 0;
                claim[s2] = c ? 1 : 0;
                any |= c;
            }
            // normally nothing is left: then skip the scan over the slices
            // (n_split iterations around an inlined merge took ~5 us on the
            // launch's critical path even when none was claimed)
            if (sync_consumers_count(any) > 0)
                for (int s2 = 0; s2 < n_split; ++s2)
                    if (claim[s2]) slice_merge(s2);
        }
        sync_consumers();
        if (tid == 0 && atomicAdd(ctr + 1, 1) == n_split - 1)
            for (int i = 0; i < 2 + n_split; ++i) ctr[i] = 0;  // ready for the next call
        return;
    }

    // ------------------------------------------ ticket; the last CTA merges
    __threadfence();
    sync_consumers();
    if (tid == 0) {
        const int32_t ticket = atomicAdd(&ws.counters[bt * H_kv + g], 1);
        flags[0] = (ticket == n_split - 1);
    }
    sync_consumers();
    if (!flags[0]) return;
    __threadfence();

    // Per query head: lse = log2 sum_s 2^lse_s; weights 2^(lse_s - lse).
    for (int e = tid; e < G * n_split; e += kThreads) {
        const int h = e / n_split, s2 = e - h * n_split;
        wts[h * n_split + s2] = __ldcg(ws.lse_part + (row_q0 + h) * n_split + s2);
    }
    sync_consumers();
    for (int h = warp; h < G; h += kConsumerWarps) {
        float M = -INFINITY;
        for (int s2 = lane; s2 < n_split; s2 += 32) M = fmaxf(M, wts[h * n_split + s2]);
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, sh));
        float sum = 0.f;
        if (M != -INFINITY) {
            // fixed order: lane-strided partial sums, then a fixed shuffle tree
            for (int s2 = lane; s2 < n_split; s2 += 32) {
                const float x = wts[h * n_split + s2];
                sum += x == -INFINITY ? 0.f : exp2f(x - M);
            }
        }
#pragma unroll
        for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
        const float lse_tot = (sum > 0.f) ? M + log2f(sum) : -INFINITY;
        __syncwarp();
        for (int s2 = lane; s2 < n_split; s2 += 32) {
            const float x = wts[h * n_split + s2];
            wts[h * n_split + s2] = (sum > 0.f && x != -INFINITY) ? exp2f(x - lse_tot) : 0.f;
        }
        if (lane == 0 && lse) lse[row_q0 + h] = lse_tot * kLn2;
    }
    sync_consumers();
    constexpr int kUnroll = 8;
    for (int e = tid; e < G * D4; e += kThreads) {
        const int h = e / D4, d4 = e - h * D4;
        const float4 *op = reinterpret_cast<const float4 *>(ws.o_part + (row_q0 + h) * n_split * D) + d4;
        const float *wh = wts + h * n_split;
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
        reinterpret_cast<float4 *>(out + (row_q0 + h) * D)[d4] = acc;
    }
    if (tid == 0) ws.counters[bt * H_kv + g] = 0;  // ready for the next call
}

// How many clusters of `n` CTAs of this kernel can be resident at once on
// device `dev` (0: none; cached per device and size).
// Sets the kernel attributes (large dynamic shared memory, non-portable
// cluster sizes) once per device for one kernel instance.
template <int D, bool A, bool X, bool F = false, bool RG = false, bool WS = false, bool CH = false>
bool prepare_kernel(int dev) {
    static int8_t done[64] = {};
    if (dev < 0 || dev >= 64) return false;
    if (done[dev]) return done[dev] > 0;
    const bool ok = cudaFuncSetAttribute(split_decode_kernel<D, A, X, F, RG, WS, CH>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<D, F, RG>::kSmemBytes) == cudaSuccess &&
                    cudaFuncSetAttribute(split_decode_kernel<D, A, X, F, RG, WS, CH>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
                    cudaFuncSetAttribute(split_decode_kernel<D, A, X, F, RG, WS, CH>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout, 100) == cudaSuccess;
    cudaGetLastError();
    done[dev] = ok ? 1 : -1;
    return ok;
}

// Sets the instance's attributes (once per device) and launches it.
template <int D, bool A, bool X, bool F, bool RG, bool WS, bool CH = false, typename... Args>
cudaError_t launch_instance(int dev, const cudaLaunchConfig_t *cfg, Args... args) {
    if (!prepare_kernel<D, A, X, F, RG, WS, CH>(dev)) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(cfg, split_decode_kernel<D, A, X, F, RG, WS, CH>, args...);
}

template <int D, bool F = false>
int cluster_capacity(int dev, int n) {
    static int16_t known[64][kMaxClusterMerge + 1] = {};
    if (n < 2 || n > kMaxClusterMerge || dev < 0 || dev >= 64) return 0;
    if (known[dev][n]) return known[dev][n] > 0 ? known[dev][n] : 0;
    bool ok = prepare_kernel<D, false, false, F>(dev);
    int clusters = 0;
    if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)n, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg<D, F>::kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = (unsigned)n;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        ok = cudaOccupancyMaxActiveClusters(&clusters, split_decode_kernel<D, false, false, F>, &cfg) == cudaSuccess &&
             clusters > 0;
        if (!ok) clusters = 0;
    }
    cudaGetLastError();  // a refused query is not an error of this call
    known[dev][n] = ok ? (int16_t)(clusters < 32767 ? clusters : 32767) : -1;
    return ok ? known[dev][n] : 0;
}

// CTAs of the plain instance the device holds at once (SMs x resident
// blocks per SM; 0 if unknown), cached per device.
template <int D, bool F = false>
int resident_capacity(int dev) {
    static int32_t known[64] = {};
    if (dev < 0 || dev >= 64) return 0;
    if (known[dev]) return known[dev] > 0 ? known[dev] : 0;
    int sms = 0, per_sm = 0;
    const bool ok = prepare_kernel<D, false, false, F>(dev) &&
                    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, split_decode_kernel<D, false, false, F>,
                                                                  kThreads, Cfg<D, F>::kSmemBytes) == cudaSuccess &&
                    sms > 0 && per_sm > 0;
    cudaGetLastError();
    known[dev] = ok ? sms * per_sm : -1;
    return ok ? known[dev] : 0;
}

template <int D, bool F>
wmtp_status launch_split_decode(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                int32_t H_kv, const void *k_pool, const void *v_pool,
                                int64_t num_slots, const int32_t *table, int64_t table_stride,
                                const int32_t *lens, float scale, float *out, float *lse,
                                void *workspace, int32_t n_split, cudaStream_t stream,
                                AppendView ap, ExtendView ev, Fp8View fv, RingView rv) {
    using C = Cfg<D, F>;
    const int64_t rows_q = (int64_t)B * n_q * H_q;
    const int64_t rows_kv = (int64_t)B * n_q * H_kv;
    // Kernel attributes are set once per device (outside any later stream
    // capture of the launches).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WMTP_ECUDA;
    const bool append = ap.n_new > 0;
    const bool chain = append && ap.chain != 0 && !F;
    const bool extend = ev.seq_lens != nullptr;
    const bool ring = rv.seq_lens != nullptr;
    // fp8 rows of at least four key tiles per split: the warp-specialised
    // instance (producer warps issue the copies, so the E4M3 widening and
    // the MMAs never hold up the next copies); same results bit for bit.
    // The bf16 instances keep their per-warp pipelines (measured faster:
    // their math per byte is half the fp8 path's).
    const bool use_ws = F && table_stride >= (int64_t)kWsMinKeysPerSplit * n_split;
    if (!prepare_kernel<D, false, false, F>(dev)) return WMTP_ECUDA;  // cluster and residency queries
    // Cluster size: all splits in one cluster, else the largest cluster that
    // divides n_split into at most kMaxClusters clusters, provided the device
    // holds every cluster of the launch at once (clusters that wait for a
    // second wave cost more than any merge saves); else no cluster: the
    // workspace merge, which needs no co-residency.
    int csz = 0;
    if (n_split > 1) {
        auto fits = [&](int c) {
            const int cap = cluster_capacity<D, F>(dev, c);
            return cap > 0 && rows_kv * (n_split / c) <= cap;
        };
        if (n_split <= kMaxClusterMerge && fits(n_split)) {
            csz = n_split;
        } else {
            for (int c = kMaxClusterMerge; c >= 2; --c) {
                if (n_split % c == 0 && n_split / c <= kMaxClusters && fits(c)) {
                    csz = c;
                    break;
                }
            }
        }
    }
    // No cluster plan: the slice merge when the whole grid fits on the
    // device at once (its waits then end as soon as the last split
    // arrives) and no slice holds more outputs than the CTA has threads,
    // else the last CTA merges.
    int slice = 0;
    if (csz == 0 && n_split > 1) {
        const int64_t total4 = (int64_t)(H_q / H_kv) * (D / 4);
        const int cap = resident_capacity<D, F>(dev);
        if ((total4 + n_split - 1) / n_split <= kThreads && cap > 0 && rows_kv * n_split <= cap)
            slice = counter_stride(n_split);
    }
    WorkspaceView ws{nullptr, nullptr, nullptr};
    if (n_split > 1 && csz == 0) ws = carve(workspace, rows_q, rows_kv, n_split);
    if (csz && n_split / csz > 1) ws = carve_two_level(workspace, rows_q, rows_kv, D, n_split, n_split / csz);
    const float scale_log2 = scale * 1.4426950408889634f;
    PdlLaunch launch(dim3((unsigned)n_split, (unsigned)H_kv, (unsigned)(B * n_q)), dim3(use_ws ? kWsThreads : kThreads),
                     ring ? Cfg<D, F, true>::kSmemBytes : C::kSmemBytes, stream);
    if (csz) launch.add_cluster((unsigned)csz);
    // ring launches (bf16): TMA maps for warps whose 16 keys sit in
    // consecutive ring slots
    CUtensorMap tmk{}, tmv{};
    int32_t tma_ok = 0;
    if (!F && ring) {
        if (num_slots <= INT32_MAX && pool_tensor_map(&tmk, k_pool, num_slots, H_kv, D, kKeysPerWarp) &&
            pool_tensor_map(&tmv, v_pool, num_slots, H_kv, D, kKeysPerWarp))
            tma_ok = 1;
    }
#define WMTP_ATTN_ARGS                                                                                          \
    dev, &launch.cfg, reinterpret_cast<const __nv_bfloat16 *>(q), n_q, H_q, H_kv, H_q / H_kv, k_pool, v_pool, \
        num_slots, table, table_stride, lens, scale_log2, out, lse, ws, n_split, (int32_t)csz, (int32_t)slice, ap, ev, fv, rv, \
        tmk, tmv, tma_ok
    cudaError_t err;
    if constexpr (F) {
        err = use_ws ? launch_instance<D, false, false, true, false, true>(WMTP_ATTN_ARGS)
                 : launch_instance<D, false, false, true, false, false>(WMTP_ATTN_ARGS);
    } else if (ring) {
        err = chain    ? launch_instance<D, true, false, false, true, false, true>(WMTP_ATTN_ARGS)
              : append ? launch_instance<D, true, false, false, true, false>(WMTP_ATTN_ARGS)
                       : launch_instance<D, false, false, false, true, false>(WMTP_ATTN_ARGS);
    } else if (extend) {
        err = launch_instance<D, false, true, false, false, false>(WMTP_ATTN_ARGS);
    } else {
        // with or without appended rows: the append instance (with n_new = 0
        // it substitutes nothing and writes nothing).  Its arithmetic is the
        // plain instance's, and it runs measurably faster (360 against 480
        // us for a 1M-key row), so the plain table-path instance is not used.
        err = chain ? launch_instance<D, true, false, false, false, false, true>(WMTP_ATTN_ARGS)
                    : launch_instance<D, true, false, false, false, false>(WMTP_ATTN_ARGS);
    }
#undef WMTP_ATTN_ARGS
    return err == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

// ------------------------------------------------ scratch without allocation
// Device scratch for wmtp_draft_decode_attn_noalloc: a fixed region of merge
// counters, then the split partials (lse, then o).  Every device that loads
// the library holds it until the process exits.
constexpr size_t kNoAllocBytes = WMTP_NOALLOC_SCRATCH_BYTES;
constexpr size_t kNoAllocCounterBytes = (size_t)WMTP_NOALLOC_MAX_COUNTERS * 4;
static_assert(kNoAllocCounterBytes % 256 == 0, "partials must stay 256-byte aligned");
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocBytes];

// Device address of the scratch array on the current device `dev`, looked up
// once per device (host code cannot use the symbol itself as an address).
// The cache is atomic: host threads whose first calls on a device overlap
// each look the address up and store the same value.  A cudaDeviceReset of
// the device makes the cached address stale (the array is re-created in the
// next context); the header says so.
void *noalloc_scratch(int dev) {
    static std::atomic<void *> addr[64] = {};
    if (dev < 0 || dev >= 64) return nullptr;
    void *cached = addr[dev].load(std::memory_order_acquire);
    if (!cached) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev].store(p, std::memory_order_release);
        cached = p;
    }
    return cached;
}

// Bytes of partials (after the counter region) a call needs.
inline size_t noalloc_partial_bytes(int64_t rows_q, int D, int n_split) {
    return align256((size_t)rows_q * n_split * 4) + (size_t)rows_q * n_split * D * 4;
}

template <int D>
wmtp_status launch_split_decode_noalloc(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                        int32_t H_kv, const uint16_t *k_pool,
                                        const uint16_t *v_pool, int64_t num_slots,
                                        const int32_t *table, int64_t table_stride,
                                        const int32_t *lens, float scale, float *out, float *lse,
                                        int32_t n_split, cudaStream_t stream) {
    using C = Cfg<D>;
    const int64_t rows_q = (int64_t)B * n_q * H_q;
    const int64_t rows_kv = (int64_t)B * n_q * H_kv;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WMTP_ECUDA;
    WorkspaceView ws{nullptr, nullptr, nullptr};
    if (n_split > 1) {
        uint8_t *base = static_cast<uint8_t *>(noalloc_scratch(dev));
        if (!base) return WMTP_ECUDA;
        ws.counters = reinterpret_cast<int32_t *>(base);
        ws.lse_part = reinterpret_cast<float *>(base + kNoAllocCounterBytes);
        ws.o_part = reinterpret_cast<float *>(base + kNoAllocCounterBytes +
                                              align256((size_t)rows_q * n_split * 4));
        // The array keeps the previous call's contents: the counters this
        // call uses must start at zero.
        if (cudaMemsetAsync(ws.counters, 0, (size_t)rows_kv * 4, stream) != cudaSuccess)
            return WMTP_ECUDA;
    }
    // the append instance with no appended rows (the table path's instance)
    if (!prepare_kernel<D, true, false>(dev)) return WMTP_ECUDA;
    const float scale_log2 = scale * 1.4426950408889634f;
    PdlLaunch launch(dim3((unsigned)n_split, (unsigned)H_kv, (unsigned)(B * n_q)), dim3(kThreads),
                     C::kSmemBytes, stream);
    const cudaError_t err = cudaLaunchKernelEx(
        &launch.cfg, split_decode_kernel<D, true, false, false>, reinterpret_cast<const __nv_bfloat16 *>(q), n_q,
        H_q, H_kv, H_q / H_kv, static_cast<const void *>(k_pool), static_cast<const void *>(v_pool), num_slots,
        table, table_stride, lens, scale_log2, out, lse, ws, n_split, (int32_t)0, (int32_t)0,
        AppendView{nullptr, nullptr, nullptr, nullptr, nullptr, 0}, ExtendView{nullptr, nullptr, 0, 0, 0},
        Fp8View{nullptr, nullptr}, RingView{nullptr, nullptr, 0, 0, 0, 0, 0}, CUtensorMap{}, CUtensorMap{}, (int32_t)0);
    return err == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

}  // namespace

cudaError_t read_attn_error(int32_t *code, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(code, g_attn_error, sizeof(int32_t));
    if (err != cudaSuccess || !clear) return err;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_attn_error, &zero, sizeof(int32_t));
}

}  // namespace wmtp

using namespace wmtp;

extern "C" {

size_t wmtp_attn_workspace_bytes(int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t D,
                                 int32_t n_split) {
    if (B < 0 || n_q < 0 || H_q < 0 || H_kv < 1 || D < 1 || n_split < 1) return 0;
    return workspace_bytes((int64_t)B * n_q * H_q, (int64_t)B * n_q * H_kv, D, n_split);
}

wmtp_status wmtp_attn_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (workspace_bytes == 0) return WMTP_OK;
    if (!workspace) return WMTP_EINVAL;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, as_stream(stream)) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"

namespace wmtp {
namespace {

// Split count of a row set: `per_sm` resident CTAs per SM of the instance,
// cluster capacity from the same instance.
template <bool F>
int32_t num_splits_for(int32_t B, int32_t n_q, int32_t H_kv, int64_t max_len, int per_sm) {
    int dev = 0, sms = 152;
    bool sms_known = false;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
        sms_known = true;
    cudaGetLastError();
    const int64_t rows = (int64_t)(B > 0 ? B : 1) * (n_q > 0 ? n_q : 1) * (H_kv > 0 ? H_kv : 1);
    const int64_t tiles = (max_len + kTileKeys - 1) / kTileKeys;
    const int64_t by_sms = (int64_t)sms * per_sm / rows;  // every resident CTA slot, one wave
    int64_t n;
    if (tiles >= 4 * by_sms) {
        // long rows: fill the SMs; the merge is small next to the copies
        n = by_sms;
    } else {
        // short rows: the launch is latency-bound and the load rate of one
        // SM is capped, so spread the row over the SMs, two key tiles per
        // split at least.  Above one cluster, keep to whole clusters of 16
        // (two-level merge) that are all resident at once: a merge through
        // global memory costs more than the extra SMs save on such rows.
        const int64_t half = tiles / 2;
        n = by_sms < half ? by_sms : half;
        if (n > kMaxClusterMerge) {
            int cap = 0;
            if (sms_known) cap = cluster_capacity<256, F>(dev, kMaxClusterMerge);
            n = n / kMaxClusterMerge * kMaxClusterMerge;
            if (n > kMaxClusterMerge * kMaxClusters) n = kMaxClusterMerge * kMaxClusters;
            while (n > kMaxClusterMerge && rows * (n / kMaxClusterMerge) > cap) n -= kMaxClusterMerge;
        }
    }
    if (n < 1) n = 1;
    if (n > kMaxSplits) n = kMaxSplits;
    // Up to one cluster: drop splits the whole-tile chunks leave empty (the
    // chunk of n splits covers ceil(tiles / n) tiles).
    if (n <= kMaxClusterMerge && tiles > 0) {
        const int64_t per = (tiles + n - 1) / n;
        n = (tiles + per - 1) / per;
    }
    return (int32_t)n;
}

}  // namespace
}  // namespace wmtp

extern "C" {

int32_t wmtp_attn_num_splits(int32_t B, int32_t n_q, int32_t H_kv, int64_t max_len) {
    return num_splits_for<false>(B, n_q, H_kv, max_len, 1);
}

int32_t wmtp_attn_num_splits_fp8(int32_t B, int32_t n_q, int32_t H_kv, int64_t max_len) {
    return num_splits_for<true>(B, n_q, H_kv, max_len, 1);
}

}  // extern "C"

namespace wmtp {
namespace {

wmtp_status draft_decode_attn_checked(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                      int32_t H_kv, int32_t D, const void *k_pool,
                                      const void *v_pool, int64_t num_slots,
                                      const int32_t *table, int64_t table_stride,
                                      const int32_t *lens, float scale, float *out, float *lse,
                                      void *workspace, size_t workspace_bytes_, int32_t n_split,
                                      void *stream, AppendView ap,
                                      ExtendView ev = ExtendView{nullptr, nullptr, 0, 0, 0},
                                      Fp8View fv = Fp8View{nullptr, nullptr},
                                      RingView rv = RingView{nullptr, nullptr, 0, 0, 0, 0, 0}) {
    if (B < 0 || n_q < 0 || H_q < 1 || H_kv < 1 || (H_q % H_kv) != 0) return WMTP_EINVAL;
    if (H_q / H_kv > kMaxGroup) return WMTP_EINVAL;
    if (D != 128 && D != 256) return WMTP_EINVAL;
    if (n_split < 1 || n_split > kMaxSplits || table_stride < 1 || num_slots < 0)
        return WMTP_EINVAL;
    if ((int64_t)B * n_q > 65535 || H_kv > 65535) return WMTP_EINVAL;
    if (ap.n_new < 0 || ap.n_new > kMaxNew) return WMTP_EINVAL;
    if (B == 0 || n_q == 0) return WMTP_OK;
    if (!q || !k_pool || !v_pool || !out) return WMTP_EINVAL;
    if (!rv.seq_lens && (!table || !lens)) return WMTP_EINVAL;
    if (rv.seq_lens && !rv.ring_base) return WMTP_EINVAL;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(q) & 3u))
        return WMTP_EINVAL;
    if (ap.n_new > 0 && (!ap.k_new || !ap.v_new || (!ap.slots && !rv.seq_lens) || !aligned16(ap.k_new) ||
                         !aligned16(ap.v_new)))
        return WMTP_EINVAL;
    if (n_split > 1) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return WMTP_EINVAL;
        if (workspace_bytes_ < wmtp_attn_workspace_bytes(B, n_q, H_q, H_kv, D, n_split))
            return WMTP_ECAPACITY;
    }
    cudaStream_t s = as_stream(stream);
    if (ev.seq_lens && !fv.k_scale && !rv.seq_lens && n_q >= 2 && n_q <= kMaxExtendTokens &&
        n_split <= kTreeExtendMaxSplits && table_stride >= kTreeExtendMinKeys && aligned16(q)) {
        // long rows: the tokens of a request are one MMA row block on the
        // tensor cores, each union key read once
        WorkspaceView w{nullptr, nullptr, nullptr};
        if (n_split > 1) w = carve(workspace, (int64_t)B * n_q * H_q, (int64_t)B * n_q * H_kv, n_split);
        return tree_extend_launch(static_cast<const uint16_t *>(q), B, n_q, H_q, H_kv, D,
                                  static_cast<const uint16_t *>(k_pool), static_cast<const uint16_t *>(v_pool),
                                  num_slots, table, table_stride, lens, ev.seq_lens, ev.n_new, ev.n_sink,
                                  ev.window, ev.windowed, scale, out, lse, w.counters, w.lse_part, w.o_part,
                                  n_split, s);
    }
    if (ev.seq_lens && !fv.k_scale && !rv.seq_lens && n_q >= 2 && n_q <= kMaxExtendTokens &&
        n_split <= kMaxExtendSplits && table_stride >= (int64_t)kExtendMinKeysPerSplit * n_split) {
        // several new tokens per request: one K/V read serves them all
        WorkspaceView w{nullptr, nullptr, nullptr};
        if (n_split > 1) w = carve(workspace, (int64_t)B * n_q * H_q, (int64_t)B * n_q * H_kv, n_split);
        return extend_multi_launch(static_cast<const uint16_t *>(q), B, n_q, H_q, H_kv, D,
                                   static_cast<const uint16_t *>(k_pool), static_cast<const uint16_t *>(v_pool),
                                   num_slots, table, table_stride, lens, ev.seq_lens, ev.n_new, ev.n_sink,
                                   ev.window, ev.windowed, scale, out, lse, w.counters, w.lse_part, w.o_part,
                                   n_split, s);
    }
    if (fv.k_scale) {
        if (!fv.v_scale) return WMTP_EINVAL;
        if (D == 256)
            return launch_split_decode<256, true>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots, table,
                                                  table_stride, lens, scale, out, lse, workspace, n_split, s,
                                                  ap, ev, fv, rv);
        return launch_split_decode<128, true>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots, table,
                                              table_stride, lens, scale, out, lse, workspace, n_split, s, ap,
                                              ev, fv, rv);
    }
    if (D == 256)
        return launch_split_decode<256, false>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots, table,
                                               table_stride, lens, scale, out, lse, workspace, n_split, s, ap,
                                               ev, fv, rv);
    return launch_split_decode<128, false>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots, table,
                                           table_stride, lens, scale, out, lse, workspace, n_split, s, ap, ev,
                                           fv, rv);
}

wmtp_status append_entry(const uint16_t *k_new, const uint16_t *v_new, const int32_t *new_slots, int32_t n_new,
                         const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv, int32_t D,
                         uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots, const int32_t *table,
                         int64_t table_stride, const int32_t *lens, float scale, float *out, float *lse,
                         void *workspace, size_t workspace_bytes_, int32_t n_split, int32_t chain,
                         int32_t hold, void *stream) {
    if (n_new < 1) return WMTP_EINVAL;
    const AppendView ap{reinterpret_cast<const __nv_bfloat16 *>(k_new),
                        reinterpret_cast<const __nv_bfloat16 *>(v_new), new_slots,
                        reinterpret_cast<__nv_bfloat16 *>(k_pool),
                        reinterpret_cast<__nv_bfloat16 *>(v_pool), n_new, chain, hold};
    return draft_decode_attn_checked(q, B, n_q, H_q, H_kv, D, k_pool, v_pool, num_slots, table,
                                     table_stride, lens, scale, out, lse, workspace,
                                     workspace_bytes_, n_split, stream, ap);
}

wmtp_status ring_entry(const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q, int32_t B, int32_t H_q,
                       int32_t H_kv, int32_t D, uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots,
                       const int32_t *seq_lens, const int32_t *ring_base, int32_t step, int32_t n_sink,
                       int32_t window, int32_t depth, int32_t tree_k, float scale, float *out, float *lse,
                       void *workspace, size_t workspace_bytes_, int32_t n_split, int32_t chain, int32_t hold,
                       void *stream) {
    if (n_sink < 0 || window < 1 || depth < 1 || tree_k < 1 || step < 0) return WMTP_EINVAL;
    // ring slots and positions stay below 2^31 (the kernel maps them in
    // 32-bit arithmetic)
    if ((int64_t)n_sink + window + (int64_t)depth * tree_k > (int64_t)1 << 30 || num_slots > INT32_MAX)
        return WMTP_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return WMTP_EINVAL;
    if (chain && k_new == nullptr) return WMTP_EINVAL;  // chained steps append
    if (B > 0 && (!seq_lens || !ring_base)) return WMTP_EINVAL;
    const AppendView ap = k_new ? AppendView{reinterpret_cast<const __nv_bfloat16 *>(k_new),
                                             reinterpret_cast<const __nv_bfloat16 *>(v_new), nullptr,
                                             reinterpret_cast<__nv_bfloat16 *>(k_pool),
                                             reinterpret_cast<__nv_bfloat16 *>(v_pool), 1, chain, hold}
                                : AppendView{nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, 0};
    return draft_decode_attn_checked(q, B, 1, H_q, H_kv, D, k_pool, v_pool, num_slots, nullptr,
                                     (int64_t)n_sink + window, nullptr, scale, out, lse, workspace,
                                     workspace_bytes_, n_split, stream, ap, ExtendView{nullptr, nullptr, 0, 0, 0},
                                     Fp8View{nullptr, nullptr},
                                     RingView{seq_lens, ring_base, n_sink, window, depth, tree_k, step});
}

}  // namespace
}  // namespace wmtp

extern "C" {

wmtp_status wmtp_draft_decode_attn(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                   int32_t H_kv, int32_t D, const uint16_t *k_pool,
                                   const uint16_t *v_pool, int64_t num_slots,
                                   const int32_t *table, int64_t table_stride,
                                   const int32_t *lens, float scale, float *out, float *lse,
                                   void *workspace, size_t workspace_bytes_, int32_t n_split,
                                   void *stream) {
    return draft_decode_attn_checked(q, B, n_q, H_q, H_kv, D, k_pool, v_pool, num_slots, table,
                                     table_stride, lens, scale, out, lse, workspace,
                                     workspace_bytes_, n_split, stream,
                                     AppendView{nullptr, nullptr, nullptr, nullptr, nullptr, 0});
}

wmtp_status wmtp_draft_decode_attn_append(const uint16_t *k_new, const uint16_t *v_new,
                                          const int32_t *new_slots, int32_t n_new,
                                          const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                          int32_t H_kv, int32_t D, uint16_t *k_pool,
                                          uint16_t *v_pool, int64_t num_slots,
                                          const int32_t *table, int64_t table_stride,
                                          const int32_t *lens, float scale, float *out,
                                          float *lse, void *workspace, size_t workspace_bytes_,
                                          int32_t n_split, void *stream) {
    return wmtp::append_entry(k_new, v_new, new_slots, n_new, q, B, n_q, H_q, H_kv, D, k_pool, v_pool,
                              num_slots, table, table_stride, lens, scale, out, lse, workspace,
                              workspace_bytes_, n_split, 0, 0, stream);
}

wmtp_status wmtp_draft_decode_attn_append_overlap(const uint16_t *k_new, const uint16_t *v_new,
                                                  const int32_t *new_slots, int32_t n_new,
                                                  const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                                  int32_t H_kv, int32_t D, uint16_t *k_pool,
                                                  uint16_t *v_pool, int64_t num_slots,
                                                  const int32_t *table, int64_t table_stride,
                                                  const int32_t *lens, float scale, float *out,
                                                  float *lse, void *workspace, size_t workspace_bytes_,
                                                  int32_t n_split, int32_t hold, void *stream) {
    if (hold < -1) return WMTP_EINVAL;
    return wmtp::append_entry(k_new, v_new, new_slots, n_new, q, B, n_q, H_q, H_kv, D, k_pool, v_pool,
                              num_slots, table, table_stride, lens, scale, out, lse, workspace,
                              workspace_bytes_, n_split, 1, hold, stream);
}

wmtp_status wmtp_draft_extend_attn(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                   int32_t H_kv, int32_t D, const uint16_t *k_pool,
                                   const uint16_t *v_pool, int64_t num_slots,
                                   const int32_t *table, int64_t table_stride,
                                   const int32_t *lens, const int32_t *seq_lens,
                                   const int32_t *n_new, int32_t n_sink, int32_t window,
                                   int32_t windowed, float scale, float *out, float *lse,
                                   void *workspace, size_t workspace_bytes_, int32_t n_split,
                                   void *stream) {
    if (!seq_lens || !n_new || n_sink < 0 || window < 1) return WMTP_EINVAL;
    return draft_decode_attn_checked(q, B, n_q, H_q, H_kv, D, k_pool, v_pool, num_slots, table,
                                     table_stride, lens, scale, out, lse, workspace,
                                     workspace_bytes_, n_split, stream,
                                     AppendView{nullptr, nullptr, nullptr, nullptr, nullptr, 0},
                                     ExtendView{seq_lens, n_new, n_sink, window, windowed ? 1 : 0});
}

wmtp_status wmtp_draft_decode_attn_noalloc(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                           int32_t H_kv, int32_t D, const uint16_t *k_pool,
                                           const uint16_t *v_pool, int64_t num_slots,
                                           const int32_t *table, int64_t table_stride,
                                           const int32_t *lens, float scale, float *out,
                                           float *lse, int32_t n_split, void *stream) {
    if (B < 0 || n_q < 0 || H_q < 1 || H_kv < 1 || (H_q % H_kv) != 0) return WMTP_EINVAL;
    if (H_q / H_kv > kMaxGroup) return WMTP_EINVAL;
    if (D != 128 && D != 256) return WMTP_EINVAL;
    if (n_split < 1 || n_split > kMaxSplits || table_stride < 1 || num_slots < 0)
        return WMTP_EINVAL;
    if ((int64_t)B * n_q > 65535 || H_kv > 65535) return WMTP_EINVAL;
    if (B == 0 || n_q == 0) return WMTP_OK;
    if (!q || !k_pool || !v_pool || !table || !lens || !out) return WMTP_EINVAL;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(q) & 3u))
        return WMTP_EINVAL;
    if (n_split > 1) {
        const int64_t rows_q = (int64_t)B * n_q * H_q;
        const int64_t rows_kv = (int64_t)B * n_q * H_kv;
        if (rows_kv > WMTP_NOALLOC_MAX_COUNTERS ||
            noalloc_partial_bytes(rows_q, D, n_split) > kNoAllocBytes - kNoAllocCounterBytes)
            return WMTP_ECAPACITY;
    }
    cudaStream_t s = as_stream(stream);
    if (D == 256)
        return launch_split_decode_noalloc<256>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots,
                                                table, table_stride, lens, scale, out, lse, n_split, s);
    return launch_split_decode_noalloc<128>(q, B, n_q, H_q, H_kv, k_pool, v_pool, num_slots, table,
                                            table_stride, lens, scale, out, lse, n_split, s);
}

}  // extern "C"

extern "C" {

wmtp_status wmtp_draft_decode_attn_fp8(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
                                       int32_t H_kv, int32_t D, const uint8_t *k_pool,
                                       const uint8_t *v_pool, const float *k_scale,
                                       const float *v_scale, int64_t num_slots,
                                       const int32_t *table, int64_t table_stride,
                                       const int32_t *lens, float scale, float *out, float *lse,
                                       void *workspace, size_t workspace_bytes_, int32_t n_split,
                                       void *stream) {
    if (B > 0 && n_q > 0 && (!k_scale || !v_scale)) return WMTP_EINVAL;
    return draft_decode_attn_checked(q, B, n_q, H_q, H_kv, D, k_pool, v_pool, num_slots, table,
                                     table_stride, lens, scale, out, lse, workspace,
                                     workspace_bytes_, n_split, stream,
                                     AppendView{nullptr, nullptr, nullptr, nullptr, nullptr, 0},
                                     ExtendView{nullptr, nullptr, 0, 0, 0}, Fp8View{k_scale, v_scale});
}

}  // extern "C"

extern "C" {

wmtp_status wmtp_draft_decode_attn_ring(const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q,
                                        int32_t B, int32_t H_q, int32_t H_kv, int32_t D, uint16_t *k_pool,
                                        uint16_t *v_pool, int64_t num_slots, const int32_t *seq_lens,
                                        const int32_t *ring_base, int32_t step, int32_t n_sink,
                                        int32_t window, int32_t depth, int32_t tree_k, float scale,
                                        float *out, float *lse, void *workspace, size_t workspace_bytes_,
                                        int32_t n_split, void *stream) {
    return wmtp::ring_entry(k_new, v_new, q, B, H_q, H_kv, D, k_pool, v_pool, num_slots, seq_lens, ring_base,
                            step, n_sink, window, depth, tree_k, scale, out, lse, workspace, workspace_bytes_,
                            n_split, 0, 0, stream);
}

wmtp_status wmtp_draft_decode_attn_ring_overlap(const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q,
                                                int32_t B, int32_t H_q, int32_t H_kv, int32_t D, uint16_t *k_pool,
                                                uint16_t *v_pool, int64_t num_slots, const int32_t *seq_lens,
                                                const int32_t *ring_base, int32_t step, int32_t n_sink,
                                                int32_t window, int32_t depth, int32_t tree_k, float scale,
                                                float *out, float *lse, void *workspace,
                                                size_t workspace_bytes_, int32_t n_split, int32_t hold,
                                                void *stream) {
    if (hold < -1) return WMTP_EINVAL;
    return wmtp::ring_entry(k_new, v_new, q, B, H_q, H_kv, D, k_pool, v_pool, num_slots, seq_lens, ring_base,
                            step, n_sink, window, depth, tree_k, scale, out, lse, workspace, workspace_bytes_,
                            n_split, 1, hold, stream);
}

}  // extern "C"
