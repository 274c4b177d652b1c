// wmtp_tree.cu -- tree-draft attention over the ring on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory) for sm_103a.
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
// The request's key list is implicit -- sinks || committed window of the
// shallowest node || the k*d draft nodes -- and ring slots are computed in
// the kernel (no table read).  The 224 query rows of a KV head (28 nodes x 8
// heads at k = 4, d = 7) meet every key of the window: a dense contraction.
//
// One CTA = 128 query rows (the MMA's M) x one key chunk of one request and
// KV head.  Warp roles:
//   warps 0-3  softmax: thread i owns query row i = tensor-memory lane i.  It
//              first writes its row of Q into tensor memory (the A operand of
//              QK), then per 64-key tile reads its row of S = Q K^T, applies
//              the tree-causal mask, keeps a running reference max (the O
//              accumulator is rescaled in tensor memory only when the max
//              grows by more than 2^8), writes P as bf16 head + tail over its
//              row of S, and at the end reads its row of O.
//   warps 4-7  gather: slots from the ring rule (or a table, below); 32-key
//              copy stages of consecutive slots arrive as TMA boxes (64 dims
//              x 1 head x 32 or 8 slots, 128-byte swizzle), other keys
//              through 16-byte cp.async into the same swizzled layout, each
//              warp one 8-key group; six stages, two per MMA tile.  Ring
//              chunks of 16 or more MMA tiles take the split instance: two
//              warps copy K rows, two V rows (one 8-key group in two each),
//              against separate K and V stage barriers, so that K is
//              refilled once its QK product is done, before V is free.
//   warp 8     one thread issues the MMAs: S(t) = Q K(t)^T (M=128, N=64,
//              K=D) into one of two S buffers, then O += P_hi V + P_lo V
//              (M=128, N=D, K=64); completion is signalled through mbarriers
//              with tcgen05.commit.  Q and P are read from tensor memory
//              (the A operands); K is K-major and V MN-major in shared
//              memory, both 128-byte swizzled.
// Table mode (the draft-extend pass of a chain): the key list of request b
// is the union table row of its accepted tokens, tree_k = 1 and depth = the
// tokens per request; token i at position S + i sees keep(S + i + 1), the
// same key sets as node (0, i) above.
// Key chunks are split over CTAs; up to 8 chunks of a (request, KV head,
// row block) run as one cluster and merge through distributed shared memory,
// more through the workspace: when the whole grid is resident, every chunk
// merges its own slice of the outputs once all have arrived (slice merge),
// else the last CTA merges in split order.  Every wait has a time limit;
// tensor memory is always released.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"
#include "wmtp_ring.cuh"
#include "wmtp_tc.cuh"

namespace wmtp {
namespace {

__device__ int32_t g_tree_tc_error = 0;

__device__ __forceinline__ void latch(int32_t code) { atomicCAS(&g_tree_tc_error, 0, code); }

constexpr int kRows = 128;  // query rows per CTA (MMA M)
constexpr int kKeys = 64;      // keys per MMA tile (N of QK^T, K of PV)
constexpr int kCopyKeys = 32;  // keys per copy stage: two stages make one MMA tile
constexpr int kKvStages = 6;   // copy stages (even: an MMA tile never wraps the ring)
// ring-mode chunks of at least this many MMA tiles take the split-role
// instance (K rows refilled once QK is done); shorter ones the combined one
constexpr int kSplitMinTiles = 16;
static_assert(kKeys == 2 * kCopyKeys && kKvStages % 2 == 0, "stage pairing");
constexpr int kSoftWarps = 4;
constexpr int kLoadWarps = 4;  // gather warps: warp w copies the 8-key groups w, w + 4, ...
constexpr int kLoadThreads = kLoadWarps * 32;
constexpr int kMmaWarp = kSoftWarps + kLoadWarps;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kMaxSplits = 128;
constexpr int kMaxClusterSplits = 8;  // key chunks merged through one (portable) cluster
constexpr uint64_t kSlicePollNs = 50000;  // a slice-merge wait gives up after 50 us (results stay exact)
constexpr float kLazyRescale = 8.f;  // log2 of the growth tolerated before rescaling O
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLn2 = 0.69314718055994530942f;

// Barrier slots: K/V copy stages, S buffers (2), P (2, written over S), PV
// done (2, which also frees the S buffer), Q.
enum {
    kKFull = 0,                      // K rows of a copy stage landed (table instance: K and V)
    kVFull = kKFull + kKvStages,     // V rows of a copy stage landed (ring instance)
    kKEmpty = kVFull + kKvStages,    // QK done with a stage's K rows (table instance: PV done with it)
    kVEmpty = kKEmpty + kKvStages,   // PV done with a stage's V rows (ring instance)
    kSFull = kVEmpty + kKvStages,
    kPFull = kSFull + 2,
    kPvDone = kPFull + 2,
    kQFull = kPvDone + 2,
    kNumBars = kQFull + 1
};

template <int D>
struct Cfg {
    // K and V each sit in shared memory as D/64 rings of 128-byte rows (one
    // ring per 64-dim swizzle atom column, the 128-byte-swizzled K-major
    // layout the MMAs read): copy stage st holds rows st*32 .. st*32+31 of
    // every ring, so the two stages of an MMA tile are 64 consecutive rows,
    // one operand with a uniform 8-row stride.
    static constexpr int kCopyBytes = kCopyKeys * D * 2;     // K (or V) rows of one copy stage
    static constexpr int kRingBlockBytes = kKvStages * kCopyKeys * 128;
    static constexpr int kRegionBytes = (D / 64) * kRingBlockBytes;  // all of K (or V)
    static constexpr int kStageBytes = 2 * kCopyBytes;
    // cluster merge: lse of the 128 rows, then the merge weights of this
    // CTA's row slice (at most kRows + kMaxClusterSplits - 1 of them)
    static constexpr int kMergeBytes = kRows * 4 + (kRows + kMaxClusterSplits) * 4;
    static constexpr int kKvOff = 0;
    static constexpr int kKOff = kKvOff;
    static constexpr int kVOff = kKOff + kRegionBytes;
    static constexpr int kMergeOff = kVOff + kRegionBytes;
    static constexpr int kBarOff = kMergeOff + kMergeBytes;
    static constexpr int kSmemUsed = kBarOff + kNumBars * 8 + 16 + 1024;  // + alignment slack
    static constexpr int kDimBlocks = D / 64;                 // 128-byte swizzle atoms per K/V row
    // tensor memory: S buffers (fp32, later P as bf16 head | tail), O, Q
    static constexpr int kOCol = 2 * kKeys;                  // O after the two S buffers
    static constexpr int kQCol = kOCol + D;                  // Q (A operand of QK): two bf16 per column
    static constexpr int kTmemCols = (kQCol + D / 2 <= 256) ? 256 : 512;
    static_assert(kQCol + D / 2 <= 512, "tensor memory budget");
    // at 512 tensor-memory columns a second CTA on the SM would only wait in
    // tcgen05.alloc: ask for more than half the SM's shared memory
    static constexpr int kSmemBytes =
        (kTmemCols == 512 && kSmemUsed < 116 * 1024) ? 116 * 1024 : kSmemUsed;
    static_assert(kRows * kMaxSplits * 4 <= kKvStages * kStageBytes, "merge weights must fit");
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kRows * D * 4 <= kKvStages * kStageBytes, "cluster-merge partial must fit the K/V stages");
};

struct TreeWs {
    int32_t *counters;
    float *lse_part;
    float *o_part;
};

// Slots from a table instead of the ring rule (the chain draft-extend pass,
// tree_k = 1, depth = tokens per request): entry e of request b's key list
// sits in slot table[b * stride + e], lens[b] (if given) must equal the
// list's length, and the request has n_new[b] nodes (rows of later nodes are
// empty: out = 0, lse = -inf).  table == nullptr: ring mode.
struct TreeTable {
    const int32_t *table;
    int64_t stride;
    const int32_t *lens;
    const int32_t *n_new;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

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

// Logical position and a code (-1 a committed key, else branch << 8 | depth
// of a draft node) of entry e of the key list.
__device__ __forceinline__ int2 key_info(const Geo &g, int64_t e, int depth) {
    if (e < g.Uc) return make_int2((int)(e < g.ns ? e : g.lo0 + (e - g.ns)), -1);
    const int64_t n = e - g.Uc;
    const int br = (int)(n / depth);
    const int dep = (int)(n - (int64_t)br * depth);
    return make_int2((int)(g.S + dep), (br << 8) | dep);
}

// The same slot in 32-bit arithmetic, for requests whose positions and ring
// slots are all below 2^31 (the caller checks): entry e of the key list is a
// sink (below ns), a committed key of the window (below Uc, at a position
// >= n_sink), or draft node e - Uc = branch * depth + depth index.
struct Geo32 {
    int32_t ns, Uc, lo0, S, base, n_sink, depth;
    uint32_t m;  // window + depth * tree_k
};

__device__ __forceinline__ int32_t tree_slot32(const Geo32 &g, int32_t e) {
    if (e < g.ns) return g.base + e;
    if (e < g.Uc) return g.base + g.n_sink + (int32_t)((uint32_t)(g.lo0 + (e - g.ns) - g.n_sink) % g.m);
    const int32_t n = e - g.Uc;
    const int32_t br = n / g.depth;
    const int32_t dep = n - br * g.depth;
    const int32_t p = g.S + dep;
    if (p < g.n_sink && br == 0) return g.base + p;
    int32_t r = (p - g.n_sink + br * g.depth) % (int32_t)g.m;
    if (r < 0) r += (int32_t)g.m;
    return g.base + g.n_sink + r;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int32_t *abort) {
    if (mbar_wait_bounded(smem_addr(bar), parity, kWaitNs)) return true;
    latch(WMTP_DEV_WAIT_TIMEOUT);
    *abort = 1;
    return false;
}

// Warp-uniform wait: the whole warp proceeds only if every lane saw the phase
// (tensor-memory loads and stores that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int32_t *abort) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

template <int D, bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) tree_tc_kernel(
    const __nv_bfloat16 *__restrict__ q, int32_t H_q, int32_t H_kv, int32_t G, int32_t n_nodes,
    const __nv_bfloat16 *__restrict__ k_pool, const __nv_bfloat16 *__restrict__ v_pool,
    int64_t num_slots, const int32_t *__restrict__ seq_lens, const int32_t *__restrict__ ring_base,
    int32_t n_sink, int32_t window, int32_t depth, int32_t tree_k, float scale_log2,
    float *__restrict__ out, float *__restrict__ lse, TreeWs ws, TreeTable tt, int32_t n_split, int32_t n_rb,
    int32_t cluster_merge, int32_t slice_stride, const __grid_constant__ CUtensorMap tm_k32, const __grid_constant__ CUtensorMap tm_v32,
    const __grid_constant__ CUtensorMap tm_k8, const __grid_constant__ CUtensorMap tm_v8) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 128-byte-swizzled K/V tiles need 1024-byte aligned atoms
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOff);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int32_t *flags = reinterpret_cast<volatile int32_t *>(tmem_slot + 1);  // [0] abort [1] ticket

    griddep_launch_dependents();
    griddep_wait();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    const int64_t base = tt.table ? 0 : ring_base[b];
    int n_b = n_nodes;  // nodes of this request
    if (tt.n_new) {
        n_b = tt.n_new[b];
        n_b = n_b < 0 ? 0 : (n_b > n_nodes ? n_nodes : n_b);
    }
    Geo geo = geometry(S, n_sink, window, n_b);
    if (tt.table && n_b == 0) {
        geo.U = geo.Uc = 0;  // no node, no row to compute: every row is 0 / -inf
    } else if (tt.table && (geo.U > tt.stride || (tt.lens && tt.lens[b] != geo.U))) {
        // a table that does not hold this request's key list: no read past its row
        if (tid == 0) latch(WMTP_DEV_LEN_RANGE);
        geo.U = geo.U < tt.stride ? geo.U : tt.stride;
        geo.Uc = geo.Uc < geo.U ? geo.Uc : geo.U;
    }
    int64_t chunk = (geo.U + n_split - 1) / n_split;
    chunk = (chunk + kKeys - 1) / kKeys * kKeys;
    const int64_t start = (int64_t)split * chunk;
    const int64_t cnt = geo.U - start < 0 ? 0 : (geo.U - start < chunk ? geo.U - start : chunk);
    const int n_tiles = (int)((cnt + kKeys - 1) / kKeys);

    // kSplit (ring mode, long chunks): two gather warps copy K rows and two
    // V rows, so that a stage's K is refilled as soon as its QK product is
    // done, before its V.  Table mode and short chunks keep every gather
    // warp on both (the split roles measured slower there).
    if (tid == 0) {
        for (int i = 0; i < kKvStages; ++i) {
            // cp.async completions of the warps feeding the barrier plus one
            // byte-count arrival per such warp
            constexpr uint32_t n_full = kSplit ? kLoadThreads / 2 + kLoadWarps / 2 : kLoadThreads + kLoadWarps;
            mbar_init(smem_addr(&bars[kKFull + i]), n_full);
            mbar_init(smem_addr(&bars[kVFull + i]), n_full);
            mbar_init(smem_addr(&bars[kKEmpty + i]), 1);
            mbar_init(smem_addr(&bars[kVEmpty + i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_addr(&bars[kSFull + i]), 1);
            mbar_init(smem_addr(&bars[kPFull + i]), kSoftWarps);
            mbar_init(smem_addr(&bars[kPvDone + i]), 1);
        }
        mbar_init(smem_addr(&bars[kQFull]), kSoftWarps);
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc_alloc(smem_addr(tmem_slot), C::kTmemCols);

    const uint32_t sbase = smem_addr(smem);
    // ring mode: the row-block CTAs of a request read the same keys, keep
    // them in L2; table mode streams a long union row once
    const uint64_t keep = tt.table ? l2_policy_evict_first() : l2_policy_evict_last();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= kSoftWarps && warp < kMmaWarp) {
        // ----------------------------------------------------------- gather
        // Four warps, one 32-key copy stage at a time (two per MMA tile); in
        // every warp lane k computes the slot of key k.  A stage of 32 valid
        // keys in consecutive pool slots comes in as one TMA box per 64-dim
        // block of K and of V (64 dims x 1 head x 32 slots, 128-byte
        // swizzle), issued by the first warp.  Otherwise warp w takes 8-key
        // group w: a group of consecutive slots comes in as 8-slot boxes,
        // other keys (ring wrap, segment edges, the tail, bad slots, a paged
        // table) are copied or zero-filled with cp.async into the same
        // swizzled layout.  The stage barrier counts the 128 cp.async
        // arrivals and one byte-count arrival per warp.
        const int lw = warp - kSoftWarps;  // gather warp index
        // split: warps 0-1 copy K, 2-3 V, each one 8-key group in two;
        // otherwise every warp copies K and V of one 8-key group in four
        const bool is_v = kSplit && lw >= kLoadWarps / 2;
        constexpr int n_roles = kSplit ? kLoadWarps / 2 : kLoadWarps;
        const int hw = kSplit ? lw % (kLoadWarps / 2) : lw;
        const uint8_t *kbase = reinterpret_cast<const uint8_t *>(k_pool) + (size_t)g * D * 2;
        const uint8_t *vbase = reinterpret_cast<const uint8_t *>(v_pool) + (size_t)g * D * 2;
        const size_t slot_bytes = (size_t)H_kv * D * 2;
        const int64_t ring_m = (int64_t)window + (int64_t)depth * tree_k;
        const bool fits32 = base >= 0 && S + (int64_t)depth * tree_k < INT32_MAX && geo.U < INT32_MAX &&
                            base + n_sink + ring_m < INT32_MAX;
        const Geo32 g32{(int32_t)geo.ns, (int32_t)geo.Uc, (int32_t)geo.lo0, (int32_t)S, (int32_t)base,
                        n_sink, depth, (uint32_t)ring_m};
        auto slot_of = [&](int64_t e) -> int64_t {
            if (fits32) return tree_slot32(g32, (int32_t)e);
            const int2 inf = key_info(geo, e, depth);
            const int br = inf.y < 0 ? 0 : (inf.y >> 8);
            return ring_slot(base, inf.x, br, n_sink, window, depth, tree_k);
        };
        // table mode: each lane's slot of the next three copy stages in
        // registers, so that no issue waits on a table load
        const int32_t *trow = tt.table ? tt.table + b * tt.stride + start : nullptr;
        auto tab_load = [&](int t_) -> int32_t {
            const int64_t k2 = (int64_t)t_ * kCopyKeys + lane;
            return k2 < cnt ? __ldg(trow + k2) : 0;
        };
        int32_t pf0 = 0, pf1 = 0, pf2 = 0;
        if (trow) {
            pf0 = tab_load(0);
            pf1 = tab_load(1);
            pf2 = tab_load(2);
        }
        for (int t = 0; t < 2 * n_tiles; ++t) {  // copy stages; keys past cnt are zero-filled
            const int st = t % kKvStages;
            if (t >= kKvStages &&
                !mbar_wait(&bars[(is_v ? kVEmpty : kKEmpty) + st], ((t / kKvStages) - 1) & 1, flags))
                break;
            if (flags[0]) break;
            const uint32_t kt = sbase + C::kKOff + st * (kCopyKeys * 128);
            const uint32_t vt = sbase + C::kVOff + st * (kCopyKeys * 128);
            const uint32_t bar = smem_addr(&bars[(is_v ? kVFull : kKFull) + st]);
            // split: this warp's operand (xt, its pool and maps); both otherwise
            const uint32_t xt = is_v ? vt : kt;
            const int64_t kk = (int64_t)t * kCopyKeys + lane;
            int64_t slot = 0;
            bool ok = false;
            if (trow) {
                slot = pf0;
                pf0 = pf1;
                pf1 = pf2;
                pf2 = tab_load(t + 3);
            }
            if (kk < cnt) {
                if (!trow) slot = slot_of(start + kk);
                ok = slot >= 0 && slot < num_slots;
            }
            const int64_t prev = __shfl_up_sync(0xffffffffu, slot, 1);
            const bool whole = __all_sync(0xffffffffu, ok && (lane == 0 || slot == prev + 1));
            if (whole) {
                const int64_t slot0 = __shfl_sync(0xffffffffu, slot, 0);
                if (lane == 0 && hw == 0) {
                    if constexpr (kSplit) {
                        mbar_arrive_expect_tx(bar, (uint32_t)C::kCopyBytes);
#pragma unroll
                        for (int db = 0; db < C::kDimBlocks; ++db)
                            tma_load_3d(xt + db * C::kRingBlockBytes, is_v ? &tm_v32 : &tm_k32, db * 64, g,
                                        (int32_t)slot0, bar);
                    } else {
                        mbar_arrive_expect_tx(bar, 2u * C::kCopyBytes);
#pragma unroll
                        for (int db = 0; db < C::kDimBlocks; ++db) {
                            tma_load_3d(kt + db * C::kRingBlockBytes, &tm_k32, db * 64, g, (int32_t)slot0, bar);
                            tma_load_3d(vt + db * C::kRingBlockBytes, &tm_v32, db * 64, g, (int32_t)slot0, bar);
                        }
                    }
                } else if (lane == 0) {
                    mbar_arrive(bar);
                }
            } else {
                if (lw == 0 && kk < cnt && !ok) latch(WMTP_DEV_SLOT_RANGE);
                // contiguity inside 8-key groups: key k continues key k-1's slot
                const bool cont = ok && ((lane & 7) == 0 || slot == prev + 1);
                const uint32_t contm = __ballot_sync(0xffffffffu, cont);
                const uint32_t okm = __ballot_sync(0xffffffffu, ok);
                uint32_t tma_groups = 0;  // bit gi: this warp's group gi by 8-slot TMA boxes
#pragma unroll
                for (int gi = 0; gi < kCopyKeys / 8; ++gi) {
                    const uint32_t gm = 0xffu << (gi * 8);
                    if (gi % n_roles == hw && (okm & gm) == gm && (contm & gm) == gm) tma_groups |= 1u << gi;
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(bar, (uint32_t)__popc(tma_groups) * (kSplit ? 1u : 2u) * 8u *
                                                   (uint32_t)(D * 2));
#pragma unroll
                for (int gi = 0; gi < kCopyKeys / 8; ++gi) {
                    if (gi % n_roles != hw) continue;
                    if ((tma_groups >> gi) & 1u) {
                        const int64_t gs = __shfl_sync(0xffffffffu, slot, gi * 8);
                        if (lane == 0) {
#pragma unroll
                            for (int db = 0; db < C::kDimBlocks; ++db) {
                                if constexpr (kSplit) {
                                    tma_load_3d(xt + db * C::kRingBlockBytes + gi * 1024, is_v ? &tm_v8 : &tm_k8,
                                                db * 64, g, (int32_t)gs, bar);
                                } else {
                                    tma_load_3d(kt + db * C::kRingBlockBytes + gi * 1024, &tm_k8, db * 64, g,
                                                (int32_t)gs, bar);
                                    tma_load_3d(vt + db * C::kRingBlockBytes + gi * 1024, &tm_v8, db * 64, g,
                                                (int32_t)gs, bar);
                                }
                            }
                        }
                    } else {
                        // 8 keys x D/8 16-byte chunks over 32 lanes; kept
                        // rolled: its code shares the instruction cache with
                        // the other roles' (unrolled by four, the table-mode
                        // pass over a 1M union ran ~20% slower)
#pragma unroll 1
                        for (int idx = lane; idx < 8 * (D / 8); idx += 32) {
                            const int kr = gi * 8 + (idx >> (D == 256 ? 5 : 4));
                            const int c = idx & (D / 8 - 1);
                            const int64_t sl = __shfl_sync(0xffffffffu, slot, kr);  // uniform index per 32 idx
                            const bool kok = (okm >> kr) & 1u;
                            const size_t off = kok ? (size_t)sl * slot_bytes + c * 16 : 0;
                            const int db = c >> 3, cb = c & 7;
                            const uint32_t dst = db * C::kRingBlockBytes + kr * 128 + ((cb ^ (kr & 7)) << 4);
                            if constexpr (kSplit) {
                                cp_async_16(xt + dst, (is_v ? vbase : kbase) + off, kok ? 16u : 0u, keep);
                            } else {
                                cp_async_16(kt + dst, kbase + off, kok ? 16u : 0u, keep);
                                cp_async_16(vt + dst, vbase + off, kok ? 16u : 0u, keep);
                            }
                        }
                    }
                }
            }
            cp_async_mbar_arrive(bar);
        }
        cp_async_wait<0>();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc_idesc_bf16(kRows, kKeys, 0);
            constexpr uint32_t idesc_pv = tc_idesc_bf16(kRows, D, 1);
            // MMA tile t = copy stages s0, s0 + 1 (same pass over the ring)
            auto issue_qk = [&](int t) -> bool {
                const int s0 = (2 * t) % kKvStages, sb = t & 1;
                const uint32_t ph = (uint32_t)((2 * t) / kKvStages) & 1u;
                if (t == 0 && !mbar_wait(&bars[kQFull], 0, flags)) return false;
                if (!mbar_wait(&bars[kKFull + s0], ph, flags)) return false;
                if (!mbar_wait(&bars[kKFull + s0 + 1], ph, flags)) return false;
                // S buffer sb last held P of tile t-2: its PV must be done
                if (t >= 2 && !mbar_wait(&bars[kPvDone + sb], ((t >> 1) - 1) & 1, flags)) return false;
                fence_proxy_async_smem();  // cp.async writes -> tensor-core reads
                tc_fence_after();
                const uint32_t kt = sbase + C::kKOff + s0 * (kCopyKeys * 128);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_bf16_ta(tmem + sb * kKeys, tmem + C::kQCol + kk * 8,
                                   tc_smem_desc_sw128(kt + (kk / 4) * C::kRingBlockBytes + (kk % 4) * 32, 16, 1024),
                                   idesc_qk, kk > 0);
                tc_commit(smem_addr(&bars[kSFull + sb]));
                if constexpr (kSplit) {
                    // the stage pair's K rows are free once this product is done
                    tc_commit(smem_addr(&bars[kKEmpty + s0]));
                    tc_commit(smem_addr(&bars[kKEmpty + s0 + 1]));
                }
                return true;
            };
            bool live = n_tiles == 0 || issue_qk(0);
            for (int t = 0; live && t < n_tiles; ++t) {
                if (t + 1 < n_tiles && !issue_qk(t + 1)) break;
                const int pb = t & 1;
                if (!mbar_wait(&bars[kPFull + pb], (t >> 1) & 1, flags)) break;
                const int s0 = (2 * t) % kKvStages;
                if constexpr (kSplit) {
                    const uint32_t vph = (uint32_t)((2 * t) / kKvStages) & 1u;
                    if (!mbar_wait(&bars[kVFull + s0], vph, flags)) break;
                    if (!mbar_wait(&bars[kVFull + s0 + 1], vph, flags)) break;
                    fence_proxy_async_smem();  // cp.async writes -> tensor-core reads
                }
                tc_fence_after();
                const uint32_t vt = sbase + C::kVOff + s0 * (kCopyKeys * 128);
                // P was written over S buffer pb: head in its first half, tail in the second
                const uint32_t p_hi = tmem + pb * kKeys, p_lo = p_hi + kKeys / 2;
#pragma unroll
                for (int kk = 0; kk < kKeys / 16; ++kk) {
                    const uint64_t vd = tc_smem_desc_sw128(vt + kk * 16 * 128, C::kRingBlockBytes, 1024);
                    tc_mma_bf16_ta(tmem + C::kOCol, p_hi + kk * 8, vd, idesc_pv, (t > 0 || kk > 0));
                    tc_mma_bf16_ta(tmem + C::kOCol, p_lo + kk * 8, vd, idesc_pv, 1);
                }
                tc_commit(smem_addr(&bars[kPvDone + pb]));
                tc_commit(smem_addr(&bars[(kSplit ? kVEmpty : kKEmpty) + s0]));
                tc_commit(smem_addr(&bars[(kSplit ? kVEmpty : kKEmpty) + s0 + 1]));
            }
        }
    } else {
        // --------------------------------------------------------- softmax
        // Q row `tid` of this block -> tensor-memory lane tid (A operand of
        // QK), while the gather warp already fetches the first tiles.
        {
            const int rq = rb * kRows + tid;
            const bool live = rq < R;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(
                q + ((b * n_nodes + (live ? rq / G : 0)) * H_q + g * G + (live ? rq % G : 0)) * (int64_t)D);
            const uint32_t qlane = tmem + ((uint32_t)(warp * 32) << 16) + C::kQCol;
            // the whole row in flight at once (one memory round trip), then
            // into tensor memory 32 columns at a time
            uint4 qv[D / 8];
#pragma unroll
            for (int j = 0; j < D / 8; ++j)
                qv[j] = live ? __ldg(reinterpret_cast<const uint4 *>(src) + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c0 = 0; c0 < D / 2; c0 += 32) {
                uint32_t r[32];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint4 v = qv[c0 / 4 + j];
                    r[4 * j] = v.x;
                    r[4 * j + 1] = v.y;
                    r[4 * j + 2] = v.z;
                    r[4 * j + 3] = v.w;
                }
                tc_st32(qlane + c0, r);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[kQFull]));
        }
        const int i = tid;  // row = tensor-memory lane
        const int rq = rb * kRows + i;
        const bool row_valid = rq < R;            // a row of the output
        const bool row_live = row_valid && rq / G < n_b;  // ... of a node this request has
        const int node = row_live ? rq / G : 0;
        const int rbr = node / depth, rdep = node - (node / depth) * depth;
        const int64_t kv = S + rdep + 1;
        const int64_t row_lo = kv > (int64_t)n_sink + window ? kv - window : 0;
        // Committed entry e (position e below ns, lo0 + e - ns after) is in the
        // row's key set iff e < ns or its position >= row_lo; draft node n is
        // iff it is on the row's branch at depth <= the row's depth and its
        // position S + depth is a sink or >= row_lo.
        const int Uc = (int)geo.Uc, ns = (int)geo.ns;
        const int e_lo = ns + (int)(row_lo - geo.lo0 > 0 ? row_lo - geo.lo0 : 0);
        const int n0 = rbr * depth, n_hi = n0 + rdep;
        const int d_sink = (int)((int64_t)n_sink - S);
        const int d_lo = (int)(row_lo - S);
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m_ref = -INFINITY, l = 0.f;
        bool o_live = false;  // O holds at least one PV product
        for (int t = 0; t < n_tiles; ++t) {
            const int sb = t & 1, pb = t & 1;
            if (!warp_wait(&bars[kSFull + sb], (t >> 1) & 1, flags)) break;
            tc_fence_after();
            float x[kKeys];
#pragma unroll
            for (int c0 = 0; c0 < kKeys; c0 += 32) {
                uint32_t r0[32];
                tc_ld32(lane_base + sb * kKeys + c0, r0);
#pragma unroll
                for (int k = 0; k < 32; ++k) x[c0 + k] = __uint_as_float(r0[k]);
            }
            // Tree-causal mask from the key index alone, with per-row int32
            // thresholds (no loads, no division): entry e is a committed key
            // when e < Uc, else draft node n = e - Uc.  Tiles whose keys every
            // row of the warp sees skip the mask.
            const int e0 = (int)(start + (int64_t)t * kKeys);
            const int valid = (int)(cnt - (int64_t)t * kKeys);
            const bool lane_all = !row_valid || (row_live && (e0 + kKeys <= ns || e0 >= e_lo));
            const bool fast = valid >= kKeys && e0 + kKeys <= Uc && __all_sync(0xffffffffu, lane_all);
            float mx = -INFINITY;
            if (fast) {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) {
                    x[k] *= scale_log2;
                    mx = fmaxf(mx, x[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kKeys; ++k) {
                    const int e = e0 + k;
                    const int n = e - Uc;
                    const bool vis_c = (e < ns) | (e >= e_lo);
                    const bool vis_n =
                        (n >= n0) & (n <= n_hi) & (((n - n0) < d_sink) | ((n - n0) >= d_lo));
                    const bool vis = row_live & (k < valid) & (e < Uc ? vis_c : vis_n);
                    x[k] = vis ? x[k] * scale_log2 : -INFINITY;
                    mx = fmaxf(mx, x[k]);
                }
            }
            // Lazy rescale: the reference max moves only when a row's max grew
            // by more than 2^8 (also the first time it becomes finite).  The
            // rescale loop is warp-uniform; rows that keep their max use 1.
            const bool need = mx > m_ref + kLazyRescale;
            float alpha = 1.f;
            if (need) {
                alpha = exp2f(m_ref - mx);  // 0 when m_ref = -inf
                l *= alpha;
                m_ref = mx;
            }
            if (o_live && __any_sync(0xffffffffu, need)) {
                // O must hold PV(t-1) before it is rescaled
                if (!warp_wait(&bars[kPvDone + ((t - 1) & 1)], ((t - 1) >> 1) & 1, flags)) break;
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    tc_ld32(lane_base + C::kOCol + c0, r);
#pragma unroll
                    for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
                    tc_st32(lane_base + C::kOCol + c0, r);
                }
            }
            const float muse = m_ref == -INFINITY ? 0.f : m_ref;
            float rs = 0.f;
#pragma unroll
            for (int k = 0; k < kKeys; ++k) {
                x[k] = exp2f(x[k] - muse);
                rs += x[k];
            }
            l += rs;
            {
                // P over this row's S (read above): bf16 head in columns 0-31
                // and tail in 32-63 of the buffer, two keys per column.  No
                // MMA still reads the buffer: QK(t) was issued only after the
                // PV of tile t-2 had finished with it.
                uint32_t ph[kKeys / 2], pl[kKeys / 2];
#pragma unroll
                for (int u = 0; u < kKeys / 2; ++u) {
                    const float a = x[2 * u], c2 = x[2 * u + 1];
                    ph[u] = pack_bf16x2(a, c2);
                    pl[u] = pack_bf16x2(a - bf16_lo_to_f32(ph[u]), c2 - bf16_hi_to_f32(ph[u]));
                }
                static_assert(kKeys / 2 == 32, "one 32-column store per half");
                tc_st32(lane_base + pb * kKeys, ph);
                tc_st32(lane_base + pb * kKeys + kKeys / 2, pl);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[kPFull + pb]));
            o_live = true;
        }
        // ---------------------------------------------------- epilogue
        bool have_o = n_tiles > 0 && !flags[0];
        if (have_o)
            have_o = warp_wait(&bars[kPvDone + ((n_tiles - 1) & 1)], ((n_tiles - 1) >> 1) & 1, flags);
        have_o = __all_sync(0xffffffffu, have_o);
        tc_fence_after();
        const int h = g * G + (row_valid ? rq % G : 0);
        const int wnode = row_valid ? rq / G : 0;  // output row (a node without keys writes 0 / -inf)
        const float inv = (have_o && l > 0.f) ? 1.f / l : 0.f;
        const float lse2 = (have_o && l > 0.f) ? m_ref + log2f(l) : -INFINITY;
        float *dst = nullptr;
        // Cluster merge: this CTA's normalised partial O goes to its own
        // shared memory (the K/V stages, idle now), row-major with the
        // float4 index of row i XOR-swizzled by i % 8; its lse to the P area.
        float *po = reinterpret_cast<float *>(smem + C::kKvOff);
        if (cluster_merge) {
            reinterpret_cast<float *>(smem + C::kMergeOff)[i] = (row_live && !flags[0]) ? lse2 : -INFINITY;
        } else if (row_valid) {
            if (n_split == 1) {
                const int64_t orow = (b * n_nodes + wnode) * H_q + h;
                dst = out + orow * D;
                if (lse) lse[orow] = flags[0] ? NAN : lse2 * kLn2;
            } else {
                const int64_t prow = ((b * H_kv + g) * R + rq) * n_split + split;
                dst = ws.o_part + prow * D;
                ws.lse_part[prow] = flags[0] ? NAN : lse2;
            }
        }
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t r[32];
            if (have_o) tc_ld32(lane_base + C::kOCol + c0, r);  // warp-uniform
            if (cluster_merge) {
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    float4 v;
                    v.x = have_o ? __uint_as_float(r[k]) * inv : 0.f;
                    v.y = have_o ? __uint_as_float(r[k + 1]) * inv : 0.f;
                    v.z = have_o ? __uint_as_float(r[k + 2]) * inv : 0.f;
                    v.w = have_o ? __uint_as_float(r[k + 3]) * inv : 0.f;
                    const int d4 = (c0 + k) / 4;
                    reinterpret_cast<float4 *>(po + i * D)[d4 ^ (i & 7)] = v;
                }
            } else if (row_valid) {
#pragma unroll
                for (int k = 0; k < 32; k += 4) {
                    float4 v;
                    v.x = have_o ? __uint_as_float(r[k]) * inv : 0.f;
                    v.y = have_o ? __uint_as_float(r[k + 1]) * inv : 0.f;
                    v.z = have_o ? __uint_as_float(r[k + 2]) * inv : 0.f;
                    v.w = have_o ? __uint_as_float(r[k + 3]) * inv : 0.f;
                    *reinterpret_cast<float4 *>(dst + c0 + k) = v;
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tmem, C::kTmemCols);
    }
    if (n_split == 1) return;

    const int row0 = rb * kRows;
    const int n_rows = R - row0 < kRows ? R - row0 : kRows;
    constexpr int D4 = D / 4;
    if (cluster_merge) {
        // ------------------------------- merge through distributed smem
        // The n_split CTAs of this (request, KV head, row block) form one
        // cluster; CTA `rank` merges a slice of the rows, reading every
        // peer's partial in split order.  The closing barrier keeps each
        // CTA's shared memory alive until its peers have read it.
        __syncwarp();
        cluster_sync();
        const int rank = (int)cluster_ctarank();
        const int per = (n_rows + n_split - 1) / n_split;
        const int r_lo = rank * per;
        const int r_hi = r_lo + per < n_rows ? r_lo + per : n_rows;
        const uint32_t po_addr = smem_addr(smem + C::kKvOff);
        const uint32_t pl_addr = smem_addr(smem + C::kMergeOff);
        float *wts = reinterpret_cast<float *>(smem + C::kMergeOff + kRows * 4);  // [per][n_split] merge weights
        for (int i = r_lo + tid; i < r_hi; i += kThreads) {
            float ls[kMaxClusterSplits];
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
                ls[s2] = s2 < n_split ? ld_dsmem_f32(map_to_rank(pl_addr + i * 4, s2)) : -INFINITY;
            float M = -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) M = fmaxf(M, ls[s2]);
            float sum = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
                    sum += ls[s2] == -INFINITY ? 0.f : exp2f(ls[s2] - M);
            }
            const float lt = sum > 0.f ? M + log2f(sum) : -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
                if (s2 < n_split) wts[(i - r_lo) * n_split + s2] = (sum > 0.f && ls[s2] != -INFINITY) ? exp2f(ls[s2] - lt) : 0.f;
            const int rq = row0 + i;
            if (lse) lse[(b * n_nodes + rq / G) * H_q + g * G + rq % G] = lt * kLn2;
        }
        __syncthreads();
        for (int e = tid; e < (r_hi - r_lo) * D4; e += kThreads) {
            const int i = r_lo + e / D4, d4 = e - (e / D4) * D4;
            const float *w = wts + (i - r_lo) * n_split;
            const uint32_t off = (uint32_t)(i * D4 + (d4 ^ (i & 7))) * 16;
            float4 v[kMaxClusterSplits];
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterSplits; ++s2)
                if (s2 < n_split) v[s2] = ld_dsmem_f32x4(map_to_rank(po_addr + off, s2));
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int s2 = 0; s2 < kMaxClusterSplits; ++s2) {
                if (s2 < n_split) {
                    acc.x += w[s2] * v[s2].x;
                    acc.y += w[s2] * v[s2].y;
                    acc.z += w[s2] * v[s2].z;
                    acc.w += w[s2] * v[s2].w;
                }
            }
            const int rq = row0 + i;
            reinterpret_cast<float4 *>(out + ((b * n_nodes + rq / G) * H_q + g * G + rq % G) * D)[d4] = acc;
        }
        __syncwarp();
        cluster_arrive();
        cluster_wait();
        return;
    }

    const int64_t cidx = (b * H_kv + g) * n_rb + rb;
    if (slice_stride) {
        // ------------------------------------------------- slice merge
        // Every split has written its partial.  Each CTA takes an arrival
        // ticket; all but the last wait (time-bounded) until every split has
        // arrived and then merge their own slice of the rows x D outputs, so
        // the merge runs on all the launch's SMs at once.  The last to arrive
        // never waits: it merges its own slice and then every slice still
        // unclaimed (one whose CTA gave up waiting), so each slice is merged
        // exactly once (claims are compare-and-swap) whatever the
        // co-residency.  The last CTA to leave returns the counters to zero.
        __threadfence();
        __syncthreads();
        int32_t *ctr = ws.counters + cidx * slice_stride;  // arrivals, departures, claims
        if (tid == 0) {
            const bool is_last = atomicAdd(ctr, 1) == n_split - 1;
            const bool all_in = is_last || poll_geq_bounded(ctr, n_split, kSlicePollNs);
            if (all_in) __threadfence();
            flags[1] = is_last;
            flags[2] = all_in && atomicCAS(ctr + 2 + split, 0, 1) == 0;
        }
        __syncthreads();
        const bool is_last = flags[1] != 0;
        const bool mine = flags[2] != 0;
        const int total4 = n_rows * D4;
        const int per4 = (total4 + n_split - 1) / n_split;
        constexpr int kWarps = kThreads / 32;
        float *sw = reinterpret_cast<float *>(smem + C::kKvOff);                  // [rows of the slice][n_split]
        float4 *red = reinterpret_cast<float4 *>(smem + C::kKvOff + 65536);       // [kThreads]
        int32_t *claim = reinterpret_cast<int32_t *>(smem + C::kKvOff + 65536 + kThreads * 16);  // [n_split]
        const int64_t prow0 = (b * H_kv + g) * R + row0;
        // Merges slice s_idx: float4 outputs [lo4, hi4) of this row block;
        // rr_n threads per output, each summing a strided subset of the
        // splits, then a fixed-order reduction.
        auto slice_merge = [&](int s_idx) {
            const int lo4 = s_idx * per4;
            const int hi4 = lo4 + per4 < total4 ? lo4 + per4 : total4;
            if (lo4 >= hi4) return;
            const int nel = hi4 - lo4;
            const int i0 = lo4 / D4;
            const int nh = (hi4 - 1) / D4 - i0 + 1;
            for (int e = tid; e < nh * n_split; e += kThreads) sw[e] = __ldcg(ws.lse_part + (prow0 + i0) * n_split + e);
            __syncthreads();
            for (int hh = warp; hh < nh; hh += kWarps) {
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
                const float lt = sum > 0.f ? M + log2f(sum) : -INFINITY;
                __syncwarp();
                for (int s2 = lane; s2 < n_split; s2 += 32)
                    x[s2] = (sum > 0.f && x[s2] != -INFINITY) ? exp2f(x[s2] - lt) : 0.f;
                const int rq = row0 + i0 + hh;
                if (lane == 0 && lse && (i0 + hh) * D4 >= lo4)
                    lse[(b * n_nodes + rq / G) * H_q + g * G + rq % G] = lt * kLn2;
            }
            __syncthreads();
            const int per_round = nel < kThreads ? nel : kThreads;
            const int rr_n = kThreads / per_round;  // >= 1
            for (int base = 0; base < nel; base += per_round) {
                const int sub = tid / per_round, el = base + (tid - sub * per_round);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (sub < rr_n && el < nel) {
                    const int f = lo4 + el;
                    const int i = f / D4, d4 = f - i * D4;
                    const float *wh = sw + (i - i0) * n_split;
                    const float4 *op = reinterpret_cast<const float4 *>(ws.o_part + (prow0 + i) * n_split * D) + d4;
                    constexpr int kBatch = 8;
                    for (int s0 = sub; s0 < n_split; s0 += kBatch * rr_n) {
                        float4 v[kBatch];
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int s2 = s0 + u * rr_n;
                            if (s2 < n_split) v[u] = __ldcg(op + (int64_t)s2 * D4);
                        }
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int s2 = s0 + u * rr_n;
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
                __syncthreads();
                if (tid < per_round && base + tid < nel) {
                    float4 t = red[tid];
                    for (int k2 = 1; k2 < rr_n; ++k2) {
                        const float4 u = red[k2 * per_round + tid];
                        t.x += u.x;
                        t.y += u.y;
                        t.z += u.z;
                        t.w += u.w;
                    }
                    const int f = lo4 + base + tid;
                    const int i = f / D4, d4 = f - i * D4;
                    const int rq = row0 + i;
                    reinterpret_cast<float4 *>(out + ((b * n_nodes + rq / G) * H_q + g * G + rq % G) * D)[d4] = t;
                }
                __syncthreads();  // red is reused by the next round
            }
        };
        if (mine) slice_merge(split);
        if (is_last) {
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
            if (__syncthreads_count(any) > 0)
                for (int s2 = 0; s2 < n_split; ++s2)
                    if (claim[s2]) slice_merge(s2);
        }
        __syncthreads();
        if (tid == 0 && atomicAdd(ctr + 1, 1) == n_split - 1)
            for (int i = 0; i < 2 + n_split; ++i) ctr[i] = 0;  // ready for the next call
        return;
    }

    // ------------------------------------------ ticket; the last CTA merges
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const int32_t ticket = atomicAdd(&ws.counters[cidx], 1);
        flags[1] = (ticket == n_split - 1);
    }
    __syncthreads();
    if (!flags[1]) return;
    __threadfence();
    float *wts = reinterpret_cast<float *>(smem + C::kKvOff);  // [rows][n_split]
    const int64_t prow0 = (b * H_kv + g) * R + row0;
    for (int e = tid; e < n_rows * n_split; e += kThreads) wts[e] = __ldcg(ws.lse_part + prow0 * n_split + e);
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
        if (lse) lse[(b * n_nodes + rq / G) * H_q + g * G + rq % G] = lt * kLn2;
    }
    __syncthreads();
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
        reinterpret_cast<float4 *>(out + ((b * n_nodes + rq / G) * H_q + g * G + rq % G) * D)[d4] = acc;
    }
    if (tid == 0) ws.counters[cidx] = 0;
}

// Whether clusters of n CTAs of the tree kernel can be resident on device
// dev (cached per device and size).
// cuTensorMapEncodeTiled from the driver, looked up once.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
                cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    }
    return fn;
}

}  // namespace
}  // namespace wmtp

namespace wmtp {

// 3-D map of a [num_slots][H_kv][D] bf16 pool: boxes of 64 dims x 1 head x
// `rows` consecutive slots, 128-byte swizzle.
bool pool_tensor_map(CUtensorMap *map, const void *pool, int64_t num_slots, int H_kv, int D, int rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn || num_slots < 1) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H_kv, (cuuint64_t)num_slots};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H_kv * D * 2};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(pool), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace wmtp

namespace wmtp {
namespace {

// Merge counters per (request, KV head, row block) for the slice merge:
// arrivals, departures and one claim per split, rounded to 16 (the same
// stride as the decode attention's workspace, whose counters the draft-extend
// pass shares).
inline int tree_counter_stride(int n_split) {
    const int n = 2 + n_split;
    return n < 16 ? 16 : (n + 15) / 16 * 16;
}

// CTAs of the tree kernel the device holds at once (0 if unknown).
template <int D>
int tree_resident_capacity(int dev) {
    static int32_t known[64] = {};
    if (dev < 0 || dev >= 64) return 0;
    if (known[dev]) return known[dev] > 0 ? known[dev] : 0;
    int sms = 0, per_sm = 0;
    const bool ok = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tree_tc_kernel<D, true>, kThreads,
                                                                  Cfg<D>::kSmemBytes) == cudaSuccess &&
                    sms > 0 && per_sm > 0;
    cudaGetLastError();
    known[dev] = ok ? sms * per_sm : -1;
    return ok ? known[dev] : 0;
}

template <int D>
bool tree_cluster_ok(int dev, int n) {
    static int8_t known[64][kMaxClusterSplits + 1] = {};
    if (n < 2 || n > kMaxClusterSplits || dev < 0 || dev >= 64) return false;
    if (known[dev][n]) return known[dev][n] > 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)n;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&clusters, tree_tc_kernel<D, true>, &cfg) == cudaSuccess &&
                    clusters > 0;
    cudaGetLastError();  // a refused query is not an error of this call
    known[dev][n] = ok ? 1 : -1;
    return ok;
}

template <int D>
wmtp_status launch_tree_tc(const uint16_t *q, int32_t B, int32_t H_q, int32_t H_kv,
                           const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                           const int32_t *seq_lens, const int32_t *ring_base, int32_t n_sink,
                           int32_t window, int32_t depth, int32_t tree_k, float scale, float *out,
                           float *lse, void *workspace, int32_t n_split, cudaStream_t stream,
                           TreeTable tt, TreeWs ws_given) {
    using C = Cfg<D>;
    const int G = H_q / H_kv;
    const int n_nodes = tree_k * depth;
    const int R = n_nodes * G;
    const int n_rb = (R + kRows - 1) / kRows;
    static int opted_in[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return WMTP_ECUDA;
    if (!opted_in[dev]) {
        if (cudaFuncSetAttribute(tree_tc_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(tree_tc_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes) != cudaSuccess)
            return WMTP_ECUDA;
        opted_in[dev] = 1;
    }
    const bool use_cluster = n_split > 1 && tree_cluster_ok<D>(dev, n_split);
    // without a cluster: the slice merge when the whole grid is resident at
    // once (its waits then end as soon as the last split arrives), else the
    // last CTA merges
    int32_t slice = 0;
    if (n_split > 1 && !use_cluster) {
        const int cap = tree_resident_capacity<D>(dev);
        if (cap > 0 && (int64_t)n_split * H_kv * n_rb * B <= cap) slice = tree_counter_stride(n_split);
    }
    TreeWs ws{nullptr, nullptr, nullptr};
    if (n_split > 1 && !use_cluster && ws_given.counters) {
        ws = ws_given;
    } else if (n_split > 1 && !use_cluster) {
        uint8_t *p = static_cast<uint8_t *>(workspace);
        ws.counters = reinterpret_cast<int32_t *>(p);
        p += align256((size_t)B * H_kv * n_rb * tree_counter_stride(n_split) * 4);
        ws.lse_part = reinterpret_cast<float *>(p);
        p += align256((size_t)B * H_kv * R * n_split * 4);
        ws.o_part = reinterpret_cast<float *>(p);
    }
    CUtensorMap tm_k32, tm_v32, tm_k8, tm_v8;
    if (!pool_tensor_map(&tm_k32, k_pool, num_slots, H_kv, D, kCopyKeys) ||
        !pool_tensor_map(&tm_v32, v_pool, num_slots, H_kv, D, kCopyKeys) ||
        !pool_tensor_map(&tm_k8, k_pool, num_slots, H_kv, D, 8) ||
        !pool_tensor_map(&tm_v8, v_pool, num_slots, H_kv, D, 8))
        return WMTP_ECUDA;
    PdlLaunch launch(dim3((unsigned)n_split, (unsigned)(H_kv * n_rb), (unsigned)B), dim3(kThreads),
                     C::kSmemBytes, stream);
    if (use_cluster) launch.add_cluster((unsigned)n_split);
    // ring mode with long chunks: the instance with split K / V gather roles
    const int64_t ring_keys = (int64_t)n_sink + window + (int64_t)depth * tree_k;
    const int64_t chunk_tiles = (ring_keys + (int64_t)n_split * kKeys - 1) / ((int64_t)n_split * kKeys);
    auto kernel = !tt.table && chunk_tiles >= kSplitMinTiles ? tree_tc_kernel<D, true> : tree_tc_kernel<D, false>;
    const cudaError_t err = cudaLaunchKernelEx(
        &launch.cfg, kernel, reinterpret_cast<const __nv_bfloat16 *>(q), H_q, H_kv, G,
        n_nodes, reinterpret_cast<const __nv_bfloat16 *>(k_pool),
        reinterpret_cast<const __nv_bfloat16 *>(v_pool), num_slots, seq_lens, ring_base, n_sink,
        window, depth, tree_k, scale * 1.4426950408889634f, out, lse, ws, tt, n_split, n_rb,
        (int32_t)(use_cluster ? 1 : 0), slice, tm_k32, tm_v32, tm_k8, tm_v8);
    return err == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

}  // namespace

cudaError_t read_tree_tc_error(int32_t *code, bool clear) {
    cudaError_t err = cudaMemcpyFromSymbol(code, g_tree_tc_error, sizeof(int32_t));
    if (err != cudaSuccess || !clear) return err;
    const int32_t zero = 0;
    return cudaMemcpyToSymbol(g_tree_tc_error, &zero, sizeof(int32_t));
}

size_t tree_tc_workspace_bytes(int64_t B, int64_t H_kv, int64_t R, int D, int n_split) {
    if (n_split <= 1) return 0;
    const int64_t n_rb = (R + kRows - 1) / kRows;
    return align256((size_t)B * H_kv * n_rb * tree_counter_stride(n_split) * 4) +
           align256((size_t)B * H_kv * R * n_split * 4) +
           (size_t)B * H_kv * R * n_split * D * 4;
}

wmtp_status tree_tc_launch(const uint16_t *q, int32_t B, int32_t H_q, int32_t H_kv, int32_t D,
                           const uint16_t *k_pool, const uint16_t *v_pool, int64_t num_slots,
                           const int32_t *seq_lens, const int32_t *ring_base, int32_t n_sink,
                           int32_t window, int32_t depth, int32_t tree_k, float scale, float *out,
                           float *lse, void *workspace, int32_t n_split, cudaStream_t stream) {
    const TreeTable tt{nullptr, 0, nullptr, nullptr};
    const TreeWs none{nullptr, nullptr, nullptr};
    if (D == 256)
        return launch_tree_tc<256>(q, B, H_q, H_kv, k_pool, v_pool, num_slots, seq_lens, ring_base,
                                   n_sink, window, depth, tree_k, scale, out, lse, workspace,
                                   n_split, stream, tt, none);
    return launch_tree_tc<128>(q, B, H_q, H_kv, k_pool, v_pool, num_slots, seq_lens, ring_base,
                               n_sink, window, depth, tree_k, scale, out, lse, workspace, n_split,
                               stream, tt, none);
}

wmtp_status tree_extend_launch(const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv,
                               int32_t D, const uint16_t *k_pool, const uint16_t *v_pool,
                               int64_t num_slots, const int32_t *table, int64_t table_stride,
                               const int32_t *lens, const int32_t *seq_lens, const int32_t *n_new,
                               int32_t n_sink, int32_t window, int32_t windowed, float scale,
                               float *out, float *lse, int32_t *ws_counters, float *ws_lse_part,
                               float *ws_o_part, int32_t n_split, cudaStream_t stream) {
    // A chain of n_q nodes whose key list is the union table row; without
    // windowing, a window no kv length reaches.
    const int32_t w = windowed ? window : INT32_MAX / 4;
    const TreeTable tt{table, table_stride, lens, n_new};
    const TreeWs ws{ws_counters, ws_lse_part, ws_o_part};
    if (D == 256)
        return launch_tree_tc<256>(q, B, H_q, H_kv, k_pool, v_pool, num_slots, seq_lens, nullptr, n_sink,
                                   w, n_q, 1, scale, out, lse, nullptr, n_split, stream, tt, ws);
    return launch_tree_tc<128>(q, B, H_q, H_kv, k_pool, v_pool, num_slots, seq_lens, nullptr, n_sink, w,
                               n_q, 1, scale, out, lse, nullptr, n_split, stream, tt, ws);
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
    const int64_t n_rb = (R + kRows - 1) / kRows;
    const int64_t per_split = (int64_t)B * H_kv * n_rb;
    const int64_t keys = (int64_t)n_sink + window + (int64_t)tree_k * depth;
    int64_t n = sms / per_split;
    const int64_t by_len = (keys + 31) / 32 / 4;  // >= 128 keys per split
    if (n > by_len) n = by_len;
    if (n < 1) n = 1;
    if (n > kMaxSplits) n = kMaxSplits;
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
    if (n_split < 1 || n_split > kMaxSplits || num_slots < 0) return WMTP_EINVAL;
    if (depth > 255) return WMTP_EINVAL;
    const int64_t R = (int64_t)tree_k * depth * (H_q / H_kv);
    const int64_t n_rb = (R + kRows - 1) / kRows;
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
