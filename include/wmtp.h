/*
 * wmtp.h -- C ABI of the GB300 (sm_103a) library for the Windowed-MTP draft
 * attention hot path.
 *
 * Method: "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
 * Million-Token Context" (arXiv 2607.21535).  The MTP/NEXTN draft head's
 * decode attention reads only [n_sink sink positions] || [the most recent W
 * positions] of the KV cache (§4 "Method", Mechanism), and the draft KV lives
 * in a compact per-request ring of n_sink + W + d*k slots (App. A "The
 * windowing change"; §6 Memory; §7 "Compatibility with tree speculation").
 *
 * Conventions shared by every call:
 *   - All pointers marked "device" point to memory of the current CUDA device;
 *     the caller owns every buffer.  The library allocates nothing and never
 *     synchronises; every call is asynchronous on `stream` (a cudaStream_t,
 *     NULL = the legacy default stream) and may be captured in a CUDA graph.
 *     A captured call keeps its pointers: every buffer it was given, the
 *     workspace included, must stay allocated while the graph may be
 *     replayed (a replay after the memory is freed is an invalid access).
 *   - bf16 values travel as their 16-bit patterns (uint16_t).
 *   - Positions and slots are 0-based.  A request's KV pool has the layout
 *     [num_slots][H_kv][D]: the K (or V) row of KV head g for slot s starts at
 *     element (s * H_kv + g) * D.
 *   - Host-side argument checks run before any launch and return
 *     WMTP_EINVAL / WMTP_ECAPACITY without touching memory.  A failed launch
 *     returns WMTP_ECUDA.  Checks that need device data (a slot outside the
 *     pool, a table longer than its row) are done in the kernels: the access is
 *     skipped, the first such error code is latched in a device word, and
 *     wmtp_get_device_error() returns it.  No kernel traps or spins without a
 *     time limit.
 *   - Draft depth d = gamma + 1 ("Windowed-MTP", §3 Eq. (1): d is the engine's
 *     num_draft_tokens and gamma = d - 1 draft forwards per decode step);
 *     tree_k = 1 is a chain.
 */
#ifndef WMTP_H
#define WMTP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t wmtp_status;

#define WMTP_OK 0
#define WMTP_EINVAL (-1)     /* bad argument (null pointer, bad size, bad config) */
#define WMTP_ECAPACITY (-2)  /* an output or workspace is too small */
#define WMTP_ECUDA (-3)      /* a CUDA launch or runtime call failed */
#define WMTP_EDEVICE (-4)    /* wmtp_get_device_error(): a device-side check failed */

/* Device-side error codes latched by the kernels (first one wins). */
#define WMTP_DEV_OK 0
#define WMTP_DEV_SLOT_RANGE 1    /* a slot index outside [0, num_slots) */
#define WMTP_DEV_TABLE_OVERFLOW 2 /* a table row needs more than `stride` entries */
#define WMTP_DEV_LEN_RANGE 3     /* a lens[] entry is negative, above the row stride, or not the length of its key list */
#define WMTP_DEV_WAIT_TIMEOUT 4  /* a pipeline wait ran out of time; results invalid */
#define WMTP_DEV_ARG_RANGE 5     /* a device-side position, branch or length is out of range */

/* Library version, e.g. 1000 for 0.1.0. */
int32_t wmtp_version(void);

/* Short English text for a wmtp_status or a device error code. */
const char *wmtp_status_string(int32_t status);

/* Reads (and, if `clear` is non-zero, resets) the device error word of the
 * current device.  Synchronises the device.  *code receives a WMTP_DEV_* code.
 * Returns WMTP_OK, or WMTP_ECUDA if the copy failed. */
wmtp_status wmtp_get_device_error(int32_t *code, int32_t clear);

/* ------------------------------------------------------------------------
 * Draft KV-index builder.
 * "Windowed-MTP", App. A "The windowing change (pseudocode)" and §4
 * Mechanism: for draft step j (0 <= j < gamma) of request b the draft sees
 * kv_len = seq_lens[b] + j + 1 positions (its own token appended before it
 * attends).  Windowed mode (windowed != 0) and kv_len > n_sink + W:
 * positions [0, n_sink) then [kv_len - W, kv_len); otherwise (or full mode)
 * positions [0, kv_len).  Each position p becomes a physical slot:
 *   paged layout (req_to_token != NULL): req_to_token[req_pool_idx[b] *
 *     rtt_stride + p] (req_pool_idx == NULL means request b uses row b);
 *   ring layout  (req_to_token == NULL): the ring slot of p on branch 0
 *     (see wmtp_ring_map) for ring_base[b].
 *
 * seq_lens      device int32 [B]: committed length S of each request.
 * table         device int32 [gamma][B][stride], written for i < lens only.
 * lens          device int32 [gamma][B]: entries written per row.
 * depth, tree_k ring geometry (used by the ring layout only).
 * Errors: WMTP_EINVAL for null pointers, B < 0, gamma < 0, n_sink < 0,
 * W < 1, depth < 1, tree_k < 1, stride < 1 or gamma * B > 65535.
 * Row lengths depend on device data, so capacity is checked in the kernel:
 * a row that needs more than `stride` entries writes `stride` entries,
 * stores its true length in lens and latches WMTP_DEV_TABLE_OVERFLOW. */
wmtp_status wmtp_build_draft_indices(const int32_t *seq_lens, int32_t B,
                                     int32_t gamma, int32_t n_sink,
                                     int32_t window, int32_t depth,
                                     int32_t tree_k, int32_t windowed,
                                     const int32_t *req_to_token,
                                     const int32_t *req_pool_idx,
                                     int64_t rtt_stride,
                                     const int32_t *ring_base, int32_t *table,
                                     int64_t stride, int32_t *lens,
                                     void *stream);

/* Far-key table of the same draft steps: for draft step j of request b
 * (kv_len = seq_lens[b] + j + 1), the positions the keep rule drops --
 * [n_sink, kv_len - W) when kv_len > n_sink + W, none otherwise -- in
 * ascending order, mapped to slots through req_to_token as above (paged
 * layout only: a ring no longer holds those positions).  The far table and
 * the windowed table of a step partition its full-context table; attention
 * over each feeds wmtp_attn_mass_diagnostics ("Windowed-MTP", §5 "A
 * partition-function view").  Arguments, capacity check and errors as
 * wmtp_build_draft_indices; req_to_token must not be NULL. */
wmtp_status wmtp_build_far_indices(const int32_t *seq_lens, int32_t B,
                                   int32_t gamma, int32_t n_sink,
                                   int32_t window, const int32_t *req_to_token,
                                   const int32_t *req_pool_idx,
                                   int64_t rtt_stride, int32_t *table,
                                   int64_t stride, int32_t *lens, void *stream);

/* Index table of a draft-extend pass (the draft forward over the n new
 * tokens a request accepted, at positions S..S+n-1, in one launch; see
 * wmtp_draft_extend_attn).  Row b is the union of the key sets of its n
 * tokens under the keep rule above: token t sees kv_len = S + t + 1, so the
 * union is the keep rule at kv_len = S + n with window W + n - 1 --
 * positions [0, n_sink) then [S + 1 - W, S + n) when S + 1 > n_sink + W
 * (windowed mode), else [0, S + n) -- mapped to slots as above.  A request
 * with n = 0 gets an empty row.
 *
 * seq_lens   device int32 [B]: committed length S before the new tokens.
 * n_new      device int32 [B]: new tokens per request (>= 0; a negative
 *            count is treated as 0 and latches WMTP_DEV_ARG_RANGE).
 * table      device int32 [B][stride]; lens device int32 [B].
 * Other arguments and errors as wmtp_build_draft_indices (gamma = 1). */
wmtp_status wmtp_build_extend_indices(const int32_t *seq_lens,
                                      const int32_t *n_new, int32_t B,
                                      int32_t n_sink, int32_t window,
                                      int32_t depth, int32_t tree_k,
                                      int32_t windowed,
                                      const int32_t *req_to_token,
                                      const int32_t *req_pool_idx,
                                      int64_t rtt_stride,
                                      const int32_t *ring_base, int32_t *table,
                                      int64_t stride, int32_t *lens,
                                      void *stream);

/* ------------------------------------------------------------------------
 * Ring slot mapper.
 * "Windowed-MTP", App. A: slot = ring_base(r) + logical position, with a
 * ring of n_sink + W + d slots per request; §7: a tree of width k reserves
 * n_sink + W + d*k and its candidates diverge only over the last d positions.
 * This library pins the sink slots and rolls the rest:
 *   branch == 0 and p < n_sink : ring_base + p
 *   otherwise                  : ring_base + n_sink
 *                                + ((p - n_sink + branch * d) mod (W + d*k))
 * (non-negative modulo).  Below n_sink + W + d*k this equals the pages'
 * literal ring_base + p; above it, live sinks are never overwritten.
 *
 * ring_base device int32 [number of requests]; pos, req_of device int32 [n];
 * branch device int32 [n] or NULL (all 0); slots device int32 [n] (output).
 * Errors: WMTP_EINVAL for null pointers, n < 0, n_sink < 0, W < 1, depth < 1,
 * tree_k < 1. */
wmtp_status wmtp_ring_map(const int32_t *ring_base, const int32_t *pos,
                          const int32_t *branch, const int32_t *req_of,
                          int32_t n, int32_t n_sink, int32_t window,
                          int32_t depth, int32_t tree_k, int32_t *slots,
                          void *stream);

/* ------------------------------------------------------------------------
 * Draft KV append: each draft forward writes its own token's K and V before
 * attending ("Windowed-MTP", §3: the draft re-reads the cache it extends).
 * Copies k_new[i] and v_new[i] (each [H_kv][D] bf16) into pool slot
 * slots[i].  k_new, v_new device bf16 [n][H_kv][D]; slots device int32 [n];
 * k_pool, v_pool device bf16 [num_slots][H_kv][D].
 * A slot outside [0, num_slots) is skipped and latches WMTP_DEV_SLOT_RANGE.
 * Errors: WMTP_EINVAL for null pointers, n < 0, H_kv < 1, D < 1, D % 8 != 0
 * or pointers not 16-byte aligned. */
wmtp_status wmtp_append_kv(const uint16_t *k_new, const uint16_t *v_new,
                           const int32_t *slots, int32_t n, int32_t H_kv,
                           int32_t D, uint16_t *k_pool, uint16_t *v_pool,
                           int64_t num_slots, void *stream);

/* ------------------------------------------------------------------------
 * Split-KV flash-decode draft attention with a log-sum-exp merge.
 * Computes, for every request b, query token t < n_q and query head h
 * (KV head g = h / (H_q / H_kv)), softmax attention over the keys listed in
 * table row b ("Windowed-MTP", §4 Mechanism: the reduced table is the key
 * set, no extra mask):
 *   s_i = scale * <q[b,t,h,:], K[table[b,i], g, :]>,  i < lens[b]
 *   out[b,t,h,:] = sum_i softmax(s)_i V[table[b,i], g, :]
 *   lse[b,t,h]   = log sum_i exp(s_i)        (natural log)
 * Each row is cut into n_split contiguous chunks whose size depends only on
 * lens[b] and n_split, so results depend on the logical key order and not
 * on the physical slots.  Partials (o, lse) are merged in split order:
 * through distributed shared memory of a thread-block cluster when
 * n_split <= 16; in two levels (clusters of up to 16, then at most 8
 * cluster partials per output slice through the workspace) when n_split
 * splits into such clusters; else through the workspace by the last CTA to
 * finish.  A cluster merge is used only when the device holds all of the
 * launch's clusters at once (cudaOccupancyMaxActiveClusters).  An empty row
 * gives out = 0, lse = -inf.
 *
 * q        device bf16 [B][n_q][H_q][D], D in {128, 256}, H_q / H_kv <= 8.
 * table    device int32, row b at table + b * table_stride.
 * lens     device int32 [B]; each must be <= table_stride.
 * out      device fp32 [B][n_q][H_q][D], 16-byte aligned;
 * lse      device fp32 [B][n_q][H_q] or NULL.
 * k_pool, v_pool 16-byte aligned; q 4-byte aligned.
 * workspace device, >= wmtp_attn_workspace_bytes(...) bytes, 256-byte
 *          aligned.  Its first bytes hold max(16, 2 + n_split rounded up
 *          to 16) merge counters per (request, query token, KV head); they
 *          must be zero when a call starts.
 *          wmtp_attn_workspace_init() zeroes them, and every completed call
 *          leaves its own counters at zero, so a workspace serves any number
 *          of calls with the same B * n_q * H_kv.  Initialise again before
 *          using it for a larger B * n_q * H_kv.  Calls that share a
 *          workspace must not overlap on the GPU.  Unused when n_split == 1,
 *          and when the splits merge through one thread-block cluster (up to
 *          16 splits, where the device can hold such a cluster).
 * Merge paths (fixed by n_split, B * n_q * H_kv and the device, so results
 * depend only on those and the inputs), in order of preference: one cluster
 * (n_split <= 16, through distributed shared memory); whole clusters of up
 * to 16 merged in two levels, when the device holds all of them at once;
 * the slice merge, when no cluster plan fits, the whole grid fits on the
 * device at once and no split's slice holds more than 128 float4 outputs
 * (ceil(G * D / 4 / n_split) <= 128) (every split writes its partial, takes an arrival ticket
 * and, once all have arrived -- a wait bounded at 50 us -- merges its own
 * slice of the output; the last to arrive also merges any slice whose split
 * gave up waiting, so the result never depends on co-residency); or the
 * last split to finish merging all of them.
 * n_split  1 .. 1024; wmtp_attn_num_splits() gives a good value.
 * Errors: WMTP_EINVAL for null pointers, bad sizes, D not 128/256,
 * H_q % H_kv != 0, group > 8, misaligned pool/q pointers;
 * WMTP_ECAPACITY if workspace_bytes is too small. */
size_t wmtp_attn_workspace_bytes(int32_t B, int32_t n_q, int32_t H_q,
                                 int32_t H_kv, int32_t D, int32_t n_split);

/* Zeroes the workspace's merge counters (an async memset on `stream`). */
wmtp_status wmtp_attn_workspace_init(void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Split count for rows of up to max_len keys on the current device.  Long
 * rows (at least four 64-key tiles per SM-sized split): one CTA per SM.
 * Short rows: two tiles per split at least, in whole clusters of 16 that
 * the device holds at once when above 16. */
int32_t wmtp_attn_num_splits(int32_t B, int32_t n_q, int32_t H_kv,
                             int64_t max_len);

wmtp_status wmtp_draft_decode_attn(const uint16_t *q, int32_t B, int32_t n_q,
                                   int32_t H_q, int32_t H_kv, int32_t D,
                                   const uint16_t *k_pool,
                                   const uint16_t *v_pool, int64_t num_slots,
                                   const int32_t *table, int64_t table_stride,
                                   const int32_t *lens, float scale,
                                   float *out, float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t n_split,
                                   void *stream);

/* wmtp_append_kv followed by wmtp_draft_decode_attn, in one launch.  A
 * draft forward stores its own K/V in the draft KV pool (§4 Mechanism: the
 * compact ring of n_sink + W + d slots) and attends over the kept
 * positions, its own included; this is the usual decode order, which the
 * pages take for granted.  Results (out, lse and the pool contents) are
 * bit-identical to the two calls in sequence.
 *
 * k_new, v_new device bf16 [B][n_new][H_kv][D], 16-byte aligned: the rows
 *              appended for request b.
 * new_slots    device int32 [B][n_new]: their pool slots.  A slot appended
 *              for request b must not appear in another request's table
 *              row in the same call, and the n_new slots of one request
 *              must differ.
 * n_new        1 .. 4.
 * Other arguments as wmtp_draft_decode_attn; k_pool, v_pool are written.
 * Keys whose slot is one of request b's new slots are read from k_new /
 * v_new; a new slot outside the pool is not written, latches
 * WMTP_DEV_SLOT_RANGE, and its key is masked, as in the two calls. */
wmtp_status wmtp_draft_decode_attn_append(const uint16_t *k_new,
                                          const uint16_t *v_new,
                                          const int32_t *new_slots, int32_t n_new,
                                          const uint16_t *q, int32_t B, int32_t n_q,
                                          int32_t H_q, int32_t H_kv, int32_t D,
                                          uint16_t *k_pool, uint16_t *v_pool,
                                          int64_t num_slots, const int32_t *table,
                                          int64_t table_stride, const int32_t *lens,
                                          float scale, float *out, float *lse,
                                          void *workspace, size_t workspace_bytes,
                                          int32_t n_split, void *stream);

/* A chained draft step: wmtp_draft_decode_attn_append whose launch starts
 * copying keys while the preceding kernel on the stream is still running.
 * The draft forwards of one decode step run back to back (§3 Eq. (1): gamma
 * forwards, each re-reading the draft KV), and step j + 1 reads the same
 * kept keys as step j except the newest one or two, so their copies need
 * not wait for step j to finish.
 *
 * Ordering (programmatic dependent launch): a launch may begin once the
 * preceding kernel on the stream has released its dependents.  This call
 * releases them only after it has waited for its own predecessor, so the
 * launch that follows it overlaps this launch alone; the other calls of
 * this library release them as soon as they start.
 * hold = -1: nothing is read before the preceding kernel has completed (a
 *            safe first step of a chain, e.g. after the index builder).
 * hold >= 0: lens, table, new_slots and the K/V rows of the entries below
 *            lens[b] - hold of every row b are read before the preceding
 *            kernel has completed; q, k_new / v_new, the rows of the last
 *            `hold` entries and of any key whose slot is a new slot are
 *            read, and every output written, only after it.  The caller
 *            guarantees that no kernel that may still be running when the
 *            launch begins writes what is read early: the preceding kernel
 *            and, if it is not a chained launch of this library, the ones
 *            it may overlap.  For fused steps j >= 1 of one decode step on
 *            the same table, each issued by this call (step 0 with
 *            hold = -1), the preceding kernel is step j - 1, which writes
 *            the row of position S + j - 1 (entry lens[b] - 2): hold = 2.
 * Results are bit-identical to wmtp_draft_decode_attn_append with the same
 * arguments: only the moment of the copies changes.  Other arguments and
 * errors as wmtp_draft_decode_attn_append; WMTP_EINVAL for hold < -1. */
wmtp_status wmtp_draft_decode_attn_append_overlap(
    const uint16_t *k_new, const uint16_t *v_new, const int32_t *new_slots,
    int32_t n_new, const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q,
    int32_t H_kv, int32_t D, uint16_t *k_pool, uint16_t *v_pool,
    int64_t num_slots, const int32_t *table, int64_t table_stride,
    const int32_t *lens, float scale, float *out, float *lse, void *workspace,
    size_t workspace_bytes, int32_t n_split, int32_t hold, void *stream);

/* Draft-extend attention: the draft forward over the n = n_new[b] tokens a
 * request accepted (positions S..S+n-1, K/V already appended), in one
 * launch.  Row t < n of request b is the attention of its query heads over
 * exactly the keys draft step t sees under the keep rule (kv_len = S + t + 1,
 * §4 Mechanism / App. A): the union table of wmtp_build_extend_indices
 * restricted to positions below S + t + 1 and, when windowed and S + t + 1 >
 * n_sink + W, to sinks and positions from S + t + 1 - W.  Rows t >= n give
 * out = 0, lse = -inf.  Keys outside a row's set are not read.
 *
 * q          device bf16 [B][n_q][H_q][D]; n_q >= max n_new.
 * table,lens the union table and lengths of wmtp_build_extend_indices built
 *            with the same seq_lens, n_new, n_sink, W and windowed flag.
 * seq_lens   device int32 [B] (S); n_new device int32 [B].
 * Other arguments, the split plan, workspace and errors as
 * wmtp_draft_decode_attn; additionally WMTP_EINVAL for null seq_lens or
 * n_new, n_sink < 0 or W < 1.
 * With 2 <= n_q <= 8, n_split <= 128, table_stride >= 65536 and q 16-byte
 * aligned, the pass runs on the 5th-generation tensor cores: a request's
 * tokens x query heads of a KV head are one 128-row MMA block over each
 * union key once (the tree kernel's chain case, slots from the table), the
 * splits merging through a cluster (n_split <= 8) or the workspace.  With
 * 2 <= n_q <= 8, n_split <= 128 and table_stride >= 1024 * n_split one
 * launch also reads each union key once for all of a request's tokens (a
 * CTA per split of the union row and KV head, one warp per token) and
 * merges the splits through the workspace; otherwise every (request, token)
 * row is its own set of CTAs, as wmtp_draft_decode_attn.  The union table
 * must hold exactly the keep set of S + n, as wmtp_build_extend_indices
 * writes it: on the tensor-core path a row whose length differs latches
 * WMTP_DEV_LEN_RANGE and reads no entry past table_stride.
 * wmtp_extend_num_splits gives the usual split count of every launch. */
wmtp_status wmtp_draft_extend_attn(const uint16_t *q, int32_t B, int32_t n_q,
                                   int32_t H_q, int32_t H_kv, int32_t D,
                                   const uint16_t *k_pool,
                                   const uint16_t *v_pool, int64_t num_slots,
                                   const int32_t *table, int64_t table_stride,
                                   const int32_t *lens, const int32_t *seq_lens,
                                   const int32_t *n_new, int32_t n_sink,
                                   int32_t window, int32_t windowed, float scale,
                                   float *out, float *lse, void *workspace,
                                   size_t workspace_bytes, int32_t n_split,
                                   void *stream);

/* Split count for wmtp_draft_extend_attn when the caller has no preference:
 * n = min(wmtp_attn_num_splits(B, 1, H_kv, max_len), 128) when
 * 2 <= n_q <= 8 and max_len >= 1024 * n (the one-read launch), else
 * wmtp_attn_num_splits(B, n_q, H_kv, max_len). */
int32_t wmtp_extend_num_splits(int32_t B, int32_t n_q, int32_t H_kv,
                               int64_t max_len);

/* Attention-mass diagnostics of the windowed draft ("Windowed-MTP", §5 "A
 * partition-function view"; App. C, Table 12), per query row.  The full key
 * set of a draft step is the disjoint union of the kept set (sinks + window)
 * and the far keys the keep rule drops, so Z = Z_w + Z_far.  Inputs are the
 * attention of the same query over each part: (o_win, lse_win) over the
 * sink + window table and (o_far, lse_far) over the far table of
 * wmtp_build_far_indices, both as wmtp_draft_decode_attn writes them
 * (normalised outputs, natural-log lse; an empty part has lse = -inf).
 * With a = Z_w / Z = 1 / (1 + exp(lse_far - lse_win)) and b = Z_far / Z
 * (from the same exponential, not 1 - a):
 *   in_win[r]        = a: softmax mass inside the kept set;
 *   o_full           = a o_win + b o_far (the full-context read-out);
 *   win_perturb[r]   = ||o_full - o_win|| / ||o_full|| = b ||o_far - o_win|| / ||o_full||;
 *   tail_out_frac[r] = ||sum over far keys of p_k v_k|| / ||o_full|| = b ||o_far|| / ||o_full||.
 * No quantity is formed by subtracting two nearly equal outputs, so a small
 * far share keeps its relative accuracy.  No far key gives in_win = 1 and
 * zero ratios; no key at all gives zeros; ||o_full|| = 0 gives 0 ratios.
 * Optionally the merged full-context attention is written: o_full[r][:] and
 * lse_full[r] = log(e^lse_win + e^lse_far).
 *
 * o_win, o_far    device fp32 [rows][D]; lse_win, lse_far device fp32 [rows].
 * in_win, win_perturb, tail_out_frac  device fp32 [rows]; o_full device fp32
 *                 [rows][D]; lse_full device fp32 [rows]; any output may be
 *                 NULL, not all five.
 * Errors: WMTP_EINVAL for rows < 0, D < 1, null inputs or no output. */
wmtp_status wmtp_attn_mass_diagnostics(const float *o_win, const float *lse_win,
                                       const float *o_far, const float *lse_far,
                                       int64_t rows, int32_t D, float *in_win,
                                       float *win_perturb, float *tail_out_frac,
                                       float *o_full, float *lse_full,
                                       void *stream);

/* ------------------------------------------------------------------------
 * Tree-draft attention over the ring.
 * "Windowed-MTP" §7 "Compatibility with tree speculation": windowing changes
 * only which KV the draft reads, not the tree; a tree of width k reserves
 * n_sink + W + d*k ring slots per request and its candidates share the
 * sink + window prefix, diverging over the last d positions.  This library's
 * reading (the pages leave the tree open): node (branch b, depth i), b < k,
 * i < d, of a request with committed length S sits at logical position S + i
 * and attends the positions App. A's keep rule gives for kv length S + i + 1,
 * where positions below S are committed tokens (ring branch 0) and positions
 * S..S+i are the nodes of its own branch (ring branch b, see wmtp_ring_map).
 * For k = 1 this is exactly the chain of wmtp_build_draft_indices +
 * wmtp_draft_decode_attn.  Slots are computed in the kernel from ring_base:
 * no table is read.
 *
 * q         device bf16 [B][k*d][H_q][D], node t = b*d + i; 16-byte aligned.
 * seq_lens  device int32 [B] (committed length S); ring_base device int32 [B].
 * out       device fp32 [B][k*d][H_q][D], 16-byte aligned; lse fp32 [B][k*d][H_q]
 *           or NULL.
 * workspace >= wmtp_tree_workspace_bytes(...), 256-byte aligned; its merge
 *           counters must be zero at the first call (wmtp_attn_workspace_init
 *           zeroes a whole workspace) and every completed call leaves them
 *           zero.  Unused when n_split == 1, and when the key chunks merge
 *           through a thread-block cluster (n_split <= 8, where the device
 *           holds such clusters).  Otherwise, when the whole grid fits on
 *           the device at once, every chunk merges its own slice of the
 *           output after all have arrived (a wait bounded at 50 us; the last
 *           to arrive merges any slice left over), else the last chunk to
 *           finish merges them all.
 * n_split   1 .. 128 key chunks per request; wmtp_tree_num_splits() gives one.
 * Errors: WMTP_EINVAL for null or misaligned pointers, bad sizes, D not
 * 128/256, H_q % H_kv != 0, W < 1, d < 1, k < 1; WMTP_ECAPACITY for a small
 * workspace; slots outside the pool latch WMTP_DEV_SLOT_RANGE. */
size_t wmtp_tree_workspace_bytes(int32_t B, int32_t H_q, int32_t H_kv,
                                 int32_t D, int32_t depth, int32_t tree_k,
                                 int32_t n_split);
int32_t wmtp_tree_num_splits(int32_t B, int32_t H_q, int32_t H_kv,
                             int32_t depth, int32_t tree_k, int32_t n_sink,
                             int32_t window);
wmtp_status wmtp_tree_draft_attn(const uint16_t *q, int32_t B, int32_t H_q,
                                 int32_t H_kv, int32_t D,
                                 const uint16_t *k_pool,
                                 const uint16_t *v_pool, int64_t num_slots,
                                 const int32_t *seq_lens,
                                 const int32_t *ring_base, int32_t n_sink,
                                 int32_t window, int32_t depth, int32_t tree_k,
                                 float scale, float *out, float *lse,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t n_split, void *stream);

/* ------------------------------------------------------------------------
 * Draft attention without a caller-provided workspace.
 * The paper has no counterpart to this call; it exists for callers that
 * cannot hand the library a workspace: an engine that has reserved nearly
 * all device memory for its KV pool and its own allocator (a cudaMalloc
 * there fails, or stalls the device while it runs), or a plugin boundary
 * that passes only input and output pointers.
 *
 * Same computation, arguments and checks as wmtp_draft_decode_attn minus
 * the workspace.  With n_split > 1 the partials always merge through the
 * "last CTA merges" path, in a scratch array that the library holds in
 * device memory: WMTP_NOALLOC_SCRATCH_BYTES per device that loads the
 * library, kept until the process exits.  The call allocates nothing.
 *   - A call needing more scratch than that -- B * n_q * H_kv merge
 *     counters above WMTP_NOALLOC_MAX_COUNTERS, or partials of
 *     B * n_q * H_q * n_split * (D + 1) floats beyond the rest of the
 *     array -- returns WMTP_ECAPACITY before launching anything.
 *   - The first call on a device (with that device current) looks up the
 *     array's device address; make that first call before any stream
 *     capture.  A failed lookup returns WMTP_ECUDA.  The address is cached
 *     per device in an atomic slot, so host threads whose first calls
 *     overlap are safe (each looks it up and stores the same value).  A
 *     cudaDeviceReset of the device makes the cached address stale: do not
 *     call this entry point on that device again in the same process.
 *   - Results: the merge path is always the workspace ("last CTA merges")
 *     merge, so they are bit-identical to wmtp_draft_decode_attn with the
 *     same n_split whenever that call takes the same merge (no thread-block
 *     cluster fits the split plan and, above 16 splits, the grid is larger
 *     than the device holds at once); where it merges through a cluster or
 *     the slice merge instead, the two agree within rounding.
 *   - Every call shares the one array and it keeps the last call's
 *     contents; each call first zeroes the merge counters it uses (an
 *     async memset on `stream`).  Calls that overlap on the GPU (other
 *     streams, other threads) race on the array: serialise them. */
#define WMTP_NOALLOC_SCRATCH_BYTES (8u << 20)
#define WMTP_NOALLOC_MAX_COUNTERS 4096
wmtp_status wmtp_draft_decode_attn_noalloc(
    const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv,
    int32_t D, const uint16_t *k_pool, const uint16_t *v_pool,
    int64_t num_slots, const int32_t *table, int64_t table_stride,
    const int32_t *lens, float scale, float *out, float *lse, int32_t n_split,
    void *stream);

/* ------------------------------------------------------------------------
 * Ring path without tables.
 *
 * Pruned draft prefill ("Windowed-MTP", §7 "Prefill sparsification and
 * TTFT"): after a prompt of S positions the windowed draft reads only its KV
 * of keep(S) = [0, n_sink) u [S - W, S) (all S positions when
 * S <= n_sink + W), so the draft's prompt pass and KV build are needed for
 * those positions only.
 *
 * wmtp_prefill_keep_positions: positions[b][i], i < counts[b] =
 * min(S_b, n_sink + W), in keep order (sinks, then the window).
 *   seq_lens device int32 [B] (prompt lengths); positions device int32
 *   [B][stride]; counts device int32 [B].  A list longer than stride is cut
 *   at stride and latches WMTP_DEV_TABLE_OVERFLOW; a negative length latches
 *   WMTP_DEV_LEN_RANGE and gives an empty list. */
wmtp_status wmtp_prefill_keep_positions(const int32_t *seq_lens, int32_t B,
                                        int32_t n_sink, int32_t window,
                                        int32_t *positions, int64_t stride,
                                        int32_t *counts, void *stream);

/* wmtp_ring_fill: writes row i of request b -- its draft K and V at kept
 * position p_i of keep(S_b), in the order of wmtp_prefill_keep_positions --
 * to ring slot ring_slot(ring_base[b], p_i) (the ring rule of
 * wmtp_ring_map, branch 0), for i < min(S_b, n_sink + W, stride).
 *   k_rows, v_rows device bf16 [B][stride][H_kv][D], 16-byte aligned;
 *   seq_lens, ring_base device int32 [B]; k_pool, v_pool as
 *   wmtp_append_kv.  A slot outside the pool is skipped and latches
 *   WMTP_DEV_SLOT_RANGE. */
wmtp_status wmtp_ring_fill(const uint16_t *k_rows, const uint16_t *v_rows,
                           const int32_t *seq_lens, int32_t B, int64_t stride,
                           int32_t H_kv, int32_t D, const int32_t *ring_base,
                           int32_t n_sink, int32_t window, int32_t depth,
                           int32_t tree_k, uint16_t *k_pool, uint16_t *v_pool,
                           int64_t num_slots, void *stream);

/* Implicit-table ring decode step: wmtp_build_draft_indices (ring layout,
 * windowed) + wmtp_draft_decode_attn_append for draft step `step`, in one
 * launch and with no table in memory.  Request b (committed length
 * S = seq_lens[b]) attends keep(S + step + 1); entry e of that list is
 * mapped to its ring slot in the kernel, in the same logical order as the
 * table, so results are bit-identical to the table path with the same
 * n_split.  When k_new / v_new (device bf16 [B][H_kv][D]) are given, the
 * step's own row is written to the slot of position S + step first (as
 * wmtp_draft_decode_attn_append with n_new = 1); both NULL: no append.
 * n_q = 1; other arguments as wmtp_draft_decode_attn; the workspace is
 * sized by wmtp_attn_workspace_bytes(B, 1, H_q, H_kv, D, n_split) and
 * wmtp_attn_num_splits(B, 1, H_kv, n_sink + W) is the usual split count.
 * Errors: WMTP_EINVAL for n_sink < 0, W < 1, depth < 1, tree_k < 1,
 * step < 0, or only one of k_new / v_new. */
wmtp_status wmtp_draft_decode_attn_ring(
    const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q, int32_t B,
    int32_t H_q, int32_t H_kv, int32_t D, uint16_t *k_pool, uint16_t *v_pool,
    int64_t num_slots, const int32_t *seq_lens, const int32_t *ring_base,
    int32_t step, int32_t n_sink, int32_t window, int32_t depth,
    int32_t tree_k, float scale, float *out, float *lse, void *workspace,
    size_t workspace_bytes, int32_t n_split, void *stream);

/* wmtp_draft_decode_attn_ring as a chained step, with the ordering and
 * the hold rule of wmtp_draft_decode_attn_append_overlap: with hold >= 0,
 * seq_lens, ring_base and the ring rows of the kept entries below the row
 * length minus hold are read before the preceding kernel has completed, q,
 * k_new / v_new and the last `hold` entries after it (hold = 2 for steps
 * >= 1 of a chain of fused ring steps, -1 for its first step).  k_new /
 * v_new are required.  Bit-identical to wmtp_draft_decode_attn_ring;
 * WMTP_EINVAL for hold < -1 or no k_new / v_new. */
wmtp_status wmtp_draft_decode_attn_ring_overlap(
    const uint16_t *k_new, const uint16_t *v_new, const uint16_t *q, int32_t B,
    int32_t H_q, int32_t H_kv, int32_t D, uint16_t *k_pool, uint16_t *v_pool,
    int64_t num_slots, const int32_t *seq_lens, const int32_t *ring_base,
    int32_t step, int32_t n_sink, int32_t window, int32_t depth,
    int32_t tree_k, float scale, float *out, float *lse, void *workspace,
    size_t workspace_bytes, int32_t n_split, int32_t hold, void *stream);

/* ------------------------------------------------------------------------
 * fp8 KV ("Windowed-MTP", §6 "Robustness to KV-cache quantization": the
 * window bounds the number of KV entries read, so its saving composes with a
 * lower-precision cache, whose bytes per entry it does not change; the
 * pages' own fp8-KV path has no fused attention kernel).  The pools hold
 * OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 fraction bits;
 * largest finite 448; no infinities) in the layout [num_slots][H_kv][D],
 * one byte per element, and each KV head g has one fp32 scale for K and one
 * for V: element = code * scale[g].  Codes 0x7F / 0xFF (NaN) are never
 * written by wmtp_append_kv_fp8; the attention reads them as NaN. */

/* Quantising append: for token i < n, KV head g and element e,
 *   k_pool[slots[i]][g][e] = E4M3_rn_satfinite(k_new[i][g][e] * (1 / k_scale[g]))
 * (likewise v), the reciprocal and the product each rounded once in fp32,
 * round to nearest even, finite values beyond +-448 saturating.
 *
 * k_new, v_new device bf16 [n][H_kv][D], 16-byte aligned; D % 16 == 0.
 * k_scale, v_scale device fp32 [H_kv], positive and finite.
 * k_pool, v_pool   device uint8 [num_slots][H_kv][D], 16-byte aligned.
 * A slot outside [0, num_slots) is not written and latches
 * WMTP_DEV_SLOT_RANGE. */
wmtp_status wmtp_append_kv_fp8(const uint16_t *k_new, const uint16_t *v_new,
                               const int32_t *slots, int32_t n, int32_t H_kv,
                               int32_t D, const float *k_scale,
                               const float *v_scale, uint8_t *k_pool,
                               uint8_t *v_pool, int64_t num_slots,
                               void *stream);

/* wmtp_draft_decode_attn over E4M3 pools:
 *   s_i = scale * <q[b,t,h,:], k_scale[g] * Kcode[table[b,i], g, :]>
 *   out = sum_i softmax(s)_i * v_scale[g] * Vcode[table[b,i], g, :]
 * Same arguments, workspace, split plan, merges and checks as
 * wmtp_draft_decode_attn (wmtp_attn_workspace_bytes sizes the workspace),
 * with uint8 pools and the per-KV-head scales k_scale, v_scale (device fp32
 * [H_kv]).  The codes are widened exactly to fp16 on chip and q is rounded
 * to fp16 (exact for |q| >= 2^-14), products accumulate in fp32. */
/* Split count wmtp_draft_decode_attn_fp8 uses when the caller has no
 * preference: as wmtp_attn_num_splits, with the cluster capacity of the fp8
 * instance (one CTA per SM, a deeper copy pipeline). */
int32_t wmtp_attn_num_splits_fp8(int32_t B, int32_t n_q, int32_t H_kv,
                                 int64_t max_len);

wmtp_status wmtp_draft_decode_attn_fp8(
    const uint16_t *q, int32_t B, int32_t n_q, int32_t H_q, int32_t H_kv,
    int32_t D, const uint8_t *k_pool, const uint8_t *v_pool,
    const float *k_scale, const float *v_scale, int64_t num_slots,
    const int32_t *table, int64_t table_stride, const int32_t *lens,
    float scale, float *out, float *lse, void *workspace,
    size_t workspace_bytes, int32_t n_split, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* WMTP_H */
