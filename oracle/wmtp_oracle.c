/*
 * wmtp_oracle.c -- plain, slow CPU oracle for the Windowed-MTP draft-attention
 * hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's shared library; the product
 * path (the CUDA library under speculative_decoding_draft_build_gb300/) never
 * does, and shares no code, header or constant with it.
 *
 * Everything is computed in plain loops, in fp64 for floating point, in the
 * order the sources state it.  No blocking, no splitting, no fusion.
 *
 * Sources (web pages, cited by title and section):
 *   [WMTP]  "Windowed-MTP: Removing the Full-Context Draft-KV Tax at
 *           Million-Token Context" (arXiv 2607.21535).
 *           - §4 "Method: Windowed-MTP", Mechanism: the draft's per-request
 *             block table is reduced to [sink blocks] || [recent W blocks]
 *             with the matching sequence length; no extra mask; RoPE is baked
 *             into the cached keys.
 *           - App. A "The windowing change (pseudocode)": the keep rule and the
 *             ring slot rule "slot = ring_base(r) + logical_pos, modulus
 *             n_sink + W + d".
 *           - §6 Experiments, Memory: ring of n_sink + W + d slots per request.
 *           - §7 "Compatibility with tree speculation": a tree of width k
 *             reserves n_sink + W + d*k slots; candidates share sink+window
 *             and diverge over the last d positions.
 *           - §3, Eq. (1) context: d = gamma + 1 (the engine's num_draft_tokens).
 *           - §5, Eq. (4): alpha_j and AL.
 *   [BLOG]  "arXiv'26 | Wind-MTP" (marsggbo.github.io), §3.1: the worked block
 *           table at S = 1,000,000 and the ring formula pos mod (n_sink+W+d).
 *
 * Readings where the pages are silent or ambiguous (each is listed in the
 * repository's design notes):
 *   R1 positions and slots are 0-based (the blog's example is 1-based);
 *   R2 draft step j (0-based) attends kv_len = S + j + 1 keys: the draft token
 *      appends its own K/V before attending;
 *   R3 the windowing test is strict (kv_len > n_sink + W), as in the pseudocode;
 *   R4 ring: sink slots are pinned; non-sink positions roll with modulus
 *      W + d*k, so the ring totals n_sink + W + d*k slots and agrees with the
 *      literal formula for every position below that total;
 *   R5 tree node (branch b, depth i) sits at logical position S + i; its slot
 *      is the ring rule shifted by b*d (side branches never use sink slots);
 *      its key set is keep(S + i + 1) with the draft positions S..S+i taken
 *      from its own branch;
 *   R6 GQA: query head h reads KV head h / (H_q / H_kv);
 *   R7 natural exp/log; lse is over the scaled logits; an empty key set gives
 *      out = 0 and lse = -inf.
 *
 * Parity of the attention function is pinned by closed forms and special cases
 * (see tests/test_oracle_attention.py); the pages print no attention values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ECAPACITY (-2)
#define ORC_EBOUNDS (-4)

/* bf16 bit pattern -> double.  bf16 is the upper half of an IEEE binary32,
 * so the conversion is exact. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Key selection: [WMTP] App. A pseudocode.
 *   if WINDOW and S > n_sink + W: keep = range(0, n_sink) + range(S - W, S)
 *   else:                         keep = range(0, S)
 * Here s_kv is the pseudocode's S (the kv length the draft step sees).
 * Writes the positions to pos_out (when non-NULL) and returns their count. */
int64_t orc_keep(int64_t s_kv, int64_t n_sink, int64_t window, int windowed,
                 int64_t *pos_out) {
    int64_t n = 0;
    if (s_kv <= 0) return 0;
    if (windowed && s_kv > n_sink + window) {
        for (int64_t p = 0; p < n_sink; ++p) {
            if (pos_out) pos_out[n] = p;
            ++n;
        }
        for (int64_t p = s_kv - window; p < s_kv; ++p) {
            if (pos_out) pos_out[n] = p;
            ++n;
        }
    } else {
        for (int64_t p = 0; p < s_kv; ++p) {
            if (pos_out) pos_out[n] = p;
            ++n;
        }
    }
    return n;
}

/* ------------------------------------------------------------------------ */
/* Ring slot of logical position p on tree branch `branch` (0 for a chain).
 * [WMTP] App. A: slot = ring_base(r) + logical_pos, modulus n_sink + W + d;
 * §7: a tree of width k reserves n_sink + W + d*k slots.  Reading R4/R5:
 * sinks pinned, the rest rolls with modulus W + d*k, branches offset by b*d.
 * Only branch 0 (the chain) uses sink slots; a side branch drafted while the
 * context is shorter than n_sink rolls in the non-sink region, since the
 * candidates share the sink prefix and diverge only over their own nodes. */
int64_t orc_ring_slot(int64_t ring_base, int64_t p, int64_t branch,
                      int64_t n_sink, int64_t window, int64_t depth,
                      int64_t tree_k) {
    if (p < n_sink && branch == 0) return ring_base + p;
    int64_t modulus = window + depth * tree_k;
    int64_t r = ((p - n_sink) + branch * depth) % modulus;
    if (r < 0) r += modulus; /* a side branch drafted inside the sink range */
    return ring_base + n_sink + r;
}

/* Ring slots for a list of (request, position, branch) triples. */
int orc_ring_map(const int32_t *ring_base, const int32_t *pos,
                 const int32_t *branch, const int32_t *req_of, int64_t n,
                 int64_t n_sink, int64_t window, int64_t depth, int64_t tree_k,
                 int32_t *slots) {
    if (n_sink < 0 || window < 1 || depth < 1 || tree_k < 1) return ORC_EINVAL;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = branch ? branch[i] : 0;
        if (pos[i] < 0 || b < 0 || b >= tree_k) return ORC_EINVAL;
        slots[i] = (int32_t)orc_ring_slot(ring_base[req_of[i]], pos[i], b,
                                          n_sink, window, depth, tree_k);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Draft KV-index builder ([WMTP] §4 Mechanism; App. A).
 * For each draft step j < gamma and request b: kv_len = seq_lens[b] + j + 1
 * (reading R2); positions = keep(kv_len); each position maps to a physical
 * slot through req_to_token[req_pool_idx[b]][p] (paged layout) or through the
 * ring (ring layout, when req_to_token is NULL).
 * Output: table[(j*B + b)*stride + i] and lens[j*B + b]. */
int orc_build_draft_indices(const int32_t *seq_lens, int64_t B, int64_t gamma,
                            int64_t n_sink, int64_t window, int64_t depth,
                            int64_t tree_k, int windowed,
                            const int32_t *req_to_token,
                            const int32_t *req_pool_idx, int64_t rtt_stride,
                            const int32_t *ring_base, int32_t *table,
                            int64_t stride, int32_t *lens) {
    if (B < 0 || gamma < 0 || n_sink < 0 || window < 1 || depth < 1 ||
        tree_k < 1)
        return ORC_EINVAL;
    if (!req_to_token && !ring_base) return ORC_EINVAL;
    for (int64_t j = 0; j < gamma; ++j) {
        for (int64_t b = 0; b < B; ++b) {
            int64_t kv_len = (int64_t)seq_lens[b] + j + 1;
            int64_t n = orc_keep(kv_len, n_sink, window, windowed, NULL);
            if (n > stride) return ORC_ECAPACITY;
            int64_t *pos = (int64_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
            if (!pos) return ORC_EINVAL;
            orc_keep(kv_len, n_sink, window, windowed, pos);
            for (int64_t i = 0; i < n; ++i) {
                int64_t slot = req_to_token
                    ? req_to_token[(int64_t)req_pool_idx[b] * rtt_stride + pos[i]]
                    : orc_ring_slot(ring_base[b], pos[i], 0, n_sink, window,
                                    depth, tree_k);
                table[(j * B + b) * stride + i] = (int32_t)slot;
            }
            lens[j * B + b] = (int32_t)n;
            free(pos);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Draft KV append: row copy of each new token's K and V ([n, H_kv, D]) into
 * pool slot slots[i] (pool layout [num_slots, H_kv, D]). */
int orc_append_kv(const uint16_t *k_new, const uint16_t *v_new,
                  const int32_t *slots, int64_t n, int64_t H_kv, int64_t D,
                  uint16_t *k_pool, uint16_t *v_pool, int64_t num_slots) {
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= num_slots) return ORC_EBOUNDS;
        for (int64_t e = 0; e < H_kv * D; ++e) {
            k_pool[(int64_t)slots[i] * H_kv * D + e] = k_new[i * H_kv * D + e];
            v_pool[(int64_t)slots[i] * H_kv * D + e] = v_new[i * H_kv * D + e];
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Softmax attention of one query row over an explicit key-slot list, fp64.
 *   s_i = scale * sum_d q[d] * k_i[d]
 *   m   = max_i s_i,  w_i = exp(s_i - m)
 *   out = sum_i w_i v_i / sum_i w_i,  lse = m + log sum_i w_i
 * k_pool/v_pool rows for KV head g sit at ((slot * H_kv) + g) * D. */
static int attend_one(const uint16_t *q, const uint16_t *k_pool,
                      const uint16_t *v_pool, int64_t num_slots, int64_t H_kv,
                      int64_t g, int64_t D, const int32_t *slots, int64_t L,
                      double scale, double *s_buf, double *out, double *lse) {
    for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double m = -INFINITY;
    for (int64_t i = 0; i < L; ++i) {
        int64_t slot = slots[i];
        if (slot < 0 || slot >= num_slots) return ORC_EBOUNDS;
        const uint16_t *k = k_pool + (slot * H_kv + g) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += bf16_to_f64(q[d]) * bf16_to_f64(k[d]);
        s_buf[i] = scale * dot;
        if (s_buf[i] > m) m = s_buf[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < L; ++i) {
        double w = exp(s_buf[i] - m);
        const uint16_t *v = v_pool + ((int64_t)slots[i] * H_kv + g) * D;
        for (int64_t d = 0; d < D; ++d) out[d] += w * bf16_to_f64(v[d]);
        z += w;
    }
    for (int64_t d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
    return ORC_OK;
}

/* Draft decode attention over a block table ([WMTP] §4 Mechanism: the reduced
 * table is the key set; no extra mask).
 * q: [B, n_q, H_q, D] bf16 bits.  Query token t of request b reads table row
 * b (table + b*stride, lens[b] entries).  out: [B, n_q, H_q, D]; lse:
 * [B, n_q, H_q].  `rows` lists which flattened (b*n_q + t)*H_q + h rows to
 * compute (NULL = all), so that large cases can be sampled; rows not listed
 * are left untouched.  s_scratch must hold max(lens) * nthreads doubles. */
int orc_draft_decode_attn(const uint16_t *q, int64_t B, int64_t n_q,
                          int64_t H_q, int64_t H_kv, int64_t D,
                          const uint16_t *k_pool, const uint16_t *v_pool,
                          int64_t num_slots, const int32_t *table,
                          int64_t stride, const int32_t *lens, double scale,
                          const int64_t *rows, int64_t n_rows, double *out,
                          double *lse, double *s_scratch, int64_t scratch_len,
                          int nthreads) {
    if (H_kv < 1 || H_q % H_kv != 0 || D < 1) return ORC_EINVAL;
    int64_t G = H_q / H_kv;
    int64_t total = rows ? n_rows : B * n_q * H_q;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        int64_t row = rows ? rows[r] : r;
        int64_t h = row % H_q;
        int64_t bt = row / H_q;
        int64_t b = bt / n_q;
        int64_t L = lens[b];
        if (L > scratch_len || L > stride) {
            status = ORC_ECAPACITY;
            continue;
        }
        int st = attend_one(q + row * D, k_pool, v_pool, num_slots, H_kv,
                            h / G, D, table + b * stride, L, scale,
                            s_scratch + (int64_t)tid * scratch_len,
                            out + row * D, lse + row);
        if (st != ORC_OK) status = st;
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Tree drafting over the ring (reading R5; [WMTP] §7).
 * Request b has committed length seq_lens[b]; its k*d draft nodes are
 * numbered t = branch*d + depth, node (branch, i) at logical position S + i.
 * Node (branch, i) attends keep(S + i + 1): positions below S map through the
 * ring on branch 0 (the committed layout), positions S..S+i map to the node's
 * own branch.  q: [B, k*d, H_q, D].  out/lse as in orc_draft_decode_attn.
 * `rows` / n_rows select (b*k*d + t)*H_q + h rows (NULL = all). */
int orc_tree_draft_attn(const uint16_t *q, int64_t B, int64_t H_q,
                        int64_t H_kv, int64_t D, const uint16_t *k_pool,
                        const uint16_t *v_pool, int64_t num_slots,
                        const int32_t *seq_lens, const int32_t *ring_base,
                        int64_t n_sink, int64_t window, int64_t depth,
                        int64_t tree_k, double scale, const int64_t *rows,
                        int64_t n_rows, double *out, double *lse,
                        int nthreads) {
    if (H_kv < 1 || H_q % H_kv != 0 || n_sink < 0 || window < 1 ||
        depth < 1 || tree_k < 1)
        return ORC_EINVAL;
    int64_t G = H_q / H_kv;
    int64_t n_nodes = tree_k * depth;
    int64_t total = rows ? n_rows : B * n_nodes * H_q;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; ++r) {
        int64_t row = rows ? rows[r] : r;
        int64_t h = row % H_q;
        int64_t bt = row / H_q;
        int64_t b = bt / n_nodes;
        int64_t t = bt % n_nodes;
        int64_t branch = t / depth;
        int64_t i = t % depth;
        int64_t S = seq_lens[b];
        int64_t kv_len = S + i + 1;
        int64_t L = orc_keep(kv_len, n_sink, window, 1, NULL);
        int64_t *pos = (int64_t *)malloc((size_t)(L + 1) * sizeof(int64_t));
        int32_t *slots = (int32_t *)malloc((size_t)(L + 1) * sizeof(int32_t));
        double *s_buf = (double *)malloc((size_t)(L + 1) * sizeof(double));
        if (!pos || !slots || !s_buf) {
            free(pos);
            free(slots);
            free(s_buf);
            status = ORC_EINVAL;
            continue;
        }
        orc_keep(kv_len, n_sink, window, 1, pos);
        for (int64_t e = 0; e < L; ++e) {
            int64_t on_branch = pos[e] < S ? 0 : branch;
            slots[e] = (int32_t)orc_ring_slot(ring_base[b], pos[e], on_branch,
                                              n_sink, window, depth, tree_k);
        }
        int st = attend_one(q + row * D, k_pool, v_pool, num_slots, H_kv,
                            h / G, D, slots, L, scale, s_buf, out + row * D,
                            lse + row);
        free(pos);
        free(slots);
        free(s_buf);
        if (st != ORC_OK) status = st;
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Acceptance length from a histogram, [WMTP] §5 Eq. (4): H[n] counts steps
 * that accepted exactly n draft tokens, n = 0..gamma.
 *   alpha_j = sum_{n>=j} H[n] / sum_{n>=j-1} H[n],  j = 1..gamma
 *   AL      = 1 + sum_{j>=1} prod_{k<=j} alpha_k
 * alpha_j is written to alpha[j-1]; a position nobody reached gets alpha = 0.
 * Returns AL (NaN for an empty histogram). */
double orc_acceptance_length(const double *H, int64_t gamma, double *alpha) {
    double total = 0.0;
    for (int64_t n = 0; n <= gamma; ++n) total += H[n];
    if (!(total > 0.0)) return NAN;
    for (int64_t j = 1; j <= gamma; ++j) {
        double num = 0.0, den = 0.0;
        for (int64_t n = j; n <= gamma; ++n) num += H[n];
        for (int64_t n = j - 1; n <= gamma; ++n) den += H[n];
        alpha[j - 1] = den > 0.0 ? num / den : 0.0;
    }
    double al = 1.0;
    for (int64_t j = 1; j <= gamma; ++j) {
        double prod = 1.0;
        for (int64_t k = 1; k <= j; ++k) prod *= alpha[k - 1];
        al += prod;
    }
    return al;
}

/* ------------------------------------------------------------------------ */
/* fp8 KV.  [WMTP] §6, "Robustness to KV-cache quantization": windowing
 * composes with an fp8 KV cache (the saving scales with bytes per entry), and
 * the pages' own fp8-KV path has no fused attention kernel; the checkpoints
 * ship per-layer fp8 KV scales.  Reading R13: K and V rows are stored
 * as OCP FP8 E4M3 codes with one fp32 scale per KV head; the stored value is
 * code_value * scale, and a new row is quantised as
 *   code = E4M3_RNE_satfinite( (float)x * (1.0f / scale) )
 * in fp32 arithmetic (the integer decision in the same precision as the
 * kernel).  E4M3: sign bit 7, exponent bits 6..3 with bias 7, mantissa bits
 * 2..0; exponent 0 encodes subnormals m * 2^-9; S.1111.111 is NaN (no
 * infinities); the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_f64(uint8_t c) {
    int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even code; finite magnitudes beyond
 * 448 (and infinities) saturate to 448; NaN gives 0x7F.  Plain search over
 * the 127 non-negative finite codes, compared in fp64 (exact). */
uint8_t orc_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    static double value[0x7F];
    static int have_values = 0;
    if (!have_values) {
        for (int c = 0; c < 0x7F; ++c) value[c] = orc_e4m3_to_f64((uint8_t)c);
        have_values = 1;
    }
    int best = 0;
    double best_d = a;  /* distance to code 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(value[c] - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Quantising append: each new token's K and V rows (bf16) become E4M3 codes
 * with the per-KV-head scales (reading R13), written to pool slot slots[i]. */
int orc_append_kv_fp8(const uint16_t *k_new, const uint16_t *v_new,
                      const int32_t *slots, int64_t n, int64_t H_kv, int64_t D,
                      const float *k_scale, const float *v_scale,
                      uint8_t *k_pool, uint8_t *v_pool, int64_t num_slots) {
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= num_slots) return ORC_EBOUNDS;
        for (int64_t g = 0; g < H_kv; ++g) {
            float ik = 1.0f / k_scale[g], iv = 1.0f / v_scale[g];
            for (int64_t d = 0; d < D; ++d) {
                int64_t e = g * D + d;
                float kx = (float)bf16_to_f64(k_new[i * H_kv * D + e]);
                float vx = (float)bf16_to_f64(v_new[i * H_kv * D + e]);
                float ky = kx * ik, vy = vx * iv;
                k_pool[(int64_t)slots[i] * H_kv * D + e] = orc_f32_to_e4m3(ky);
                v_pool[(int64_t)slots[i] * H_kv * D + e] = orc_f32_to_e4m3(vy);
            }
        }
    }
    return ORC_OK;
}

/* attend_one over an fp8 pool: k_i = code * k_scale, v_i = code * v_scale
 * (fp64), otherwise the same definition. */
static int attend_one_fp8(const uint16_t *q, const uint8_t *k_pool,
                          const uint8_t *v_pool, int64_t num_slots, int64_t H_kv,
                          int64_t g, int64_t D, const int32_t *slots, int64_t L,
                          double scale, double k_scale, double v_scale,
                          double *s_buf, double *out, double *lse) {
    for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) {
        *lse = -INFINITY;
        return ORC_OK;
    }
    double m = -INFINITY;
    for (int64_t i = 0; i < L; ++i) {
        int64_t slot = slots[i];
        if (slot < 0 || slot >= num_slots) return ORC_EBOUNDS;
        const uint8_t *k = k_pool + (slot * H_kv + g) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += bf16_to_f64(q[d]) * (orc_e4m3_to_f64(k[d]) * k_scale);
        s_buf[i] = scale * dot;
        if (s_buf[i] > m) m = s_buf[i];
    }
    double z = 0.0;
    for (int64_t i = 0; i < L; ++i) {
        double w = exp(s_buf[i] - m);
        const uint8_t *v = v_pool + ((int64_t)slots[i] * H_kv + g) * D;
        for (int64_t d = 0; d < D; ++d) out[d] += w * (orc_e4m3_to_f64(v[d]) * v_scale);
        z += w;
    }
    for (int64_t d = 0; d < D; ++d) out[d] /= z;
    *lse = m + log(z);
    return ORC_OK;
}

/* orc_draft_decode_attn over fp8 pools with per-KV-head scales. */
int orc_draft_decode_attn_fp8(const uint16_t *q, int64_t B, int64_t n_q,
                              int64_t H_q, int64_t H_kv, int64_t D,
                              const uint8_t *k_pool, const uint8_t *v_pool,
                              const float *k_scale, const float *v_scale,
                              int64_t num_slots, const int32_t *table,
                              int64_t stride, const int32_t *lens, double scale,
                              const int64_t *rows, int64_t n_rows, double *out,
                              double *lse, double *s_scratch, int64_t scratch_len,
                              int nthreads) {
    if (H_kv < 1 || H_q % H_kv != 0 || D < 1) return ORC_EINVAL;
    int64_t G = H_q / H_kv;
    int64_t total = rows ? n_rows : B * n_q * H_q;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        int64_t row = rows ? rows[r] : r;
        int64_t h = row % H_q;
        int64_t bt = row / H_q;
        int64_t b = bt / n_q;
        int64_t L = lens[b];
        if (L > scratch_len || L > stride) {
            status = ORC_ECAPACITY;
            continue;
        }
        int64_t g = h / G;
        int st = attend_one_fp8(q + row * D, k_pool, v_pool, num_slots, H_kv, g, D,
                                table + b * stride, L, scale, (double)k_scale[g],
                                (double)v_scale[g],
                                s_scratch + (int64_t)tid * scratch_len,
                                out + row * D, lse + row);
        if (st != ORC_OK) status = st;
    }
    return status;
}
