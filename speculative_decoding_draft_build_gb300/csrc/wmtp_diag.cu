// wmtp_diag.cu -- attention-mass diagnostics of the windowed draft.
//
// "Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
// Context" (arXiv 2607.21535), §5 "A partition-function view" and App. C,
// Table 12: for a draft query with logits z_k over the full key set, the
// partition function splits as Z = Z_w + Z_far over the kept set (sinks +
// window) and the dropped ("far") keys.  The quantities are the in-window
// mass Z_w / Z, win_perturb = ||o_full - o_win|| / ||o_full|| (the relative
// change of the read-out o = sum_k p_k v_k when the far keys are dropped) and
// the tail out-frac ||sum_far p_k v_k|| / ||o_full||.
//
// They are computed from the two disjoint parts of the full key set, each an
// attention output with its log partition function: (o_win, lse_win) over
// the kept keys and (o_far, lse_far) over the far keys.  With
//   a = Z_w / Z = 1 / (1 + e^(lse_far - lse_win)),  b = Z_far / Z = 1 - a
// (both taken from the same exponential, so b is never 1 - a rounded),
//   o_full = a o_win + b o_far,
//   tail   = b ||o_far|| / ||o_full||,
//   win_perturb = ||o_full - o_win|| / ||o_full|| = b ||o_far - o_win|| / ||o_full||,
// so a small far share is never obtained by subtracting two nearly equal
// outputs.  The merged (o_full, lse_full) is the full-context attention
// itself (the LSE merge of the two parts) and can be written too.  One warp
// per query row.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "wmtp.h"
#include "wmtp_internal.h"
#include "wmtp_ptx.cuh"

namespace wmtp {
namespace {

constexpr int kRowsPerCta = 8;  // one warp per row

__global__ void __launch_bounds__(kRowsPerCta * 32) attn_mass_kernel(
    const float *__restrict__ o_win, const float *__restrict__ lse_win,
    const float *__restrict__ o_far, const float *__restrict__ lse_far, int64_t rows, int32_t D,
    float *__restrict__ in_win, float *__restrict__ win_perturb, float *__restrict__ tail_frac,
    float *__restrict__ o_full, float *__restrict__ lse_full) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float lw = lse_win[row], lf = lse_far[row];
    // shares of the two parts; an empty part (lse = -inf) has share 0, and a
    // row with both parts empty gets a = b = 0
    float a = 0.f, b = 0.f;
    if (lw != -INFINITY || lf != -INFINITY) {
        const float d = lf - lw;  // +inf: no kept key; -inf: no far key
        if (d > 0.f) {
            const float e = expf(-d);
            a = e / (1.f + e);
            b = 1.f / (1.f + e);
        } else {
            const float e = expf(d);
            a = 1.f / (1.f + e);
            b = e / (1.f + e);
        }
    }
    const float *ow = o_win + row * D, *of = o_far + row * D;
    float n_full = 0.f, n_far = 0.f, n_diff = 0.f;  // ||o_full||^2, ||o_far||^2, ||o_far - o_win||^2
    for (int d = lane; d < D; d += 32) {
        const float w = a > 0.f ? ow[d] : 0.f;
        const float f = b > 0.f ? of[d] : 0.f;
        const float full = a * w + b * f;
        if (o_full) o_full[row * D + d] = full;
        n_full += full * full;
        n_far += f * f;
        n_diff += (f - w) * (f - w);
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        n_full += __shfl_xor_sync(0xffffffffu, n_full, sh);
        n_far += __shfl_xor_sync(0xffffffffu, n_far, sh);
        n_diff += __shfl_xor_sync(0xffffffffu, n_diff, sh);
    }
    if (lane == 0) {
        const float inv = n_full > 0.f ? 1.f / sqrtf(n_full) : 0.f;
        if (in_win) in_win[row] = a;
        if (win_perturb) win_perturb[row] = b > 0.f ? b * sqrtf(n_diff) * inv : 0.f;
        if (tail_frac) tail_frac[row] = b > 0.f ? b * sqrtf(n_far) * inv : 0.f;
        if (lse_full) {
            const float m = fmaxf(lw, lf);
            lse_full[row] = m == -INFINITY ? -INFINITY : m + log1pf(expf(-fabsf(lw - lf)));
        }
    }
}

}  // namespace
}  // namespace wmtp

using namespace wmtp;

extern "C" {

wmtp_status wmtp_attn_mass_diagnostics(const float *o_win, const float *lse_win, const float *o_far,
                                       const float *lse_far, int64_t rows, int32_t D, float *in_win,
                                       float *win_perturb, float *tail_out_frac, float *o_full,
                                       float *lse_full, void *stream) {
    if (rows < 0 || D < 1) return WMTP_EINVAL;
    if (rows == 0) return WMTP_OK;
    if (!o_win || !lse_win || !o_far || !lse_far) return WMTP_EINVAL;
    if (!in_win && !win_perturb && !tail_out_frac && !o_full && !lse_full) return WMTP_EINVAL;
    const int64_t blocks = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (blocks > 0x7fffffffLL) return WMTP_EINVAL;
    PdlLaunch L(dim3((unsigned)blocks), dim3(kRowsPerCta * 32), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, attn_mass_kernel, o_win, lse_win, o_far, lse_far, rows, D, in_win,
                              win_perturb, tail_out_frac, o_full, lse_full) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"
