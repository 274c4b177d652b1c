// wmtp_diag.cu -- attention-mass diagnostics of the windowed draft.
//
// "Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
// Context" (arXiv 2607.21535), §5 "A partition-function view" and App. C,
// Table 12: for a draft query with logits z_k over the full key set, the
// mass inside the kept set (sinks + window) is Z_w / Z, the mass beyond it
// Z_far / Z = 1 - Z_w / Z; win_perturb = ||o_full - o_win|| / ||o_full|| is
// the relative change of the read-out o = sum_k p_k v_k when the far keys are
// dropped; tail out-frac = ||sum_far p_k v_k|| / ||o_full||.
//
// Both attentions carry their log partition function (lse), so with
// a = Z_w / Z = exp(lse_win - lse_full) and o_full = a o_win + sum_far p v,
// every quantity follows from (o_full, lse_full, o_win, lse_win): one warp
// per query row, three fp32 norms over D.
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
    const float *__restrict__ o_full, const float *__restrict__ lse_full,
    const float *__restrict__ o_win, const float *__restrict__ lse_win, int64_t rows, int32_t D,
    float *__restrict__ in_win, float *__restrict__ win_perturb, float *__restrict__ tail_frac) {
    griddep_launch_dependents();
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float lf = lse_full[row], lw = lse_win[row];
    // a = Z_w / Z; an empty kept set (lse_win = -inf) gives 0, an empty row 0
    const float a = (lf == -INFINITY || lw == -INFINITY) ? 0.f : fminf(expf(lw - lf), 1.f);
    const float *of = o_full + row * D, *ow = o_win + row * D;
    float nf = 0.f, nd = 0.f, nt = 0.f;  // ||o_full||^2, ||o_full - o_win||^2, ||o_full - a o_win||^2
    for (int d = lane; d < D; d += 32) {
        const float f = of[d], w = ow[d];
        nf += f * f;
        nd += (f - w) * (f - w);
        nt += (f - a * w) * (f - a * w);
    }
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) {
        nf += __shfl_xor_sync(0xffffffffu, nf, sh);
        nd += __shfl_xor_sync(0xffffffffu, nd, sh);
        nt += __shfl_xor_sync(0xffffffffu, nt, sh);
    }
    if (lane == 0) {
        const float inv = nf > 0.f ? rsqrtf(nf) : 0.f;
        if (in_win) in_win[row] = a;
        if (win_perturb) win_perturb[row] = sqrtf(nd) * inv;
        if (tail_frac) tail_frac[row] = sqrtf(nt) * inv;
    }
}

}  // namespace
}  // namespace wmtp

using namespace wmtp;

extern "C" {

wmtp_status wmtp_attn_mass_diagnostics(const float *o_full, const float *lse_full,
                                       const float *o_win, const float *lse_win, int64_t rows,
                                       int32_t D, float *in_win, float *win_perturb,
                                       float *tail_out_frac, void *stream) {
    if (rows < 0 || D < 1) return WMTP_EINVAL;
    if (rows == 0) return WMTP_OK;
    if (!o_full || !lse_full || !o_win || !lse_win) return WMTP_EINVAL;
    if (!in_win && !win_perturb && !tail_out_frac) return WMTP_EINVAL;
    const int64_t blocks = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (blocks > 0x7fffffffLL) return WMTP_EINVAL;
    PdlLaunch L(dim3((unsigned)blocks), dim3(kRowsPerCta * 32), 0, as_stream(stream));
    return cudaLaunchKernelEx(&L.cfg, attn_mass_kernel, o_full, lse_full, o_win, lse_win, rows, D,
                              in_win, win_perturb, tail_out_frac) == cudaSuccess
               ? WMTP_OK
               : WMTP_ECUDA;
}

}  // extern "C"
