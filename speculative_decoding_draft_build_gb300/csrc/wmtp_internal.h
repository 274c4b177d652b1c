// wmtp_internal.h -- host-side helpers shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "wmtp.h"

namespace wmtp {

// Each translation unit keeps its own device error word (no relocatable
// device code is needed); these read-and-optionally-clear them.
cudaError_t read_index_error(int32_t *code, bool clear);
cudaError_t read_attn_error(int32_t *code, bool clear);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline wmtp_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? WMTP_OK : WMTP_ECUDA;
}

}  // namespace wmtp
