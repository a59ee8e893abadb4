// TMA tensor-map creation for [B, H, rows, D] bf16/fp16/fp32 views (host only).  The
// driver entry point is resolved at run time through the runtime API, so
// the library does not link against libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace sca {

// 4-D map (D, rows, H, B), box (box_d, box_rows, 1, 1), 128-byte swizzle,
// out-of-range elements read as zero.  Returns cudaErrorNotSupported when
// the layout breaks a TMA rule (alignment, stride multiple of 16 bytes).
cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                           const View& v, int box_d, int box_rows);

// Same for fp16 tensors (the same layout rules as bf16).
cudaError_t make_tmap_f16(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                          const View& v, int box_d, int box_rows);

// Same for fp32 tensors (box_d * 4 bytes must be 128 for the swizzle).
cudaError_t make_tmap_f32(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                          const View& v, int box_d, int box_rows);

}  // namespace sca
