#include "tmap.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace sca {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

static cudaError_t make_tmap(CUtensorMap* map, CUtensorMapDataType type, int64_t eb, const void* base, int D,
                             int64_t rows, int H, int B, const View& v, int box_d, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  if (reinterpret_cast<uintptr_t>(base) % 16) return cudaErrorNotSupported;
  // strides of size-1 dimensions are never used; keep them legal
  int64_t ss = v.s, sh = v.h, sb = v.b;
  if (H == 1) sh = ss * (rows > 0 ? rows : 1);
  if (B == 1) sb = sh * H;
  if ((ss * eb) % 16 || (sh * eb) % 16 || (sb * eb) % 16) return cudaErrorNotSupported;
  if (rows < 1) rows = 1;  // an empty slab is never read; keep the map legal
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ss * eb), static_cast<cuuint64_t>(sh * eb),
                           static_cast<cuuint64_t>(sb * eb)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_d), static_cast<cuuint32_t>(box_rows), 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, type, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorNotSupported;
}

cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                           const View& v, int box_d, int box_rows) {
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, D, rows, H, B, v, box_d, box_rows);
}

cudaError_t make_tmap_f16(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                          const View& v, int box_d, int box_rows) {
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, D, rows, H, B, v, box_d, box_rows);
}

cudaError_t make_tmap_f32(CUtensorMap* map, const void* base, int D, int64_t rows, int H, int B,
                          const View& v, int box_d, int box_rows) {
  return make_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, D, rows, H, B, v, box_d, box_rows);
}

}  // namespace sca
