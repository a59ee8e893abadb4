// HBM-bound kernels: zigzag permute, ring staging copy, exact lse merge, the
// backward's delta = rowsum(dO * O) and its bf16 -> fp16 input cast.  All
// move 16-byte vectors where the layout allows; none allocates.
#include <cmath>

#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "ptx.cuh"

namespace sca {

// ------------------------------------------------------------ zigzag permute
//
// The permute moves whole chunks of c = S/(2P) rows: destination chunk x of
// sequence o is a contiguous copy of one source chunk.  Forward (natural ->
// shard-major): destination chunk 2r holds natural chunk r and 2r+1 holds
// natural chunk 2P-1-r.  Inverse: natural chunk n comes from shard-major
// chunk 2n (n < P) or 2(2P-1-n)+1.
//
// Work is cut into tiles of kPermThreads * kPermUnroll vectors inside one
// chunk (a chunk's last tile may be short).  The grid is one wave of
// resident blocks, and block b copies tiles b, b + grid, ...: every block
// gets the same number of tiles to within one, so no partial second wave
// idles most of the GPU.  Each thread has kPermUnroll 16-byte loads in
// flight before its first store; loads and stores are fully coalesced.

constexpr int kPermThreads = 256;
constexpr int kPermUnroll = 8;

__host__ __device__ __forceinline__ int zz_src_chunk(int ch, int P, int inverse) {
  if (!inverse) {
    const int r = ch >> 1;
    return (ch & 1) ? (2 * P - 1 - r) : r;
  }
  return ch < P ? 2 * ch : 2 * (2 * P - 1 - ch) + 1;
}

template <typename V>
__global__ void __launch_bounds__(kPermThreads) zigzag_permute_kernel(const V* __restrict__ src,
                                                                      V* __restrict__ dst, int64_t nseg,
                                                                      int64_t chunk_vecs, int64_t tiles_per_chunk,
                                                                      int P, int inverse) {
  constexpr int64_t kTile = static_cast<int64_t>(kPermThreads) * kPermUnroll;
  const int two_p = 2 * P;
  const int64_t n_tiles = nseg * tiles_per_chunk;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t g = t / tiles_per_chunk;             // destination chunk (o, ch)
    const int64_t base = (t - g * tiles_per_chunk) * kTile;
    const int64_t o = g / two_p;
    const int ch = static_cast<int>(g - o * two_p);
    const V* s = src + (o * two_p + zz_src_chunk(ch, P, inverse)) * chunk_vecs + base;
    V* d = dst + g * chunk_vecs + base;
    const int64_t n = chunk_vecs - base < kTile ? chunk_vecs - base : kTile;
    V tmp[kPermUnroll];
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int i = u * kPermThreads + threadIdx.x;
      if (i < n) tmp[u] = s[i];
    }
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int i = u * kPermThreads + threadIdx.x;
      if (i < n) d[i] = tmp[u];
    }
  }
}

// The same permute by bulk copies.  Every chunk is contiguous in both
// tensors, so it is cut into pieces of up to kBulkPiece bytes, each moved
// global -> shared -> global by the TMA unit.  One thread drives a block:
// loads run kBulkStages-1 pieces ahead of the stores, and a stage is
// reloaded once the store that used it has read it.  Two blocks per SM keep
// ~128 KB of loads and as many stores in flight per SM.  Waits are bounded:
// one that gives up records SCA_ERR_TIMEOUT and ends the block.

constexpr int kBulkStages = 3;
constexpr int kBulkPiece = 32 * 1024;
constexpr int kBulkSmem = kBulkStages * kBulkPiece + 64;

__global__ void __launch_bounds__(32) zigzag_permute_bulk_kernel(const uint8_t* __restrict__ src,
                                                                 uint8_t* __restrict__ dst, int64_t nseg,
                                                                 int64_t chunk_bytes, int64_t pieces_per_chunk,
                                                                 int P, int inverse, int* status) {
  extern __shared__ __align__(128) uint8_t bsm[];
  uint64_t* full = reinterpret_cast<uint64_t*>(bsm + kBulkStages * kBulkPiece);
  int* abort = reinterpret_cast<int*>(full + kBulkStages);
  if (threadIdx.x != 0) return;   // one thread drives the copies
  for (int s = 0; s < kBulkStages; ++s) mbar_init(&full[s], 1);
  *abort = 0;
  fence_mbar_init();
  const int two_p = 2 * P;
  const int64_t n_pieces = nseg * pieces_per_chunk;
  const int64_t mine = n_pieces > blockIdx.x ? (n_pieces - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto locate = [&](int64_t i, const uint8_t*& s, uint8_t*& d, uint32_t& bytes) {
    const int64_t p = blockIdx.x + i * gridDim.x;
    const int64_t g = p / pieces_per_chunk;                 // destination chunk (o, ch)
    const int64_t off = (p - g * pieces_per_chunk) * kBulkPiece;
    const int64_t o = g / two_p;
    const int ch = static_cast<int>(g - o * two_p);
    s = src + (o * two_p + zz_src_chunk(ch, P, inverse)) * chunk_bytes + off;
    d = dst + g * chunk_bytes + off;
    bytes = static_cast<uint32_t>(min64(kBulkPiece, chunk_bytes - off));
  };
  constexpr int kAhead = kBulkStages - 1;
  for (int64_t i = 0; i < mine + kAhead; ++i) {
    const int64_t j = i - kAhead;   // the piece stored this iteration
    if (j >= 0 && j < mine) {
      const int st = static_cast<int>(j % kBulkStages);
      if (!mbar_wait(&full[st], static_cast<uint32_t>((j / kBulkStages) & 1), abort, status)) break;
      const uint8_t* s;
      uint8_t* d;
      uint32_t bytes;
      locate(j, s, d, bytes);
      bulk_store(d, bsm + st * kBulkPiece, bytes);
      bulk_commit();
    }
    if (i < mine) {
      const int st = static_cast<int>(i % kBulkStages);
      // the stage's previous piece (i - kBulkStages) was stored last
      // iteration: let that store read it (the one just issued may pend)
      if (i >= kBulkStages) bulk_wait_read<1>();
      const uint8_t* s;
      uint8_t* d;
      uint32_t bytes;
      locate(i, s, d, bytes);
      mbar_arrive_expect_tx(&full[st], bytes);
      bulk_load(bsm + st * kBulkPiece, s, bytes, &full[st]);
    }
  }
  if (*abort) {   // let loads still in flight land before the block's shared memory goes away
    for (int64_t i = (mine > kBulkStages ? mine - kBulkStages : 0); i < mine; ++i)
      mbar_wait_drain(&full[i % kBulkStages], static_cast<uint32_t>((i / kBulkStages) & 1));
  }
  bulk_wait_read<0>();   // every store has read shared memory before the block exits
}

// ------------------------------------------------------------ ring hand-off
//
// Every copy of one hand-off (strided 2-D copies of 16-byte vectors) in one
// launch of kCopyBlocksPerSm blocks of kCopyThreads per SM at 72 registers:
// two such blocks (9216 registers) fit next to a forward CTA (160 x 352)
// or a backward one (168 x 320), so the hand-off proceeds while the SMs
// compute.  Beside a running attention step a copy moves only a few hundred
// GB/s; the second block per SM nearly halved the copy stream's busy time
// on the 2D split (8.3 -> 5.0 ms per step) and the step time it exposes
// (9.2% -> 4.1%).  The copies are cut into units of one row by kCopySlice
// vectors (16 KB); block b takes units b, b + grid, ...  Each thread keeps
// kCopyUnroll 16-byte loads in flight.

constexpr int kCopyThreads = 64;
constexpr int kCopyUnroll = 12;
constexpr int kCopyBlocksPerSm = 2;
constexpr int kCopySlice = kCopyThreads * kCopyUnroll;   // vectors per unit

struct CopyJob {
  const uint4* src;
  uint4* dst;
  int64_t spitch, dpitch;     // row pitches, vectors
  int32_t height, width;      // rows, vectors per row
  int32_t slices;             // units per row
  int32_t units_before;       // units of the jobs before this one
};

struct CopyBatch {
  CopyJob job[SCA_MAX_COPIES];
  int32_t n, units;
};
static_assert(sizeof(CopyBatch) <= 32764, "kernel parameters");

__global__ void __launch_bounds__(kCopyThreads) ring_copy_kernel(const __grid_constant__ CopyBatch cb) {
  for (int32_t u = blockIdx.x; u < cb.units; u += gridDim.x) {
    int j = 0;
    while (j + 1 < cb.n && cb.job[j + 1].units_before <= u) ++j;
    const CopyJob& c = cb.job[j];
    const int32_t local = u - c.units_before;
    const int32_t r = local / c.slices;
    const int32_t c0 = (local - r * c.slices) * kCopySlice;
    const int32_t nv = c.width - c0 < kCopySlice ? c.width - c0 : kCopySlice;
    const uint4* s = c.src + r * c.spitch + c0;
    uint4* d = c.dst + r * c.dpitch + c0;
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) {
      const int32_t i = k * kCopyThreads + threadIdx.x;
      if (i < nv) v[k] = s[i];
    }
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) {
      const int32_t i = k * kCopyThreads + threadIdx.x;
      if (i < nv) d[i] = v[k];
    }
  }
}

// ---------------------------------------------------------------- lse merge
//
// One group of L = D/4 lanes per row; each lane owns 4 consecutive columns
// (one 16-byte vector) of every partial.  The lse values are read by the
// lanes of the group and reduced with shuffles.

constexpr int kMergeThreads = 256;
// up to NF partials (a template parameter, 4 or 8) every load of a row is
// issued at once; more go through the two-pass path
constexpr int kMergeMaxFast = 8;

__device__ __forceinline__ int64_t zz_natural_row(int64_t row, int64_t S, int P) {
  const int64_t o = row / S;
  const int64_t x = row - o * S;
  const int64_t c = S / (2 * P);
  const int64_t r = x / (2 * c);
  const int64_t w = x - r * 2 * c;
  const int64_t nat = w < c ? r * c + w : (2 * P - 1 - r) * c + (w - c);
  return o * S + nat;
}

// o_out / lse_out may be partial p's own rows (the host allows that exact
// alias and no other overlap), so the inputs are not declared __restrict__,
// and every lane of a row's group has finished reading before any lane of
// the group stores (the lse of a row is read by all L lanes and written by
// lane 0).
template <int L, int NF>
__global__ void __launch_bounds__(kMergeThreads) merge_lse_kernel(
    const float* o_parts, const float* lse_parts, int n, int64_t rows,
    int64_t ops, int64_t lps, float* o_out, float* lse_out, __nv_bfloat16* ob_out, int uP, int64_t S) {
  constexpr int RPW = 32 / L;  // rows per warp
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, li = lane % L;
  const unsigned gmask = (L == 32) ? 0xffffffffu : (((1u << L) - 1u) << (sub * L));
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kMergeThreads) >> 5;
  const int D = 4 * L;
  for (int64_t row0 = warp * RPW; row0 < rows; row0 += nwarps * RPW) {
    const int64_t row = row0 + sub;
    const bool active = row < rows;
    float M = -INFINITY;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (n <= NF) {
      // every partial's o chunk and lse issued together (one round trip to
      // memory per row, not two), then the same sums in the same order as
      // the general path below
      if (active) {
        float4 v[NF];
        float w[NF];
#pragma unroll
        for (int u = 0; u < NF; ++u)
          if (u < n) {
            v[u] = *reinterpret_cast<const float4*>(o_parts + u * ops + row * D + 4 * li);
            w[u] = lse_parts[u * lps + row];
          }
#pragma unroll
        for (int u = 0; u < NF; ++u)
          if (u < n) M = fmaxf(M, w[u]);
        const float M0 = (M == -INFINITY) ? 0.f : M;
#pragma unroll
        for (int u = 0; u < NF; ++u)
          if (u < n) {
            const float wu = expf(w[u] - M0);   // exp(-inf) = 0 for empty partials
            wsum += wu;
            acc.x += wu * v[u].x; acc.y += wu * v[u].y; acc.z += wu * v[u].z; acc.w += wu * v[u].w;
          }
      }
    } else {
      // max lse over partials: lane li reads partials li, li+L, ...
      if (active)
        for (int p = li; p < n; p += L) M = fmaxf(M, lse_parts[p * lps + row]);
#pragma unroll
      for (int off = L / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(gmask, M, off));
      const float M0 = (M == -INFINITY) ? 0.f : M;
      if (active) {
        int p = 0;
        for (; p + 4 <= n; p += 4) {
          float4 v[4];
          float w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            v[u] = *reinterpret_cast<const float4*>(o_parts + (p + u) * ops + row * D + 4 * li);
            w[u] = lse_parts[(p + u) * lps + row];
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float wu = expf(w[u] - M0);   // exp(-inf) = 0 for empty partials
            wsum += wu;
            acc.x += wu * v[u].x; acc.y += wu * v[u].y; acc.z += wu * v[u].z; acc.w += wu * v[u].w;
          }
        }
        for (; p < n; ++p) {
          const float4 v = *reinterpret_cast<const float4*>(o_parts + p * ops + row * D + 4 * li);
          const float wu = expf(lse_parts[p * lps + row] - M0);
          wsum += wu;
          acc.x += wu * v.x; acc.y += wu * v.y; acc.z += wu * v.z; acc.w += wu * v.w;
        }
      }
    }
    __syncwarp(gmask);   // a row's group is uniform in `active`; all its loads are done
    if (active) {
      const float M0 = (M == -INFINITY) ? 0.f : M;
      const bool empty = (M == -INFINITY);
      const float inv = empty ? 0.f : 1.f / wsum;
      acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
      const int64_t orow = uP > 0 ? zz_natural_row(row, S, uP) : row;
      *reinterpret_cast<float4*>(o_out + orow * D + 4 * li) = acc;
      if (ob_out) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(ob_out + orow * D + 4 * li) = pk;
      }
      if (li == 0) lse_out[orow] = empty ? -INFINITY : M0 + logf(wsum);
    }
  }
}

// -------------------------------------------------------------------- delta

template <int L, typename T>
__global__ void __launch_bounds__(kMergeThreads) delta_kernel(const float* __restrict__ o,
                                                              const T* __restrict__ dout,
                                                              float* __restrict__ delta, int64_t rows) {
  constexpr int RPW = 32 / L;
  const int lane = threadIdx.x & 31;
  const int sub = lane / L, li = lane % L;
  const unsigned gmask = (L == 32) ? 0xffffffffu : (((1u << L) - 1u) << (sub * L));
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kMergeThreads) >> 5;
  const int D = 4 * L;
  for (int64_t row0 = warp * RPW; row0 < rows; row0 += nwarps * RPW) {
    const int64_t row = row0 + sub;
    float s = 0.f;
    if (row < rows) {
      const float4 ov = *reinterpret_cast<const float4*>(o + row * D + 4 * li);
      const T* dp = dout + row * D + 4 * li;
      s = ov.x * to_f32(dp[0]) + ov.y * to_f32(dp[1]) + ov.z * to_f32(dp[2]) + ov.w * to_f32(dp[3]);
    }
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) s += __shfl_xor_sync(gmask, s, off);
    if (row < rows && li == 0) delta[row] = s;
  }
}

// ------------------------------------------------------- bf16 -> fp16 cast
//
// Eight values per 16-byte vector; grid-stride over the vectors.  Each bf16
// is widened exactly to fp32 (its bits in the high half) and rounded to fp16
// by the hardware conversion.  A finite bf16 value above the fp16 range
// (|x| >= 65536; the largest bf16 below that, 65280, converts exactly)
// becomes +-inf in fp16: the kernel records SCA_ERR_RANGE in the status word
// when it meets one, and still writes the converted value.

constexpr int kCastThreads = 256;

__global__ void __launch_bounds__(kCastThreads) cast_bf16_f16_kernel(const uint4* __restrict__ src,
                                                                     uint4* __restrict__ dst, int64_t nvec,
                                                                     int* status) {
  bool bad = false;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(kCastThreads) + threadIdx.x; i < nvec;
       i += static_cast<int64_t>(gridDim.x) * kCastThreads) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      bad |= bf16x2_beyond_f16(w[k]);
      const __half2 h = __floats2half2_rn(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
      o[k] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (bad) report(status, SCA_ERR_RANGE);
}

static int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

static int grid_for(int64_t work_items, int per_block) {
  int64_t blocks = (work_items + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

// Do [a, a + a_bytes) and [b, b + b_bytes) intersect?
static bool overlap(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(b_bytes) && y < x + static_cast<uintptr_t>(a_bytes);
}

// Does [out, out + bytes) overlap one of the n regions base + p * stride of
// `bytes` each, other than (when exact_ok) by coinciding with it exactly?
static bool bad_overlap(const void* out, int64_t bytes, const void* base, int64_t stride_bytes, int n,
                        int64_t part_bytes, bool exact_ok) {
  for (int p = 0; p < n; ++p) {
    const void* part = static_cast<const char*>(base) + p * stride_bytes;
    if (!overlap(out, bytes, part, part_bytes)) continue;
    if (!(exact_ok && out == part && bytes == part_bytes)) return true;
  }
  return false;
}

}  // namespace sca

using namespace sca;

extern "C" int cast_bf16_to_f16(const void* src, void* dst, int64_t n, int* dev_status, void* stream) {
  SCA_REQUIRE(src && dst, SCA_ERR_ARG, "cast_bf16_to_f16: NULL pointer");
  SCA_REQUIRE(n >= 0 && n % 8 == 0, SCA_ERR_ARG, "cast_bf16_to_f16: n=%lld must be a non-negative multiple of 8",
              static_cast<long long>(n));
  SCA_REQUIRE(aligned(src, 16) && aligned(dst, 16), SCA_ERR_ALIGN, "cast_bf16_to_f16: pointers not 16-byte aligned");
  SCA_REQUIRE(!overlap(src, 2 * n, dst, 2 * n), SCA_ERR_ARG, "cast_bf16_to_f16: src and dst overlap");
  if (n == 0) return SCA_OK;
  const int64_t nvec = n / 8;
  cast_bf16_f16_kernel<<<grid_for(nvec, kCastThreads * 4), kCastThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec, dev_status);
  return cuda_status(cudaGetLastError(), "cast_bf16_to_f16 launch");
}

extern "C" int zigzag_permute(const void* src, void* dst, int64_t outer, int64_t S, int64_t row_bytes, int P,
                              int inverse, int* dev_status, void* stream) {
  SCA_REQUIRE(src && dst, SCA_ERR_ARG, "zigzag_permute: NULL pointer");
  SCA_REQUIRE(P >= 1, SCA_ERR_ARG, "zigzag_permute: P=%d must be >= 1", P);
  SCA_REQUIRE(outer >= 0 && S >= 0, SCA_ERR_ARG, "zigzag_permute: negative size");
  SCA_REQUIRE(S % (2 * P) == 0, SCA_ERR_ARG, "zigzag_permute: S=%lld not divisible by 2P=%d",
              static_cast<long long>(S), 2 * P);
  SCA_REQUIRE(row_bytes > 0 && row_bytes % 4 == 0, SCA_ERR_ARG,
              "zigzag_permute: row_bytes=%lld must be a positive multiple of 4",
              static_cast<long long>(row_bytes));
  SCA_REQUIRE(aligned(src, 4) && aligned(dst, 4), SCA_ERR_ALIGN, "zigzag_permute: pointers not 4-byte aligned");
  const int64_t total = outer * S * row_bytes;
  SCA_REQUIRE(!overlap(src, total, dst, total), SCA_ERR_ARG, "zigzag_permute: src and dst overlap");
  if (total == 0) return SCA_OK;
  const int64_t chunk_bytes = (S / (2 * P)) * row_bytes;
  const int64_t nseg = outer * 2 * P;
  const bool vec16 = chunk_bytes % 16 == 0 && aligned(src, 16) && aligned(dst, 16);
  cudaStream_t st = as_stream(stream);
  if (vec16) {   // bulk copies through shared memory
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
      std::lock_guard<std::mutex> g(mu);
      if (!attr_set[dev]) {
        const cudaError_t e =
            cudaFuncSetAttribute(zigzag_permute_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkSmem);
        if (e != cudaSuccess) return cuda_status(e, "zigzag_permute attribute");
        attr_set[dev] = true;
      }
      const int64_t ppc = (chunk_bytes + kBulkPiece - 1) / kBulkPiece;
      const int64_t n_pieces = nseg * ppc;
      const int64_t blocks = static_cast<int64_t>(sm_count()) * 2;
      const unsigned grid = static_cast<unsigned>(n_pieces < blocks ? n_pieces : blocks);
      zigzag_permute_bulk_kernel<<<grid, 32, kBulkSmem, st>>>(static_cast<const uint8_t*>(src),
                                                              static_cast<uint8_t*>(dst), nseg, chunk_bytes, ppc, P,
                                                              inverse, dev_status);
      return cuda_status(cudaGetLastError(), "zigzag_permute launch");
    }
  }
  const int64_t vsz = vec16 ? 16 : 4;
  const int64_t chunk_vecs = chunk_bytes / vsz;
  const int64_t tile = static_cast<int64_t>(kPermThreads) * kPermUnroll;
  const int64_t tiles_per_chunk = (chunk_vecs + tile - 1) / tile;
  // one wave: 2048 resident threads per SM at 256 per block
  const int64_t resident = static_cast<int64_t>(sm_count()) * (2048 / kPermThreads);
  const int64_t n_tiles = nseg * tiles_per_chunk;
  const unsigned grid = static_cast<unsigned>(n_tiles < resident ? n_tiles : resident);
  if (vec16)
    zigzag_permute_kernel<uint4><<<grid, kPermThreads, 0, st>>>(static_cast<const uint4*>(src),
                                                                static_cast<uint4*>(dst), nseg, chunk_vecs,
                                                                tiles_per_chunk, P, inverse);
  else
    zigzag_permute_kernel<uint32_t><<<grid, kPermThreads, 0, st>>>(static_cast<const uint32_t*>(src),
                                                                   static_cast<uint32_t*>(dst), nseg,
                                                                   chunk_vecs, tiles_per_chunk, P, inverse);
  return cuda_status(cudaGetLastError(), "zigzag_permute launch");
}

// Launches the copy kernel over copies [0, n) (n <= SCA_MAX_COPIES, every
// address, width and pitch a multiple of 16 bytes, checked by the caller).
static int launch_copies(const sca_copy* copies, int n, cudaStream_t st, const char* what) {
  CopyBatch cb;
  int64_t units = 0;
  cb.n = 0;
  for (int i = 0; i < n; ++i) {
    if (copies[i].height == 0 || copies[i].width == 0) continue;
    CopyJob& j = cb.job[cb.n++];
    j.src = static_cast<const uint4*>(copies[i].src);
    j.dst = static_cast<uint4*>(copies[i].dst);
    j.spitch = copies[i].src_pitch / 16;
    j.dpitch = copies[i].dst_pitch / 16;
    j.height = static_cast<int32_t>(copies[i].height);
    j.width = static_cast<int32_t>(copies[i].width / 16);
    j.slices = (j.width + kCopySlice - 1) / kCopySlice;
    j.units_before = static_cast<int32_t>(units);
    units += static_cast<int64_t>(j.height) * j.slices;
  }
  if (cb.n == 0) return SCA_OK;
  SCA_REQUIRE(units < (int64_t(1) << 31), SCA_ERR_UNSUPPORTED, "%s: copy too large for one launch", what);
  cb.units = static_cast<int32_t>(units);
  const int64_t blocks = static_cast<int64_t>(kCopyBlocksPerSm) * sm_count();
  const int grid = static_cast<int>(units < blocks ? units : blocks);
  ring_copy_kernel<<<grid, kCopyThreads, 0, st>>>(cb);
  return cuda_status(cudaGetLastError(), what);
}

static bool copy_ok(const sca_copy& c) {
  return c.height >= 0 && c.width >= 0 && c.width % 16 == 0 && c.src_pitch % 16 == 0 && c.dst_pitch % 16 == 0 &&
         c.width / 16 < (int64_t(1) << 31) && c.height < (int64_t(1) << 31) &&
         (c.height <= 1 || (c.src_pitch >= c.width && c.dst_pitch >= c.width));
}

// height rows of `width` bytes, pitches in bytes: the hand-off copy kernel
// when every address and size is a whole number of 16-byte vectors, else
// the runtime's 2-D copy.
static int stage_copy(void* dst, int64_t dpitch, const void* src, int64_t spitch, int64_t width, int64_t height,
                      cudaStream_t st, const char* what) {
  if (width == 0 || height == 0) return SCA_OK;
  sca_copy c;
  c.src = src;
  c.dst = dst;
  c.height = height;
  c.width = width;
  c.src_pitch = spitch;
  c.dst_pitch = dpitch;
  if (aligned(src, 16) && aligned(dst, 16) && copy_ok(c)) return launch_copies(&c, 1, st, what);
  return cuda_status(cudaMemcpy2DAsync(dst, static_cast<size_t>(dpitch), src, static_cast<size_t>(spitch),
                                       static_cast<size_t>(width), static_cast<size_t>(height),
                                       cudaMemcpyDeviceToDevice, st),
                     what);
}

extern "C" int ring_stage_block(const void* src, void* dst, int64_t outer, int64_t S_src, int64_t row0,
                                int64_t rows, int64_t row_bytes, void* stream) {
  SCA_REQUIRE(src && dst, SCA_ERR_ARG, "ring_stage_block: NULL pointer");
  SCA_REQUIRE(outer >= 0 && rows >= 0 && row_bytes > 0 && row0 >= 0 && row0 + rows <= S_src, SCA_ERR_ARG,
              "ring_stage_block: rows [%lld, %lld) outside [0, %lld)", static_cast<long long>(row0),
              static_cast<long long>(row0 + rows), static_cast<long long>(S_src));
  if (outer == 0 || rows == 0) return SCA_OK;
  const char* s = static_cast<const char*>(src) + row0 * row_bytes;
  return stage_copy(dst, rows * row_bytes, s, S_src * row_bytes, rows * row_bytes, outer, as_stream(stream),
                    "ring_stage_block copy");
}

extern "C" int ring_stage_segments(const void* src, void* dst, int64_t outer, int64_t S_src, const sca_segs* seg,
                                   int64_t row_bytes, void* stream) {
  SCA_REQUIRE(src && dst && seg, SCA_ERR_ARG, "ring_stage_segments: NULL pointer");
  SCA_REQUIRE(seg->n == 1 || seg->n == 2, SCA_ERR_ARG, "ring_stage_segments: seg->n=%d must be 1 or 2", seg->n);
  SCA_REQUIRE(outer >= 0 && seg->len >= 0 && row_bytes > 0, SCA_ERR_ARG, "ring_stage_segments: negative size");
  for (int i = 0; i < seg->n; ++i)
    SCA_REQUIRE(seg->start[i] >= 0 && seg->start[i] + seg->len <= S_src, SCA_ERR_ARG,
                "ring_stage_segments: segment %d rows [%lld, %lld) outside [0, %lld)", i,
                static_cast<long long>(seg->start[i]), static_cast<long long>(seg->start[i] + seg->len),
                static_cast<long long>(S_src));
  if (outer == 0 || seg->len == 0) return SCA_OK;
  const size_t width = static_cast<size_t>(seg->len * row_bytes);
  const size_t dpitch = static_cast<size_t>(seg->n) * width;
  SCA_REQUIRE(!overlap(src, outer * S_src * row_bytes,
                       dst, outer * static_cast<int64_t>(dpitch)),
              SCA_ERR_ARG, "ring_stage_segments: src and dst overlap");
  for (int i = 0; i < seg->n; ++i) {
    const char* s = static_cast<const char*>(src) + seg->start[i] * row_bytes;
    const int rc = stage_copy(static_cast<char*>(dst) + i * width, static_cast<int64_t>(dpitch), s,
                              S_src * row_bytes, static_cast<int64_t>(width), outer, as_stream(stream),
                              "ring_stage_segments copy");
    if (rc != SCA_OK) return rc;
  }
  return SCA_OK;
}

extern "C" int ring_stage_copies(const sca_copy* copies, int n, void* stream) {
  SCA_REQUIRE(n >= 0 && n <= SCA_MAX_COPIES, SCA_ERR_ARG, "ring_stage_copies: n=%d outside [0, %d]", n,
              SCA_MAX_COPIES);
  SCA_REQUIRE(n == 0 || copies, SCA_ERR_ARG, "ring_stage_copies: NULL copies");
  for (int i = 0; i < n; ++i) {
    const sca_copy& c = copies[i];
    SCA_REQUIRE(c.src && c.dst, SCA_ERR_ARG, "ring_stage_copies: copy %d has a NULL pointer", i);
    SCA_REQUIRE(copy_ok(c), SCA_ERR_ARG,
                "ring_stage_copies: copy %d: sizes must be non-negative, width and pitches multiples of 16 bytes, "
                "pitches at least the width",
                i);
    SCA_REQUIRE(aligned(c.src, 16) && aligned(c.dst, 16), SCA_ERR_ALIGN,
                "ring_stage_copies: copy %d: pointers not 16-byte aligned", i);
    const int64_t sb = c.height == 0 ? 0 : (c.height - 1) * c.src_pitch + c.width;
    const int64_t db = c.height == 0 ? 0 : (c.height - 1) * c.dst_pitch + c.width;
    SCA_REQUIRE(!overlap(c.src, sb, c.dst, db), SCA_ERR_ARG, "ring_stage_copies: copy %d: src and dst overlap", i);
  }
  return launch_copies(copies, n, as_stream(stream), "ring_stage_copies launch");
}

extern "C" int attn_merge_lse(const float* o_parts, const float* lse_parts, int n, int64_t rows, int D,
                              int64_t o_part_stride, int64_t lse_part_stride, float* o_out, float* lse_out,
                              void* o_bf16_out, int unpermute_P, int64_t S, void* stream) {
  SCA_REQUIRE(o_parts && lse_parts && o_out && lse_out, SCA_ERR_ARG, "attn_merge_lse: NULL pointer");
  SCA_REQUIRE(n >= 1 && n <= 64, SCA_ERR_ARG, "attn_merge_lse: n=%d outside [1, 64]", n);
  SCA_REQUIRE(rows >= 0, SCA_ERR_ARG, "attn_merge_lse: rows < 0");
  SCA_REQUIRE(D == 4 || D == 8 || D == 16 || D == 32 || D == 64 || D == 128, SCA_ERR_ARG,
              "attn_merge_lse: D=%d must be one of 4, 8, 16, 32, 64, 128", D);
  SCA_REQUIRE(o_part_stride >= rows * D && lse_part_stride >= rows, SCA_ERR_ARG,
              "attn_merge_lse: partial strides smaller than one partial");
  SCA_REQUIRE(o_part_stride % 4 == 0, SCA_ERR_ALIGN, "attn_merge_lse: o_part_stride not a multiple of 4");
  SCA_REQUIRE(aligned(o_parts, 16) && aligned(o_out, 16) && aligned(o_bf16_out, 8), SCA_ERR_ALIGN,
              "attn_merge_lse: o pointers must be 16-byte aligned (bf16 copy 8-byte)");
  if (unpermute_P > 0)
    SCA_REQUIRE(S > 0 && S % (2 * unpermute_P) == 0 && rows % S == 0, SCA_ERR_ARG,
                "attn_merge_lse: unpermute needs S %% 2P == 0 and rows %% S == 0");
  {
    // An output may be exactly one partial's rows when rows keep their
    // places (no unpermute): every element is then read by the lanes that
    // write it.  Any other overlap with an input, or between outputs, races.
    const bool exact_ok = unpermute_P == 0;
    const int64_t ob = rows * D * 4, lb = rows * 4;
    SCA_REQUIRE(!bad_overlap(o_out, ob, o_parts, o_part_stride * 4, n, ob, exact_ok) &&
                    !bad_overlap(o_out, ob, lse_parts, lse_part_stride * 4, n, lb, false) &&
                    !bad_overlap(lse_out, lb, lse_parts, lse_part_stride * 4, n, lb, exact_ok) &&
                    !bad_overlap(lse_out, lb, o_parts, o_part_stride * 4, n, ob, false) && !overlap(o_out, ob, lse_out, lb),
                SCA_ERR_ARG,
                exact_ok ? "attn_merge_lse: an output overlaps an input other than by being one partial's rows exactly"
                         : "attn_merge_lse: outputs may not overlap inputs when unpermuting");
    if (o_bf16_out) {
      const int64_t bb = rows * D * 2;
      SCA_REQUIRE(!bad_overlap(o_bf16_out, bb, o_parts, o_part_stride * 4, n, ob, false) &&
                      !bad_overlap(o_bf16_out, bb, lse_parts, lse_part_stride * 4, n, lb, false) &&
                      !overlap(o_bf16_out, bb, o_out, ob) && !overlap(o_bf16_out, bb, lse_out, lb),
                  SCA_ERR_ARG, "attn_merge_lse: o_bf16_out overlaps another buffer");
    }
  }
  if (rows == 0) return SCA_OK;
  const int L = D / 4;
  const int64_t warps = (rows + (32 / L) - 1) / (32 / L);
  const int grid = grid_for(warps * 32, kMergeThreads);
  cudaStream_t st = as_stream(stream);
  auto* ob = static_cast<__nv_bfloat16*>(o_bf16_out);
#define SCA_MERGE_CASE(LL)                                                                               \
  case LL:                                                                                               \
    if (n <= 4)                                                                                          \
      merge_lse_kernel<LL, 4><<<grid, kMergeThreads, 0, st>>>(o_parts, lse_parts, n, rows, o_part_stride,  \
                                                              lse_part_stride, o_out, lse_out, ob,        \
                                                              unpermute_P, S);                             \
    else                                                                                                 \
      merge_lse_kernel<LL, kMergeMaxFast><<<grid, kMergeThreads, 0, st>>>(                                \
          o_parts, lse_parts, n, rows, o_part_stride, lse_part_stride, o_out, lse_out, ob, unpermute_P, S); \
    break;
  switch (L) {
    SCA_MERGE_CASE(1)
    SCA_MERGE_CASE(2)
    SCA_MERGE_CASE(4)
    SCA_MERGE_CASE(8)
    SCA_MERGE_CASE(16)
    SCA_MERGE_CASE(32)
  }
#undef SCA_MERGE_CASE
  return cuda_status(cudaGetLastError(), "attn_merge_lse launch");
}

extern "C" int attn_bwd_delta(const float* o, const void* dout, int dout_dtype, float* delta, int64_t rows,
                              int D, void* stream) {
  SCA_REQUIRE(o && dout && delta, SCA_ERR_ARG, "attn_bwd_delta: NULL pointer");
  SCA_REQUIRE(rows >= 0, SCA_ERR_ARG, "attn_bwd_delta: rows < 0");
  SCA_REQUIRE(D == 64 || D == 128, SCA_ERR_UNSUPPORTED, "attn_bwd_delta: D=%d not in {64, 128}", D);
  SCA_REQUIRE(dout_dtype == SCA_BF16 || dout_dtype == SCA_F32, SCA_ERR_ARG, "attn_bwd_delta: bad dtype");
  SCA_REQUIRE(aligned(o, 16) && aligned(dout, 8), SCA_ERR_ALIGN, "attn_bwd_delta: misaligned pointer");
  if (rows == 0) return SCA_OK;
  const int L = D / 4;
  const int64_t warps = (rows + (32 / L) - 1) / (32 / L);
  const int grid = grid_for(warps * 32, kMergeThreads);
  cudaStream_t st = as_stream(stream);
  if (dout_dtype == SCA_BF16) {
    if (L == 32)
      delta_kernel<32, __nv_bfloat16><<<grid, kMergeThreads, 0, st>>>(
          o, static_cast<const __nv_bfloat16*>(dout), delta, rows);
    else
      delta_kernel<16, __nv_bfloat16><<<grid, kMergeThreads, 0, st>>>(
          o, static_cast<const __nv_bfloat16*>(dout), delta, rows);
  } else {
    if (L == 32)
      delta_kernel<32, float><<<grid, kMergeThreads, 0, st>>>(o, static_cast<const float*>(dout), delta, rows);
    else
      delta_kernel<16, float><<<grid, kMergeThreads, 0, st>>>(o, static_cast<const float*>(dout), delta, rows);
  }
  return cuda_status(cudaGetLastError(), "attn_bwd_delta launch");
}
