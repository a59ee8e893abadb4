// Causal linear attention over P contiguous shards on the tensor cores
// (linear attention sequence parallelism: "Effiziente Parallelisierung
// linearer Aufmerksamkeitssequenzen fuer skalierbare Sprachmodelle" -
// intermediate states passed point to point between shards, the
// right-product trick).  bf16 inputs, D = 128, blocks of kBlk = 128 rows.
//
// The same block algebra as the CUDA-core kernels of lasp.cu, with every
// product on tcgen05 (kind::f16, fp32 accumulation in tensor memory):
//
//   states:  st_j = A_j^T B_j                    (k^T v, or q^T dO backward)
//   forward: o_j  = scale (q_j F + tril(q_j k_j^T) v_j)
//   dq_j = scale (dO_j F^T + tril(dO_j v_j^T) k_j)
//   dk_j = scale (v_j G^T + tril(dO_j v_j^T)^T q_j)
//   dv_j = scale (k_j G + tril(q_j k_j^T)^T dO_j)
//
// with F, G the fp32 states before / after the block.  Two operands are not
// bf16 inputs: the state (fp32, entries up to ~sqrt(S)) and the masked
// block product (fp32).  Each is split as x = hi + lo with hi = bf16(x) and
// lo = bf16(x - hi) (error below 2^-16 |x|) and multiplied twice, so every
// product keeps about fp32 accuracy.
//
// Each kernel computes the TRANSPOSE of its output block, out^T[a][r]
// (feature a in tensor-memory lane, block row r in column): the epilogue
// then writes, for every block row, 32 consecutive features per warp
// (128-byte stores), and every operand is a natural tile:
//
//   M[s][t] = x_s . y_t  (t >= s, else 0): A = X (K-major), B = Y (K-major)
//   out^T   = A1 B1 + Z^T M-or-M^T
//
//   kernel  X  Y   Z   state term A1 (tile = state, row-major)  B1   mask as B
//   fwd     k  q   v   F[b][a]: MN-major                         q    MN-major (k = s)
//   dq      v  dO  k   F[a][b]: K-major                          dO   MN-major (k = s)
//   dk      v  dO  q   G[a][b]: K-major                          v    K-major  (k = t)
//   dv      k  q   dO  G[b][a]: MN-major                         k    K-major  (k = t)
//
// Shared-memory tiles are [128 rows][128 bf16] as two 128-byte-swizzled
// panels of 64 columns (the layout TMA writes); the state and the mask are
// written there by the threads in the same layout.
#include <cuda.h>

#include "common.cuh"
#include "host_common.h"
#include "lasp_tc.h"
#include "ptx.cuh"
#include "tmap.h"

namespace sca {
namespace lasp_tc {

constexpr int kBlk = 128;
constexpr int kD = 128;
constexpr int PANEL = 128 * 128;      // 128 rows x 64 bf16
constexpr int TILE = 2 * PANEL;       // 128 x 128 bf16
constexpr int kThreads = 256;

SCA_INLINE void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// byte offset of the 16-byte chunk with columns [8c, 8c + 8) of `row`
SCA_INLINE uint32_t chunk_off(int row, int c) {
  return (c >> 3) * PANEL + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// operand descriptors of k-step kk (16 elements of the contraction)
SCA_INLINE uint64_t kmajor(uint32_t base, int kk) {   // tile rows = M or N, K along the row
  return sdesc_sw128(base + (kk >> 2) * PANEL + (kk & 3) * 32, 16, 1024);
}
SCA_INLINE uint64_t mnmajor(uint32_t base, int kk) {  // tile rows = K, M or N along the row
  return sdesc_sw128(base + kk * 2048, PANEL, 1024);
}

// x = hi + lo, both bf16 (round to nearest even), for 8 values
SCA_INLINE void split8(const float* x, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    const float2 hf = __bfloat1622float2(hv);
    const __nv_bfloat162 lv = __floats2bfloat162_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y);
    h[i] = *reinterpret_cast<const uint32_t*>(&hv);
    l[i] = *reinterpret_cast<const uint32_t*>(&lv);
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

struct Bars {
  uint64_t in_full, mask_done, t1_done, t2_done;
  uint32_t tmem_base;
  int abort;
};

// Kernel arguments: X, Y, Z tile maps ([BH, S, D] bf16 views), the block
// states and shard inputs, the output.
struct Args {
  CUtensorMap mx, my, mz;
  const float* st;     // [BH, S/kBlk, D, D]
  const float* shard_in;   // [BH, P, D, D]
  float* out;          // [BH, S, D]
  int64_t S;
  int P;
  float scale;
  int* status;
};

enum Mode { kFwd = 0, kDq = 1, kDk = 2, kDv = 3 };

constexpr int X_OFF = 0, Y_OFF = TILE, Z_OFF = 2 * TILE, W0_OFF = 3 * TILE, W1_OFF = 4 * TILE, BAR_OFF = 5 * TILE;
constexpr int kSmem = BAR_OFF + 1024 + 1024;   // bars, alignment slack

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) block_kernel(const __grid_constant__ Args a) {
  constexpr bool kStateMN = MODE == kFwd || MODE == kDv;   // A1 = state, MN-major (else K-major)
  constexpr bool kB1isY = MODE == kFwd || MODE == kDq;     // B1 = Y (else X)
  constexpr bool kMaskMN = MODE == kFwd || MODE == kDq;    // mask as B: MN-major (else K-major)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + BAR_OFF);
  const int j = blockIdx.x, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nblk = a.S / kBlk;
  const int r = static_cast<int>(j / (nblk / a.P));
  const int row0 = j * kBlk;

  if (threadIdx.x == 0) {
    mbar_init(&bars->in_full, 1);
    mbar_init(&bars->mask_done, 1);
    mbar_init(&bars->t1_done, 1);
    mbar_init(&bars->t2_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tM = bars->tmem_base, tO = tM + 128;
  volatile int* abort = &bars->abort;
  const uint32_t sX = smem_u32(smem + X_OFF), sY = smem_u32(smem + Y_OFF), sZ = smem_u32(smem + Z_OFF);
  const uint32_t sW0 = smem_u32(smem + W0_OFF), sW1 = smem_u32(smem + W1_OFF);

  if (threadIdx.x == 0) {
    tma_prefetch_map(&a.mx);
    tma_prefetch_map(&a.my);
    tma_prefetch_map(&a.mz);
    mbar_arrive_expect_tx(&bars->in_full, 3 * TILE);
    for (int p = 0; p < 2; ++p) {
      tma_load_4d(smem + X_OFF + p * PANEL, &a.mx, &bars->in_full, 64 * p, row0, bh, 0);
      tma_load_4d(smem + Y_OFF + p * PANEL, &a.my, &bars->in_full, 64 * p, row0, bh, 0);
      tma_load_4d(smem + Z_OFF + p * PANEL, &a.mz, &bars->in_full, 64 * p, row0, bh, 0);
    }
  }

  // the state st[j] + sin[r] into W0 (hi) and W1 (lo), row-major: 16
  // threads per row, 8 columns each (coalesced 512-byte rows)
  {
    const float* s0 = a.st + (static_cast<int64_t>(bh) * nblk + j) * kD * kD;
    const float* s1 = a.shard_in + (static_cast<int64_t>(bh) * a.P + r) * kD * kD;
    const int c = threadIdx.x & 15;
#pragma unroll 2
    for (int row = threadIdx.x >> 4; row < kD; row += kThreads / 16) {
      const float4* p0 = reinterpret_cast<const float4*>(s0 + row * kD + 8 * c);
      const float4* p1 = reinterpret_cast<const float4*>(s1 + row * kD + 8 * c);
      const float4 u0 = p0[0], u1 = p0[1], v0 = p1[0], v1 = p1[1];
      const float x[8] = {u0.x + v0.x, u0.y + v0.y, u0.z + v0.z, u0.w + v0.w,
                          u1.x + v1.x, u1.y + v1.y, u1.z + v1.z, u1.w + v1.w};
      uint4 hi, lo;
      split8(x, hi, lo);
      *reinterpret_cast<uint4*>(smem + W0_OFF + chunk_off(row, c)) = hi;
      *reinterpret_cast<uint4*>(smem + W1_OFF + chunk_off(row, c)) = lo;
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();

  bool ok = true;
  int issued = 0;   // MMA groups committed by thread 0 (for the abort drain)
  if (threadIdx.x == 0) {
    tc_fence_after();
    ok = mbar_wait(&bars->in_full, 0, abort, a.status);
    if (ok) {
      constexpr uint32_t id_m = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_1 = idesc_bf16_f32(128, 128, kStateMN, false);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) umma_ss(tM, kmajor(sX, kk), kmajor(sY, kk), id_m, kk > 0 ? 1u : 0u);
      umma_commit(&bars->mask_done);
      const uint32_t sB1 = kB1isY ? sY : sX;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t b1 = kmajor(sB1, kk);
        umma_ss(tO, kStateMN ? mnmajor(sW0, kk) : kmajor(sW0, kk), b1, id_1, kk > 0 ? 1u : 0u);
        umma_ss(tO, kStateMN ? mnmajor(sW1, kk) : kmajor(sW1, kk), b1, id_1, 1u);
      }
      umma_commit(&bars->t1_done);
      issued = 2;
    }
  }

  // the masked block product M[s][t] (t >= s) into W0/W1 (hi, lo) once the
  // state products have read them: warp w reads lanes 32 (w & 3) .. + 31
  // (rows s) and columns 64 (w >> 2) .. + 63 (t)
  const int q4 = warp & 3, half = warp >> 2;
  const int lrow = q4 * 32 + lane;
  const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
  // (every thread takes part in each vote; a failed wait has set *abort,
  // so the later waits return at once)
  ok = __all_sync(0xffffffffu, mbar_wait(&bars->mask_done, 0, abort, a.status) && ok);
  ok = __all_sync(0xffffffffu, mbar_wait(&bars->t1_done, 0, abort, a.status) && ok);
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      tmem_ld32(tM + lane_off + 64 * half + 32 * cc, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int t = 64 * half + 32 * cc + 8 * u + i;
          x[i] = t >= lrow ? __uint_as_float(v[8 * u + i]) : 0.f;
        }
        uint4 hi, lo;
        split8(x, hi, lo);
        const int c = 8 * half + 4 * cc + u;
        *reinterpret_cast<uint4*>(smem + W0_OFF + chunk_off(lrow, c)) = hi;
        *reinterpret_cast<uint4*>(smem + W1_OFF + chunk_off(lrow, c)) = lo;
      }
    }
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  ok = ok && !*abort;
  if (threadIdx.x == 0 && ok) {
    tc_fence_after();
    constexpr uint32_t id_2 = idesc_bf16_f32(128, 128, true, kMaskMN);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t a2 = mnmajor(sZ, kk);
      umma_ss(tO, a2, kMaskMN ? mnmajor(sW0, kk) : kmajor(sW0, kk), id_2, 1u);
      umma_ss(tO, a2, kMaskMN ? mnmajor(sW1, kk) : kmajor(sW1, kk), id_2, 1u);
    }
    umma_commit(&bars->t2_done);
    issued = 3;
  }

  // out[row0 + r][a] = scale * out^T[a][r]: lanes are features, so each
  // store instruction writes 32 consecutive floats of one row
  ok = __all_sync(0xffffffffu, mbar_wait(&bars->t2_done, 0, abort, a.status) && ok);
  if (ok) {
    tc_fence_after();
    float* out = a.out + (static_cast<int64_t>(bh) * a.S + row0) * kD + lrow;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t v[32];
      tmem_ld32(tO + lane_off + 64 * half + 32 * cc, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) out[(64 * half + 32 * cc + i) * kD] = a.scale * __uint_as_float(v[i]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {   // let issued copies and MMAs finish before the memory goes
    mbar_wait_drain(&bars->in_full, 0);
    if (issued >= 2) mbar_wait_drain(&bars->t1_done, 0);
    if (issued >= 3) mbar_wait_drain(&bars->t2_done, 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tM, 256);
  }
}

// st[bh][j] = A_j^T B_j: computed transposed, D^T[m = b-feature][n =
// a-feature] with both tiles MN-major (rows = the contraction), so that the
// epilogue writes 32 consecutive floats of a state row per store.
struct StArgs {
  CUtensorMap ma, mb;
  float* st;
  int64_t S;
  int* status;
};

constexpr int kStSmem = 2 * TILE + 1024 + 1024;

__global__ void __launch_bounds__(128, 1) states_kernel(const __grid_constant__ StArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + 2 * TILE);
  const int j = blockIdx.x, bh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars->in_full, 1);
    mbar_init(&bars->t1_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tD = bars->tmem_base;
  volatile int* abort = &bars->abort;
  bool ok = true;
  int issued = 0;
  if (threadIdx.x == 0) {
    tma_prefetch_map(&a.ma);
    tma_prefetch_map(&a.mb);
    mbar_arrive_expect_tx(&bars->in_full, 2 * TILE);
    for (int p = 0; p < 2; ++p) {
      tma_load_4d(smem + p * PANEL, &a.ma, &bars->in_full, 64 * p, j * kBlk, bh, 0);
      tma_load_4d(smem + TILE + p * PANEL, &a.mb, &bars->in_full, 64 * p, j * kBlk, bh, 0);
    }
    ok = mbar_wait(&bars->in_full, 0, abort, a.status);
    if (ok) {
      tc_fence_after();
      const uint32_t sA = smem_u32(smem), sB = smem_u32(smem + TILE);
      constexpr uint32_t id = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) umma_ss(tD, mnmajor(sB, kk), mnmajor(sA, kk), id, kk > 0 ? 1u : 0u);
      umma_commit(&bars->t1_done);
      issued = 1;
    }
  }
  ok = __all_sync(0xffffffffu, mbar_wait(&bars->t1_done, 0, abort, a.status));
  if (ok) {
    tc_fence_after();
    const int jb = warp * 32 + lane;   // b-feature (lane)
    float* st = a.st + (static_cast<int64_t>(bh) * (a.S / kBlk) + j) * kD * kD + jb;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      tmem_ld32(tD + lane_off + 32 * cc, v);
      tmem_wait_ld32(v);
#pragma unroll
      for (int i = 0; i < 32; ++i) st[(32 * cc + i) * kD] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) {
    mbar_wait_drain(&bars->in_full, 0);
    if (issued) mbar_wait_drain(&bars->t1_done, 0);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tD, 128);
  }
}

// [BH, S, 128] bf16 tensor as a TMA map with 64 x 128 boxes
static cudaError_t map_of(CUtensorMap* m, const void* p, int64_t BH, int64_t S) {
  View v;
  v.s = kD;
  v.h = S * kD;
  v.b = BH * S * kD;
  return make_tmap_bf16(m, p, kD, S, static_cast<int>(BH), 1, v, 64, kBlk);
}

template <typename K>
static cudaError_t allow(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace lasp_tc

using namespace lasp_tc;

int lasp_tc_states(const void* a, const void* b, float* st, int64_t BH, int64_t S, int* status,
                   cudaStream_t stream) {
  StArgs sa;
  cudaError_t e = map_of(&sa.ma, a, BH, S);
  if (e == cudaSuccess) e = map_of(&sa.mb, b, BH, S);
  SCA_REQUIRE(e == cudaSuccess, SCA_ERR_ALIGN, "lasp_block_states: inputs are not TMA-addressable (16-byte base)");
  sa.st = st;
  sa.S = S;
  sa.status = status;
  if ((e = allow(states_kernel, kStSmem)) != cudaSuccess) return cuda_status(e, "lasp_block_states");
  states_kernel<<<dim3(static_cast<unsigned>(S / kBlk), static_cast<unsigned>(BH)), 128, kStSmem, stream>>>(sa);
  return cuda_status(cudaGetLastError(), "lasp_block_states launch");
}

template <int MODE>
static int launch_block(const void* x, const void* y, const void* z, const float* st, const float* shard_in, float* out,
                        int64_t BH, int64_t S, int P, float scale, int* status, cudaStream_t stream,
                        const char* who) {
  Args a;
  cudaError_t e = map_of(&a.mx, x, BH, S);
  if (e == cudaSuccess) e = map_of(&a.my, y, BH, S);
  if (e == cudaSuccess) e = map_of(&a.mz, z, BH, S);
  SCA_REQUIRE(e == cudaSuccess, SCA_ERR_ALIGN, "%s: inputs are not TMA-addressable (16-byte base)", who);
  a.st = st;
  a.shard_in = shard_in;
  a.out = out;
  a.S = S;
  a.P = P;
  a.scale = scale;
  a.status = status;
  if ((e = allow(block_kernel<MODE>, kSmem)) != cudaSuccess) return cuda_status(e, who);
  block_kernel<MODE><<<dim3(static_cast<unsigned>(S / kBlk), static_cast<unsigned>(BH)), kThreads, kSmem, stream>>>(a);
  return cuda_status(cudaGetLastError(), who);
}

int lasp_tc_fwd(const void* q, const void* k, const void* v, const float* st, const float* shard_in, float* o,
                int64_t BH, int64_t S, int P, float scale, int* status, cudaStream_t stream) {
  return launch_block<kFwd>(k, q, v, st, shard_in, o, BH, S, P, scale, status, stream, "lasp_fwd");
}

int lasp_tc_bwd(const void* q, const void* k, const void* v, const void* dout, const float* st_f, const float* in_f,
                const float* st_b, const float* in_b, float* dq, float* dk, float* dv, int64_t BH, int64_t S, int P,
                float scale, int* status, cudaStream_t stream) {
  int rc = launch_block<kDq>(v, dout, k, st_f, in_f, dq, BH, S, P, scale, status, stream, "lasp_bwd (dq)");
  if (rc == SCA_OK) rc = launch_block<kDk>(v, dout, q, st_b, in_b, dk, BH, S, P, scale, status, stream, "lasp_bwd (dk)");
  if (rc == SCA_OK) rc = launch_block<kDv>(k, q, dout, st_b, in_b, dv, BH, S, P, scale, status, stream, "lasp_bwd (dv)");
  return rc;
}

}  // namespace sca
