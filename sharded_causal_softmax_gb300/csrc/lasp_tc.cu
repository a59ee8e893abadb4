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
//   kernel  X  Y   Z   state term A1 (in tensor memory)   B1   mask as B
//   fwd     k  q   v   A1[a][b] = F[b][a]                  q    MN-major (k = s)
//   dq      v  dO  k   A1[a][b] = F[a][b]                  dO   MN-major (k = s)
//   dk      v  dO  q   A1[a][b] = G[a][b]                  v    K-major  (k = t)
//   dv      k  q   dO  A1[a][b] = G[b][a]                  k    K-major  (k = t)
//
// Shared-memory tiles are [128 rows][128 bf16] as two 128-byte-swizzled
// panels of 64 columns (the layout TMA writes); the masked product is
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
  const float* st;         // [BH, S/kBlk, D, D]
  const float* shard_in;   // [BH, P, D, D]
  float* out;              // [BH, S, D]
  int64_t S;
  int BH;
  int P;
  float scale;
  int* status;
};

enum Mode { kFwd = 0, kDq = 1, kDk = 2, kDv = 3 };

// Persistent, pipelined block kernel: one CTA per SM walks blocks n =
// blockIdx.x, + gridDim.x, ...  Roles: warp 8 loads X, Y, Z by TMA into two
// shared-memory stages; one thread of warp 9 issues the MMAs; warps 0-7 put
// each block's state into tensor memory (the A operand of the state term),
// turn the masked product into shared-memory operands and write the output.
// Tensor memory (512 columns): M (128), two output accumulators (2 x 128),
// the state's hi and lo parts (64 + 64, bf16 pairs).  Shared memory: two
// stages of X, Y, Z; the masked product's hi and lo parts overwrite X and Y
// of their stage once the products that read them are done.
constexpr int kPThreads = 320;
constexpr int kConv = 256;                  // converter / epilogue threads (warps 0-7)
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int STAGE = 3 * TILE;             // X, Y, Z
constexpr int P_BAR_OFF = 2 * STAGE;
constexpr int kSmem = P_BAR_OFF + 1024 + 1024;

struct PBars {
  uint64_t in_full[2], stage_free[2];
  uint64_t mask_full, tm_free, state_full, t1_done, m_full;
  uint64_t o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// The block's state (st[j] + shard_in[r]) as the A operand in tensor memory:
// lane a holds A[a][b] for b in [64 half, 64 half + 64) as bf16 pairs, hi
// and lo parts.  ROWWISE: A[a][b] = state[a][b] (a row per thread, 16-byte
// loads); else A[a][b] = state[b][a] (a column per thread; each load
// instruction reads 32 consecutive floats of one row).
template <bool ROWWISE>
SCA_INLINE void load_state(const float* st, const float* sin, uint32_t t_hi, uint32_t t_lo, int a, int half) {
  float x[64];
  if (ROWWISE) {
    const float4* p = reinterpret_cast<const float4*>(st + a * kD + 64 * half);
    const float4* q = reinterpret_cast<const float4*>(sin + a * kD + 64 * half);
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const float4 s4 = p[u], i4 = q[u];
      x[4 * u] = s4.x + i4.x;
      x[4 * u + 1] = s4.y + i4.y;
      x[4 * u + 2] = s4.z + i4.z;
      x[4 * u + 3] = s4.w + i4.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < 64; ++u) x[u] = st[(64 * half + u) * kD + a] + sin[(64 * half + u) * kD + a];
  }
  uint32_t hi[32], lo[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * c], x[2 * c + 1]);
    const float2 hf = __bfloat1622float2(hv);
    const __nv_bfloat162 lv = __floats2bfloat162_rn(x[2 * c] - hf.x, x[2 * c + 1] - hf.y);
    hi[c] = *reinterpret_cast<const uint32_t*>(&hv);
    lo[c] = *reinterpret_cast<const uint32_t*>(&lv);
  }
  tmem_st32(t_hi + 32 * half, hi);
  tmem_st32(t_lo + 32 * half, lo);
  tmem_wait_st();
}

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1) block_kernel(const __grid_constant__ Args a) {
  constexpr bool kRowwise = MODE == kDq || MODE == kDk;   // state term A = state (else its transpose)
  constexpr bool kB1isY = MODE == kFwd || MODE == kDq;    // B1 = Y (else X)
  constexpr bool kMaskMN = MODE == kFwd || MODE == kDq;   // mask as B: MN-major (else K-major)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  PBars* bars = reinterpret_cast<PBars*>(smem + P_BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nblk = a.S / kBlk;
  const int64_t total = static_cast<int64_t>(a.BH) * nblk;
  const int64_t per_shard = nblk / a.P;
  // local block i of this CTA -> global block n
  auto block_of = [&](int i) { return static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * gridDim.x; };
  int n_local = 0;
  if (blockIdx.x < total) n_local = static_cast<int>((total - 1 - blockIdx.x) / gridDim.x) + 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->in_full[i], 1);
      mbar_init(&bars->stage_free[i], 1);
      mbar_init(&bars->o_full[i], 1);
      mbar_init(&bars->o_free[i], kConv);
    }
    mbar_init(&bars->mask_full, 1);
    mbar_init(&bars->tm_free, kConv);
    mbar_init(&bars->state_full, kConv);
    mbar_init(&bars->t1_done, 1);
    mbar_init(&bars->m_full, kConv);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tM = tmem, tO0 = tmem + 128, tA_hi = tmem + 384, tA_lo = tmem + 448;
  volatile int* abort = &bars->abort;
  int* status = a.status;
  const uint32_t s0 = smem_u32(smem);

  if (warp == kProdWarp) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_map(&a.mx);
      tma_prefetch_map(&a.my);
      tma_prefetch_map(&a.mz);
      int i = 0;
      for (; i < n_local; ++i) {
        const int s = i & 1;
        if (i >= 2 && !mbar_wait(&bars->stage_free[s], ((i >> 1) + 1) & 1, abort, status)) break;
        const int64_t n = block_of(i);
        const int bh = static_cast<int>(n / nblk), row0 = static_cast<int>((n % nblk) * kBlk);
        uint8_t* st = smem + s * STAGE;
        mbar_arrive_expect_tx(&bars->in_full[s], 3 * TILE);
        for (int p = 0; p < 2; ++p) {
          tma_load_4d(st + p * PANEL, &a.mx, &bars->in_full[s], 64 * p, row0, bh, 0);
          tma_load_4d(st + TILE + p * PANEL, &a.my, &bars->in_full[s], 64 * p, row0, bh, 0);
          tma_load_4d(st + 2 * TILE + p * PANEL, &a.mz, &bars->in_full[s], 64 * p, row0, bh, 0);
        }
      }
      if (*abort)   // let the copies in flight land before the CTA goes away
        for (int j = (i > 2 ? i - 2 : 0); j < i; ++j) mbar_wait_drain(&bars->in_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_m = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_1 = idesc_bf16_f32(128, 128, false, false);   // A (state) from tensor memory
      constexpr uint32_t id_2 = idesc_bf16_f32(128, 128, true, kMaskMN);
      for (int i = 0; i < n_local; ++i) {
        const int s = i & 1;
        const uint32_t sX = s0 + s * STAGE, sY = sX + TILE, sZ = sX + 2 * TILE;
        const uint32_t tO = tO0 + 128 * s;
        if (!mbar_wait(&bars->in_full[s], (i >> 1) & 1, abort, status)) break;
        if (i >= 1 && !mbar_wait(&bars->tm_free, (i - 1) & 1, abort, status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) umma_ss(tM, kmajor(sX, kk), kmajor(sY, kk), id_m, kk > 0 ? 1u : 0u);
        umma_commit(&bars->mask_full);
        if (!mbar_wait(&bars->state_full, i & 1, abort, status)) break;
        if (i >= 2 && !mbar_wait(&bars->o_free[s], ((i >> 1) + 1) & 1, abort, status)) break;
        tc_fence_after();
        const uint32_t sB1 = kB1isY ? sY : sX;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b1 = kmajor(sB1, kk);
          umma_ts(tO, tA_hi + 8 * kk, b1, id_1, kk > 0 ? 1u : 0u);
          umma_ts(tO, tA_lo + 8 * kk, b1, id_1, 1u);
        }
        umma_commit(&bars->t1_done);
        if (!mbar_wait(&bars->m_full, i & 1, abort, status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a2 = mnmajor(sZ, kk);
          umma_ss(tO, a2, kMaskMN ? mnmajor(sX, kk) : kmajor(sX, kk), id_2, 1u);   // hi part (over X)
          umma_ss(tO, a2, kMaskMN ? mnmajor(sY, kk) : kmajor(sY, kk), id_2, 1u);   // lo part (over Y)
        }
        umma_commit(&bars->o_full[s]);
        umma_commit(&bars->stage_free[s]);
      }
      if (*abort) {   // every MMA issued has finished before the memory goes
        umma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    // ---------------------------------------------------- warps 0-7
    const int q4 = warp & 3, half = warp >> 2;
    const int lrow = q4 * 32 + lane;   // tensor-memory lane: row s of M, feature a of the output
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    auto state_ptrs = [&](int i, const float*& st, const float*& sin) {
      const int64_t n = block_of(i);
      const int64_t bh = n / nblk, j = n % nblk;
      st = a.st + (bh * nblk + j) * kD * kD;
      sin = a.shard_in + (bh * a.P + j / per_shard) * kD * kD;
    };
    bool ok = true;
    if (n_local > 0) {
      const float *st, *sin;
      state_ptrs(0, st, sin);
      load_state<kRowwise>(st, sin, tA_hi + lane_off, tA_lo + lane_off, lrow, half);
      tc_fence_before();
      mbar_arrive(&bars->state_full);
    }
    for (int i = 0; ok && i < n_local; ++i) {
      const int s = i & 1;
      uint8_t* sX = smem + s * STAGE;
      uint8_t* sY = sX + TILE;
      // the masked block product out of tensor memory
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->mask_full, i & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tM + lane_off + 64 * half, v);
      tmem_ld32(tM + lane_off + 64 * half + 32, v + 32);
      tmem_wait_ld32(v);
      tmem_wait_ld32(v + 32);
      tc_fence_before();
      mbar_arrive(&bars->tm_free);
      // X and Y of this stage are free once the state term has read them
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->t1_done, i & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int t = 64 * half + 8 * u + e;
          x[e] = t >= lrow ? __uint_as_float(v[8 * u + e]) : 0.f;
        }
        uint4 hi, lo;
        split8(x, hi, lo);
        const int c = 8 * half + u;
        *reinterpret_cast<uint4*>(sX + chunk_off(lrow, c)) = hi;
        *reinterpret_cast<uint4*>(sY + chunk_off(lrow, c)) = lo;
      }
      fence_async_smem();
      mbar_arrive(&bars->m_full);
      // the next block's state (its tensor memory is free after t1_done)
      if (i + 1 < n_local) {
        const float *st, *sin;
        state_ptrs(i + 1, st, sin);
        load_state<kRowwise>(st, sin, tA_hi + lane_off, tA_lo + lane_off, lrow, half);
        tc_fence_before();
        mbar_arrive(&bars->state_full);
      }
      // out[row0 + r][a] = scale * out^T[a][r]: lanes are features, so each
      // store instruction writes 32 consecutive floats of one row
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_full[s], (i >> 1) & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const int64_t n = block_of(i);
      float* out = a.out + (n / nblk * a.S + (n % nblk) * kBlk) * kD + lrow;
      const uint32_t tO = tO0 + 128 * s;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t w[32];
        tmem_ld32(tO + lane_off + 64 * half + 32 * cc, w);
        tmem_wait_ld32(w);
#pragma unroll
        for (int e = 0; e < 32; ++e) out[(64 * half + 32 * cc + e) * kD] = a.scale * __uint_as_float(w[e]);
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free[s]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

static int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (n[dev & 63] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0) c = 148;
    n[dev & 63] = c;
  }
  return n[dev & 63];
}

template <int MODE>
static int launch_block(const void* x, const void* y, const void* z, const float* st, const float* shard_in, float* out,
                        int64_t BH, int64_t S, int P, float scale, int* status, cudaStream_t stream,
                        const char* who) {
  SCA_REQUIRE(reinterpret_cast<uintptr_t>(st) % 16 == 0 && reinterpret_cast<uintptr_t>(shard_in) % 16 == 0,
              SCA_ERR_ALIGN, "%s: states must be 16-byte aligned", who);
  Args a;
  cudaError_t e = map_of(&a.mx, x, BH, S);
  if (e == cudaSuccess) e = map_of(&a.my, y, BH, S);
  if (e == cudaSuccess) e = map_of(&a.mz, z, BH, S);
  SCA_REQUIRE(e == cudaSuccess, SCA_ERR_ALIGN, "%s: inputs are not TMA-addressable (16-byte base)", who);
  a.st = st;
  a.shard_in = shard_in;
  a.out = out;
  a.S = S;
  a.BH = static_cast<int>(BH);
  a.P = P;
  a.scale = scale;
  a.status = status;
  if ((e = allow(block_kernel<MODE>, kSmem)) != cudaSuccess) return cuda_status(e, who);
  const int64_t total = BH * (S / kBlk);
  const int grid = static_cast<int>(total < sm_count() ? total : sm_count());
  block_kernel<MODE><<<grid, kPThreads, kSmem, stream>>>(a);
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
