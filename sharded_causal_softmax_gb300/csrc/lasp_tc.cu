// Causal linear attention over P contiguous shards on the tensor cores
// (linear attention sequence parallelism: "Effiziente Parallelisierung
// linearer Aufmerksamkeitssequenzen fuer skalierbare Sprachmodelle" -
// intermediate states passed point to point between shards, the
// right-product trick, fused kernels, cached k^T v states).  bf16 inputs,
// D = 128; the sequence goes in blocks of L rows (a multiple of 128), each
// taken as L/128 sub-blocks of 128 rows.
//
// The block algebra is that of the CUDA-core kernels in lasp.cu, with every
// product on tcgen05 (kind::f16, fp32 accumulation in tensor memory):
//
//   states:  st_j = A_j^T B_j                    (k^T v, or q^T dO backward)
//   forward: o_u  = scale (q_u F_u + tril(q_u k_u^T) v_u)
//   dq_u = scale (dO_u F_u^T + tril(dO_u v_u^T) k_u)
//   dk_u = scale (v_u G_u^T + tril(dO_u v_u^T)^T q_u)
//   dv_u = scale (k_u G_u + tril(q_u k_u^T)^T dO_u)
//
// for every sub-block u, where F_u (G_u) is the fp32 state of everything
// before (after) it.  A kernel starts each block from its stored state
// (st[j] + shard_in[r]) and carries the state from sub-block to sub-block
// itself (F += k_u^T v_u, or G += q_u^T dO_u walking the block backwards),
// so states are stored and scanned once per L rows.
//
// Two kinds of operand are not bf16 inputs: the state (fp32, entries up to
// ~sqrt(S)) and the masked block product (fp32).  Each is split as
// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi) (error below
// 2^-16 |x|) and multiplied twice, so every product keeps about fp32
// accuracy.
//
// Each kernel computes the TRANSPOSE of its output sub-block, out^T[a][r]
// (feature a in tensor-memory lane, row r in column): the epilogue then
// writes, for every row, 32 consecutive features per warp (128-byte
// stores), and every operand is a natural tile:
//
//   M[s][t] = x_s . y_t  (t >= s, else 0): A = X (K-major), B = Y (K-major)
//   out^T   = A1 B1 + Z^T M-or-M^T
//   U       = Z^T W (the sub-block's own state, in A1's orientation)
//
//   kernel  X  Y   Z   state term A1 (in tensor memory)  B1   mask as B          W
//   fwd     k  q   v   A1[a][b] = F[b][a]                 q    MN-major (k = s)   k
//   dq      v  dO  k   A1[a][b] = F[a][b]                 dO   MN-major (k = s)   v
//   dk      v  dO  q   A1[a][b] = G[a][b]                 v    K-major  (k = t)   dO
//   dv      k  q   dO  A1[a][b] = G[b][a]                 k    K-major  (k = t)   q
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

constexpr int kSub = 128;                // rows of a sub-block (the MMA tile)
constexpr int kD = 128;
constexpr int PANEL = 128 * 128;         // 128 rows x 64 bf16
constexpr int TILE = 2 * PANEL;          // 128 x 128 bf16

SCA_INLINE void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// byte offset of the 16-byte chunk with columns [8c, 8c + 8) of `row`
SCA_INLINE uint32_t chunk_off(int row, int c) {
  return (c >> 3) * PANEL + row * 128 + (((c & 7) ^ (row & 7)) << 4);
}

// operand descriptors of k-step kk (16 elements of the contraction)
// (the base descriptor is common to a loop's k-steps, which only add)
SCA_INLINE uint64_t kmajor(uint32_t base, int kk) {   // tile rows = M or N, K along the row
  return sdesc_step(sdesc_sw128(base, 16, 1024), (kk >> 2) * PANEL + (kk & 3) * 32);
}
SCA_INLINE uint64_t mnmajor(uint32_t base, int kk) {  // tile rows = K, M or N along the row
  return sdesc_step(sdesc_sw128(base, PANEL, 1024), kk * 2048);
}

// x = hi + lo, both bf16 (round to nearest even), for a pair
SCA_INLINE void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(hv);
  const __nv_bfloat162 lv = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&hv);
  lo = *reinterpret_cast<const uint32_t*>(&lv);
}

// Kernel arguments: X, Y, Z tile maps ([BH, S, D] bf16 views), the block
// states and shard inputs, the output.
struct Args {
  CUtensorMap mx, my, mz;
  const float* st;         // [BH, S/L, D, D]
  const float* shard_in;   // [BH, P, D, D]
  float* out;              // [BH, S, D]
  int64_t S;
  int BH;
  int P;
  int L;                   // rows per block
  float scale;
  int* status;
};

enum Mode { kFwd = 0, kDq = 1, kDk = 2, kDv = 3 };

// Persistent, pipelined block kernel: one CTA per SM walks blocks n =
// blockIdx.x, + gridDim.x, ..., each as L/128 sub-blocks.  Roles: warp 8
// loads X, Y, Z by TMA into two shared-memory stages; one thread of warp 9
// issues the MMAs; warps 0-7 keep the running state (fp32, in registers:
// lane a, half of the b range each), put it into tensor memory as the A
// operand of the state term, turn the masked product into shared-memory
// operands and write the output.  Tensor memory (512 columns): M (128);
// two output accumulators (2 x 128); the state's hi and lo parts (64 + 64,
// bf16 pairs), which the sub-block's own state product U (fp32, 128)
// overwrites once the state term has read them (MMAs from one thread run
// in order).  The masked product's hi and lo parts overwrite X and Y of
// their stage once the products that read them are done.
constexpr int kThreads = 320;
constexpr int kConv = 256;                  // warps 0-7
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int STAGE = 3 * TILE;             // X, Y, Z
constexpr int BAR_OFF = 2 * STAGE;
constexpr int kSmem = BAR_OFF + 1024 + 1024;

struct Bars {
  uint64_t in_full[2], stage_free[2];
  uint64_t mask_full;    // M of sub-block c in tM
  uint64_t tm_free;      // converters done with M of sub-block c
  uint64_t state_full;   // A1 of sub-block c in tensor memory
  uint64_t t1u_done;     // state term and U of sub-block c done: X, Y free, U over A1
  uint64_t m_full;       // masked product of sub-block c in X, Y
  uint64_t u_read;       // every converter warp has read U (phase per sub-block with a U)
  uint64_t o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// run[u] = A1[a][64 half + u] of block state st + shard input sin.
// ROWWISE: A1[a][b] = state[a][b] (a row per thread); else
// A1[a][b] = state[b][a] (a column per thread; each load instruction reads
// 32 consecutive floats of one row).
template <bool ROWWISE>
SCA_INLINE void load_state(float (&run)[64], const float* st, const float* sin, int a, int half) {
  if (ROWWISE) {
#pragma unroll
    for (int u = 0; u < 64; ++u) run[u] = st[a * kD + 64 * half + u] + sin[a * kD + 64 * half + u];
  } else {
#pragma unroll
    for (int u = 0; u < 64; ++u) run[u] = st[(64 * half + u) * kD + a] + sin[(64 * half + u) * kD + a];
  }
}

// the running state's hi and lo parts into tensor memory (lane-offset
// addresses of this warp's quadrant)
SCA_INLINE void put_state(const float (&run)[64], uint32_t t_hi, uint32_t t_lo, int half) {
  uint32_t hi[32], lo[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) split2(run[2 * c], run[2 * c + 1], hi[c], lo[c]);
  tmem_st32(t_hi + 32 * half, hi);
  tmem_st32(t_lo + 32 * half, lo);
  tmem_wait_st();
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) block_kernel(const __grid_constant__ Args a) {
  constexpr bool kRowwise = MODE == kDq || MODE == kDk;   // A1 = state (else its transpose)
  constexpr bool kFwdDir = MODE == kFwd || MODE == kDq;   // sub-blocks in order (else backwards)
  constexpr bool kB1isY = MODE == kFwd || MODE == kDq;    // B1 = Y (else X)
  constexpr bool kMaskMN = MODE == kFwd || MODE == kDq;   // mask as B: MN-major (else K-major)
  constexpr bool kWisX = MODE == kFwd || MODE == kDq;     // U = Z^T X (else Z^T Y)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsub = a.L / kSub;
  const int64_t nblk = a.S / a.L;
  const int64_t total = static_cast<int64_t>(a.BH) * nblk;
  const int64_t per_shard = nblk / a.P;
  int n_local = 0;
  if (blockIdx.x < total) n_local = static_cast<int>((total - 1 - blockIdx.x) / gridDim.x) + 1;
  const int n_sub = n_local * nsub;   // sub-blocks of this CTA, c = i * nsub + u
  auto block_of = [&](int i) { return static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * gridDim.x; };
  // first row (within its head) of sub-block c
  auto row_of = [&](int c) {
    const int i = c / nsub, u = c % nsub;
    const int uo = kFwdDir ? u : nsub - 1 - u;
    return (block_of(i) % nblk) * a.L + static_cast<int64_t>(uo) * kSub;
  };

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
    mbar_init(&bars->t1u_done, 1);
    mbar_init(&bars->m_full, kConv);
    mbar_init(&bars->u_read, kConv);
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
      int c = 0;
      for (; c < n_sub; ++c) {
        const int s = c & 1;
        if (c >= 2 && !mbar_wait(&bars->stage_free[s], ((c >> 1) + 1) & 1, abort, status)) break;
        const int bh = static_cast<int>(block_of(c / nsub) / nblk), row0 = static_cast<int>(row_of(c));
        uint8_t* st = smem + s * STAGE;
        mbar_arrive_expect_tx(&bars->in_full[s], 3 * TILE);
        for (int p = 0; p < 2; ++p) {
          tma_load_4d(st + p * PANEL, &a.mx, &bars->in_full[s], 64 * p, row0, bh, 0);
          tma_load_4d(st + TILE + p * PANEL, &a.my, &bars->in_full[s], 64 * p, row0, bh, 0);
          tma_load_4d(st + 2 * TILE + p * PANEL, &a.mz, &bars->in_full[s], 64 * p, row0, bh, 0);
        }
      }
      if (*abort)   // let the copies in flight land before the CTA goes away
        for (int j = (c > 2 ? c - 2 : 0); j < c; ++j) mbar_wait_drain(&bars->in_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_m = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t id_1 = idesc_bf16_f32(128, 128, false, false);   // A1 from tensor memory
      constexpr uint32_t id_2 = idesc_bf16_f32(128, 128, true, kMaskMN);
      constexpr uint32_t id_u = idesc_bf16_f32(128, 128, true, true);
      // M of sub-block c into tM once its tiles have landed and the
      // converters hold M of sub-block c - 1
      auto issue_mask = [&](int c) -> bool {
        const int s = c & 1;
        const uint32_t sX = s0 + s * STAGE, sY = sX + TILE;
        if (!mbar_wait(&bars->in_full[s], (c >> 1) & 1, abort, status)) return false;
        if (c >= 1 && !mbar_wait(&bars->tm_free, (c - 1) & 1, abort, status)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) umma_ss(tM, kmajor(sX, kk), kmajor(sY, kk), id_m, kk > 0 ? 1u : 0u);
        umma_commit(&bars->mask_full);
        return true;
      };
      bool ok = n_sub == 0 || issue_mask(0);
      for (int c = 0; ok && c < n_sub; ++c) {
        const int s = c & 1;
        const bool last = c % nsub == nsub - 1;   // no U: the next block starts from its stored state
        const uint32_t sX = s0 + s * STAGE, sY = sX + TILE, sZ = sX + 2 * TILE;
        const uint32_t tO = tO0 + 128 * s;
        if (!mbar_wait(&bars->state_full, c & 1, abort, status)) break;
        if (c >= 2 && !mbar_wait(&bars->o_free[s], ((c >> 1) + 1) & 1, abort, status)) break;
        tc_fence_after();
        const uint32_t sB1 = kB1isY ? sY : sX;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t b1 = kmajor(sB1, kk);
          umma_ts(tO, tA_hi + 8 * kk, b1, id_1, kk > 0 ? 1u : 0u);
          umma_ts(tO, tA_lo + 8 * kk, b1, id_1, 1u);
        }
        if (!last) {   // U over the state's columns, after the state term has read them
          const uint32_t sW = kWisX ? sX : sY;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) umma_ss(tA_hi, mnmajor(sZ, kk), mnmajor(sW, kk), id_u, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->t1u_done);
        // the next masked product fills the wait for m_full when its tiles
        // are already there; otherwise it follows this sub-block's products
        const int cn = c + 1;
        const bool early = cn < n_sub && mbar_try_wait(&bars->in_full[cn & 1], (cn >> 1) & 1);
        if (early && !issue_mask(cn)) break;
        if (!mbar_wait(&bars->m_full, c & 1, abort, status)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t a2 = mnmajor(sZ, kk);
          umma_ss(tO, a2, kMaskMN ? mnmajor(sX, kk) : kmajor(sX, kk), id_2, 1u);   // hi part (over X)
          umma_ss(tO, a2, kMaskMN ? mnmajor(sY, kk) : kmajor(sY, kk), id_2, 1u);   // lo part (over Y)
        }
        umma_commit(&bars->o_full[s]);
        umma_commit(&bars->stage_free[s]);
        if (cn < n_sub && !early && !issue_mask(cn)) break;
      }
      if (*abort) {   // every MMA issued has finished before the memory goes
        umma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    // ---------------------------------------------------- warps 0-7
    const int q4 = warp & 3, half = warp >> 2;
    const int lrow = q4 * 32 + lane;   // tensor-memory lane: row s of M, feature a of U and the output
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    auto load_block_state = [&](int i, float (&run)[64]) {
      const int64_t n = block_of(i);
      const int64_t bh = n / nblk, j = n % nblk;
      load_state<kRowwise>(run, a.st + (bh * nblk + j) * kD * kD, a.shard_in + (bh * a.P + j / per_shard) * kD * kD,
                           lrow, half);
    };
    float run[64];
    bool ok = true;
    int n_u = 0;   // sub-blocks so far whose U was read (phase of u_read)
    if (n_sub > 0) {
      load_block_state(0, run);
      put_state(run, tA_hi + lane_off, tA_lo + lane_off, half);
      tc_fence_before();
      mbar_arrive(&bars->state_full);
    }
    for (int c = 0; ok && c < n_sub; ++c) {
      const int s = c & 1;
      const bool last = c % nsub == nsub - 1;
      uint8_t* sX = smem + s * STAGE;
      uint8_t* sY = sX + TILE;
      // the masked product out of tensor memory
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->mask_full, c & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld32(tM + lane_off + 64 * half, v);
      tmem_ld32(tM + lane_off + 64 * half + 32, v + 32);
      tmem_wait_ld32(v);
      tmem_wait_ld32(v + 32);
      tc_fence_before();
      mbar_arrive(&bars->tm_free);
      // X and Y are free, U is over the state's columns
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->t1u_done, c & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 64 * half + 8 * u + 2 * e;
          split2(t >= lrow ? __uint_as_float(v[8 * u + 2 * e]) : 0.f,
                 t + 1 >= lrow ? __uint_as_float(v[8 * u + 2 * e + 1]) : 0.f, h[e], l[e]);
        }
        const int ch = 8 * half + u;
        *reinterpret_cast<uint4*>(sX + chunk_off(lrow, ch)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(sY + chunk_off(lrow, ch)) = make_uint4(l[0], l[1], l[2], l[3]);
      }
      fence_async_smem();
      mbar_arrive(&bars->m_full);
      // the state of the next sub-block: run + U, or the next block's
      // stored state
      if (!last) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t w[32];
          tmem_ld32(tA_hi + lane_off + 64 * half + 32 * cc, w);
          tmem_wait_ld32(w);
#pragma unroll
          for (int e = 0; e < 32; ++e) run[32 * cc + e] += __uint_as_float(w[e]);
        }
        // every warp has read its part of U before any overwrites it (a
        // bounded mbarrier: a warp that gave up on an earlier wait must not
        // leave the others in a hardware barrier)
        tc_fence_before();
        mbar_arrive(&bars->u_read);
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->u_read, n_u & 1, abort, status));
        ++n_u;
        if (!ok) break;
        tc_fence_after();
      } else if (c + 1 < n_sub) {
        load_block_state(c / nsub + 1, run);
      }
      if (c + 1 < n_sub) {
        put_state(run, tA_hi + lane_off, tA_lo + lane_off, half);
        tc_fence_before();
        mbar_arrive(&bars->state_full);
      }
      // out[row0 + r][a] = scale * out^T[a][r]: lanes are features, so each
      // store instruction writes 32 consecutive floats of one row
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_full[s], (c >> 1) & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const int64_t bh = block_of(c / nsub) / nblk;
      float* out = a.out + (bh * a.S + row_of(c)) * kD + lrow;
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

// st[bh][j] = A_j^T B_j over the L rows of block j, accumulated over its
// sub-blocks in tensor memory.  Computed transposed, D^T[m = b-feature][n =
// a-feature] with both tiles MN-major (rows = the contraction), so that the
// epilogue writes 32 consecutive floats of a state row per store.
// Persistent: warp 4 loads A, B tiles by TMA (two stages), one thread of
// warp 5 issues the MMAs into two accumulators, warps 0-3 write the states.
struct StArgs {
  CUtensorMap ma, mb;
  float* st;
  int64_t S;
  int BH;
  int L;
  int* status;
};

constexpr int kStThreads = 192;
constexpr int ST_STAGE = 2 * TILE;
constexpr int ST_BAR_OFF = 2 * ST_STAGE;
constexpr int kStSmem = ST_BAR_OFF + 1024 + 1024;

struct StBars {
  uint64_t in_full[2], stage_free[2], acc_full[2], acc_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kStThreads, 1) states_kernel(const __grid_constant__ StArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  StBars* bars = reinterpret_cast<StBars*>(smem + ST_BAR_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsub = a.L / kSub;
  const int64_t nblk = a.S / a.L;
  const int64_t total = static_cast<int64_t>(a.BH) * nblk;
  int n_local = 0;
  if (blockIdx.x < total) n_local = static_cast<int>((total - 1 - blockIdx.x) / gridDim.x) + 1;
  auto block_of = [&](int i) { return static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(i) * gridDim.x; };
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->in_full[i], 1);
      mbar_init(&bars->stage_free[i], 1);
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_free[i], 128);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  int* status = a.status;

  if (warp == 4) {
    if (lane == 0) {
      tma_prefetch_map(&a.ma);
      tma_prefetch_map(&a.mb);
      const int n_sub = n_local * nsub;
      int c = 0;
      for (; c < n_sub; ++c) {
        const int s = c & 1;
        if (c >= 2 && !mbar_wait(&bars->stage_free[s], ((c >> 1) + 1) & 1, abort, status)) break;
        const int64_t n = block_of(c / nsub);
        const int bh = static_cast<int>(n / nblk);
        const int row0 = static_cast<int>((n % nblk) * a.L + static_cast<int64_t>(c % nsub) * kSub);
        uint8_t* st = smem + s * ST_STAGE;
        mbar_arrive_expect_tx(&bars->in_full[s], 2 * TILE);
        for (int p = 0; p < 2; ++p) {
          tma_load_4d(st + p * PANEL, &a.ma, &bars->in_full[s], 64 * p, row0, bh, 0);
          tma_load_4d(st + TILE + p * PANEL, &a.mb, &bars->in_full[s], 64 * p, row0, bh, 0);
        }
      }
      if (*abort)
        for (int j = (c > 2 ? c - 2 : 0); j < c; ++j) mbar_wait_drain(&bars->in_full[j & 1], (j >> 1) & 1);
    }
  } else if (warp == 5) {
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, 128, true, true);
      int c = 0;
      bool ok = true;
      for (int i = 0; ok && i < n_local; ++i) {
        const uint32_t tD = tmem + 128 * (i & 1);
        if (i >= 2 && !mbar_wait(&bars->acc_free[i & 1], ((i >> 1) + 1) & 1, abort, status)) break;
        for (int u = 0; u < nsub; ++u, ++c) {
          const int s = c & 1;
          if (!mbar_wait(&bars->in_full[s], (c >> 1) & 1, abort, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + s * ST_STAGE), sB = sA + TILE;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss(tD, mnmajor(sB, kk), mnmajor(sA, kk), id, (u > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->stage_free[s]);
        }
        if (ok) umma_commit(&bars->acc_full[i & 1]);
      }
      if (*abort) {
        umma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    const int jb = warp * 32 + lane;   // b-feature (lane)
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    for (int i = 0; i < n_local; ++i) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_full[i & 1], (i >> 1) & 1, abort, status))) break;
      tc_fence_after();
      float* st = a.st + block_of(i) * kD * kD + jb;   // blocks are numbered bh * nblk + j
      const uint32_t tD = tmem + 128 * (i & 1);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(tD + lane_off + 32 * cc, v);
        tmem_wait_ld32(v);
#pragma unroll
        for (int e = 0; e < 32; ++e) st[(32 * cc + e) * kD] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      mbar_arrive(&bars->acc_free[i & 1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// [BH, S, 128] bf16 tensor as a TMA map with 64 x 128 boxes
static cudaError_t map_of(CUtensorMap* m, const void* p, int64_t BH, int64_t S) {
  View v;
  v.s = kD;
  v.h = S * kD;
  v.b = BH * S * kD;
  return make_tmap_bf16(m, p, kD, S, static_cast<int>(BH), 1, v, 64, kSub);
}

template <typename K>
static cudaError_t allow(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
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

static int persistent_grid(int64_t blocks) {
  const int sms = sm_count();
  return static_cast<int>(blocks < sms ? blocks : sms);
}

}  // namespace lasp_tc

using namespace lasp_tc;

int lasp_tc_states(const void* a, const void* b, float* st, int64_t BH, int64_t S, int L, int* status,
                   cudaStream_t stream) {
  StArgs sa;
  cudaError_t e = map_of(&sa.ma, a, BH, S);
  if (e == cudaSuccess) e = map_of(&sa.mb, b, BH, S);
  SCA_REQUIRE(e == cudaSuccess, SCA_ERR_ALIGN, "lasp_block_states: inputs are not TMA-addressable (16-byte base)");
  sa.st = st;
  sa.S = S;
  sa.BH = static_cast<int>(BH);
  sa.L = L;
  sa.status = status;
  if ((e = allow(states_kernel, kStSmem)) != cudaSuccess) return cuda_status(e, "lasp_block_states");
  states_kernel<<<persistent_grid(BH * (S / L)), kStThreads, kStSmem, stream>>>(sa);
  return cuda_status(cudaGetLastError(), "lasp_block_states launch");
}

template <int MODE>
static int launch_block(const void* x, const void* y, const void* z, const float* st, const float* shard_in, float* out,
                        int64_t BH, int64_t S, int P, int L, float scale, int* status, cudaStream_t stream,
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
  a.L = L;
  a.scale = scale;
  a.status = status;
  if ((e = allow(block_kernel<MODE>, kSmem)) != cudaSuccess) return cuda_status(e, who);
  block_kernel<MODE><<<persistent_grid(BH * (S / L)), kThreads, kSmem, stream>>>(a);
  return cuda_status(cudaGetLastError(), who);
}

int lasp_tc_fwd(const void* q, const void* k, const void* v, const float* st, const float* shard_in, float* o,
                int64_t BH, int64_t S, int P, int L, float scale, int* status, cudaStream_t stream) {
  return launch_block<kFwd>(k, q, v, st, shard_in, o, BH, S, P, L, scale, status, stream, "lasp_fwd");
}

int lasp_tc_bwd(const void* q, const void* k, const void* v, const void* dout, const float* st_f, const float* in_f,
                const float* st_b, const float* in_b, float* dq, float* dk, float* dv, int64_t BH, int64_t S, int P,
                int L, float scale, int* status, cudaStream_t stream) {
  int rc = launch_block<kDq>(v, dout, k, st_f, in_f, dq, BH, S, P, L, scale, status, stream, "lasp_bwd (dq)");
  if (rc == SCA_OK)
    rc = launch_block<kDk>(v, dout, q, st_b, in_b, dk, BH, S, P, L, scale, status, stream, "lasp_bwd (dk)");
  if (rc == SCA_OK)
    rc = launch_block<kDv>(k, q, dout, st_b, in_b, dv, BH, S, P, L, scale, status, stream, "lasp_bwd (dv)");
  return rc;
}

}  // namespace sca
