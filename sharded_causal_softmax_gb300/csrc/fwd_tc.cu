// Forward (o, lse) partial on the 5th-generation tensor cores (sm_103a).
//
// One CTA owns a tile of 128 query rows of one (item, batch, head) and walks
// the item's visible key/value tiles of 128 rows:
//
//   warp 4      TMA producer for Q (once) and the K ring (3 stages)
//   warp 6      TMA producer for the V ring (2 stages)
//   warp 5      tensor-memory allocation, and one thread issuing tcgen05.mma:
//                 S[n%2] = Q K_n^T           (A, B from shared memory)
//                 O     += P_{n-1} V_{n-1}   (A = P from tensor memory)
//   warps 0-3   softmax: thread t owns query row t (tensor-memory lane t),
//               reads its S row, keeps the running max/sum in fp32, writes
//               P (bf16) back over its S row and rescales O when the max
//               grows by more than 2^8 (lazy rescale; exact after the final
//               division); then the epilogue o = O / l, lse = m + ln l.
//
// S is double-buffered in tensor memory so QK^T of tile n+1 runs while the
// softmax of tile n is computed; K/V stages mirror the ring step's double
// buffer.  Tiles with no visible (query, key) pair are skipped; tiles that
// may hold masked pairs or ragged rows are masked elementwise.
//
// Tensor memory: S0 cols [0,128), S1 [128,256), O [256, 256+D); 512 columns
// allocated (one CTA per SM: shared memory use is above half the SM).
// Every mbarrier wait is bounded (ptx.cuh); on expiry the CTA records
// SCA_ERR_TIMEOUT, drains its in-flight copies and MMAs (bounded), frees
// its tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "simt_launch.h"
#include "tmap.h"

namespace sca {
namespace fwdtc {

constexpr int BM = 128;        // query rows per CTA
constexpr int BN = 128;        // keys per tile
constexpr int KST = 3;         // K stages
constexpr int VST = 2;         // V stages
constexpr int PANEL = 128 * 128;  // bytes of 128 rows x 64 bf16 (one 128B-swizzle panel column)
constexpr int kThreads = 224;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units)

template <int D>
struct Layout {
  static constexpr int TILE = (D / 64) * PANEL;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + KST * TILE;
  static constexpr int BAR_OFF = V_OFF + VST * TILE;
  static constexpr int BAR_BYTES = 256;
  static constexpr int USED = BAR_OFF + BAR_BYTES;
  // keep one CTA per SM (tensor memory is allocated whole): above half the SM
  static constexpr int SMEM = (USED + 1024 > 120 * 1024 ? USED + 1024 : 120 * 1024);
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct TcArgs {
  CUtensorMap maps[SCA_MAX_ITEMS][3];  // q, k, v
  AttnArgs a;
};

struct TileInfo {
  int64_t k0;
  int nk;
  bool visible, full;
};

SCA_INLINE TileInfo tile_info(const Item& it, int kt, bool causal, int64_t qmin, int64_t qmax) {
  TileInfo t;
  t.k0 = static_cast<int64_t>(kt) * BN;
  t.nk = static_cast<int>(min64(BN, it.Skv - t.k0));
  int64_t kmin, kmax;
  tile_pos_range(it.ks, t.k0, t.nk, kmin, kmax);
  t.visible = !causal || kmin <= qmax;
  t.full = t.nk == BN && (!causal || kmax <= qmin);
  return t;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcArgs ta) {
  using L = Layout<D>;
  const AttnArgs& a = ta.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::BAR_OFF);

  const int item_idx = blockIdx.z;
  const Item& it = a.items[item_idx];
  const int64_t q0 = static_cast<int64_t>(a.max_q_tiles - 1 - blockIdx.x) * BM;  // heavy tiles first
  if (q0 >= it.Sq) return;
  const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
  const int nq = static_cast<int>(min64(BM, it.Sq - q0));
  int64_t qmin, qmax;
  tile_pos_range(it.qs, q0, nq, qmin, qmax);
  const int nkt = static_cast<int>((it.Skv + BN - 1) / BN);
  const bool causal = a.causal != 0;

  int n_vis = 0;
  for (int kt = 0; kt < nkt; ++kt) n_vis += tile_info(it, kt, causal, qmin, qmax).visible ? 1 : 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (n_vis == 0) {
    // no visible key: the empty partial
    if (warp < 4) {
      const int row = threadIdx.x;
      if (row < nq) {
        float* op = it.o + b * a.o.b + h * a.o.h + (q0 + row) * a.o.s;
        for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(op + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        it.lse[b * a.lse_b + h * a.lse_h + q0 + row] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], BM);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  int* status = a.status;

  const uint32_t sQ = smem_u32(smem + L::Q_OFF);
  const uint32_t sK = smem_u32(smem + L::K_OFF);
  const uint32_t sV = smem_u32(smem + L::V_OFF);

  if (warp == 4) {
    // ------------------------------------------------ Q + K producer
    if (lane == 0) {
      const CUtensorMap* mq = &ta.maps[item_idx][0];
      const CUtensorMap* mk = &ta.maps[item_idx][1];
      tma_prefetch_map(mq);
      tma_prefetch_map(mk);
      mbar_arrive_expect_tx(&bars->q_full, L::TILE);
      for (int p = 0; p < D / 64; ++p)
        tma_load_4d(smem + L::Q_OFF + p * PANEL, mq, &bars->q_full, 64 * p, static_cast<int>(q0), h, b);
      int n = 0;
      for (int kt = 0; kt < nkt; ++kt) {
        const TileInfo ti = tile_info(it, kt, causal, qmin, qmax);
        if (!ti.visible) continue;
        const int st = n % KST;
        if (!mbar_wait(&bars->k_empty[st], ((n / KST) & 1) ^ 1, abort, status)) break;
        mbar_arrive_expect_tx(&bars->k_full[st], L::TILE);
        for (int p = 0; p < D / 64; ++p)
          tma_load_4d(smem + L::K_OFF + st * L::TILE + p * PANEL, mk, &bars->k_full[st], 64 * p,
                      static_cast<int>(ti.k0), h, b);
        ++n;
      }
      if (*abort) {  // let issued copies land before the CTA goes away
        for (int j = (n > KST ? n - KST : 0); j < n; ++j) mbar_wait_drain(&bars->k_full[j % KST], (j / KST) & 1);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------ V producer
    if (lane == 0) {
      const CUtensorMap* mv = &ta.maps[item_idx][2];
      tma_prefetch_map(mv);
      int n = 0;
      for (int kt = 0; kt < nkt; ++kt) {
        const TileInfo ti = tile_info(it, kt, causal, qmin, qmax);
        if (!ti.visible) continue;
        const int st = n % VST;
        if (!mbar_wait(&bars->v_empty[st], ((n / VST) & 1) ^ 1, abort, status)) break;
        mbar_arrive_expect_tx(&bars->v_full[st], L::TILE);
        for (int p = 0; p < D / 64; ++p)
          tma_load_4d(smem + L::V_OFF + st * L::TILE + p * PANEL, mv, &bars->v_full[st], 64 * p,
                      static_cast<int>(ti.k0), h, b);
        ++n;
      }
      if (*abort) {
        for (int j = (n > VST ? n - VST : 0); j < n; ++j) mbar_wait_drain(&bars->v_full[j % VST], (j / VST) & 1);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      const uint32_t tO = tmem + 256;
      bool ok = mbar_wait(&bars->q_full, 0, abort, status);
      auto issue_pv = [&](int j) -> bool {
        const int vs = j % VST;
        if (!mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abort, status)) return false;
        if (!mbar_wait(&bars->v_full[vs], (j / VST) & 1, abort, status)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + (j & 1) * 128;
        const uint32_t vbase = sV + vs * L::TILE;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          // B = V tile, MN-major: 64-column panels LBO apart, 8-key groups 1024 B apart
          const uint64_t bdesc = sdesc_sw128(vbase + kk * 2048, PANEL, 1024);
          umma_ts(tO, tP + kk * 8, bdesc, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&bars->v_empty[vs]);
        umma_commit(&bars->pv_done[j & 1]);
        return true;
      };
      int n = 0;
      for (int kt = 0; ok && kt < nkt; ++kt) {
        const TileInfo ti = tile_info(it, kt, causal, qmin, qmax);
        if (!ti.visible) continue;
        const int ks = n % KST;
        if (!mbar_wait(&bars->k_full[ks], (n / KST) & 1, abort, status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tS = tmem + (n & 1) * 128;
        const uint32_t kbase = sK + ks * L::TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;   // K-major: panel, then 32 B steps
          umma_ss(tS, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(kbase + off, 16, 1024), idesc_qk,
                  kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s_full[n & 1]);
        umma_commit(&bars->k_empty[ks]);
        if (n > 0 && !issue_pv(n - 1)) { ok = false; break; }
        ++n;
      }
      if (ok && n > 0) ok = issue_pv(n - 1);
      if (!ok) {  // make sure no MMA still writes tensor memory
        umma_commit(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    // -------------------------------------------- softmax (warps 0..3)
    const int row = threadIdx.x;  // == tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const bool row_valid = row < nq;
    const int64_t qpos = row_valid ? seg_pos(it.qs, q0 + row) : INT64_MIN;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    int n = 0;
    bool ok = true;
    for (int kt = 0; kt < nkt; ++kt) {
      const TileInfo ti = tile_info(it, kt, causal, qmin, qmax);
      if (!ti.visible) continue;
      const int sb = n & 1;
      bool w = n < 2 || mbar_wait(&bars->pv_done[sb], ((n - 2) >> 1) & 1, abort, status);
      w = w && mbar_wait(&bars->s_full[sb], (n >> 1) & 1, abort, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[BN];
      const uint32_t tS = tmem + lane_off + sb * 128;
#pragma unroll
      for (int c = 0; c < BN; c += 32) tmem_ld32(tS + c, sr + c);
#pragma unroll
      for (int c = 0; c < BN; c += 32) tmem_wait_ld32(sr + c);
      float* s = reinterpret_cast<float*>(sr);
      if (!ti.full) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const bool vis = c < ti.nk && (!causal || seg_pos(it.ks, ti.k0 + c) <= qpos);
          if (!vis) s[c] = -INFINITY;
        }
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx0 = fmaxf(mx0, s[c]); mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]); mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float mt = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
      const float m_new = fmaxf(m_used, mt);
      const bool need = m_new > m_used + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m_used - m_new) : 1.f;   // m_used = -inf gives 0
        if (need) m_used = m_new;
        l *= alpha;
        if (n > 0) {
          const bool w1 = mbar_wait(&bars->pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort, status);
          if (!__all_sync(0xffffffffu, w1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tO = tmem + lane_off + 256;
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(tO + c, r);
            tmem_wait_ld32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + c, r);
          }
        }
      }
      const float msub = (m_used == -INFINITY) ? 0.f : m_used;
      float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = half * 64 + 2 * i;
          const float p0 = ex2(fmaf(s[c], sl2, -msub));
          const float p1 = ex2(fmaf(s[c + 1], sl2, -msub));
          sum0 += p0;
          sum1 += p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st32(tS + half * 32, pk);
      }
      l += sum0 + sum1;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[sb]);
      ++n;
    }
    // epilogue
    if (ok && n > 0) ok = mbar_wait(&bars->pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort, status);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      float* op = it.o + b * a.o.b + h * a.o.h + (q0 + (row_valid ? row : 0)) * a.o.s;
      const uint32_t tO = tmem + lane_off + 256;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tO + c, r);
        tmem_wait_ld32(r);
        if (row_valid) {
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 v = make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                         __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
            *reinterpret_cast<float4*>(op + c + i) = v;
          }
        }
      }
      if (row_valid)
        it.lse[b * a.lse_b + h * a.lse_h + q0 + row] = l > 0.f ? (m_used + log2f(l)) * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch(TcArgs& ta, cudaStream_t st) {
  using L = Layout<D>;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] = cudaFuncSetAttribute(fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  dim3 grid(ta.a.max_q_tiles, ta.a.B * ta.a.H, ta.a.n_items);
  fwd_tc_kernel<D><<<grid, kThreads, L::SMEM, st>>>(ta);
  return cudaGetLastError();
}

}  // namespace fwdtc

cudaError_t tc_forward(AttnArgs& a, cudaStream_t st) {
  using namespace fwdtc;
  static TcArgs ta;  // large; filled per call on the host (calls are host-serialised per thread)
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  int64_t mt = 0;
  for (int i = 0; i < a.n_items; ++i) {
    const Item& it = a.items[i];
    const int64_t t = (it.Sq + BM - 1) / BM;
    if (t > mt) mt = t;
    cudaError_t e;
    if ((e = make_tmap_bf16(&ta.maps[i][0], it.q, a.D, it.Sq, a.H, a.B, a.q, 64, BM)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&ta.maps[i][1], it.k, a.D, it.Skv, a.H, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&ta.maps[i][2], it.v, a.D, it.Skv, a.H, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
  }
  a.max_q_tiles = static_cast<int>(mt);
  ta.a = a;
  return a.D == 64 ? launch<64>(ta, st) : launch<128>(ta, st);
}

}  // namespace sca
