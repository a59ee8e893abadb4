// Backward of one (query shard, key block) item on the 5th-generation
// tensor cores (sm_103a), recomputing P from the saved lse.
//
// One CTA owns a tile of 128 keys of one (item, batch, key/value head),
// keeps dK and dV for it in tensor memory, and walks the query tiles (128
// rows) that can see it, of every query head that reads this key/value head
// (one head, or a group under grouped-query attention), so dK and dV sum
// over the group in tensor memory.  Per query tile i:
//
//   S^T = K Q_i^T          dP^T = V dO_i^T        (A = K/V, B = Q/dO; smem)
//   P^T = exp(scale S^T - lse_i)                   (warps 0-7, phase 1)
//   dV += P^T dO_i                                 (A = P^T in tmem)
//   dS^T = P^T (dP^T - delta_i)                    (warps 0-7, phase 2)
//   dK += dS^T Q_i         dQ_i = dS K             (A = dS^T in tmem / dS in smem)
//   dq[rows of tile i] += dQ_i                     (TMA reduce-add, fp32)
//
// dS carries the score scale: phase 2 forms P^T (scale dP^T - scale delta)
// with one fused multiply-add against -scale*delta staged by the producer,
// so dK and dQ come out of the products already scaled.
//
// The MMAs run in that order, so phase 1 overlaps dP^T, phase 2 overlaps
// dV, and the next tile's S^T overlaps the read-back of dQ_i.  Both phases
// signal each 32-query chunk, and dV and dK each run as two halves, so an
// MMA half starts as soon as its chunk is written.
//
// Roles: warps 0-7 elementwise (two warpgroups; warpgroup g owns query
// columns [64g, 64g+64), thread = key row = tensor-memory lane), then read
// back dQ (thread = query row) and, at the end, dK / dV; warp 8 issues TMA
// loads (K, V once; Q_i, dO_i double-buffered) and stages lse / delta; warp
// 9 allocates tensor memory and runs the MMA loop, the whole warp waiting
// and one elected lane issuing each tcgen05.mma.
//
// Tensor memory (512 columns): S^T [0,128), dP^T [128,256), dV [256,256+D),
// dK [256+D, 256+2D).  Warpgroup g writes its P^T (bf16, 32 columns) over the
// S^T columns it has already read, [64g, 64g+32), and dS^T over
// [128+64g, 128+64g+32).  dQ_i (D columns) goes over the dP^T columns once
// dK has read dS^T (MMAs execute in issue order); the next tile's dP^T waits
// until dQ_i has been read back, its S^T only for dV to have read P^T.
//
// Precision: S^T, dK and dQ run as fp16 MMAs.  The elementwise warps convert
// the K tile (once) and each Q tile in shared memory from bf16 to fp16
// (exact for |x| in [2^-14, 65280]; a finite |x| >= 65536 would become
// +-inf and is recorded as SCA_ERR_RANGE in the status word), and round dS
// to fp16 (2^-11 relative) instead of bf16 (2^-8):
// with few visible keys a query's dQ is a short sum of large dS terms and
// bf16 dS alone would cost more than 1e-2.  dP^T and dV take bf16 V, dO, P^T,
// except under grouped-query attention (F16PV), where dV sums P^T dO over
// every query head of the group and bf16 P missed 1e-2: there V (once) and
// each dO tile are converted too and P^T is rounded to fp16.  Q (and, under
// F16PV, dO) may arrive already in fp16, converted once per call by the
// caller (launch flag f16_inputs): then their tiles are used as loaded.
//
// Every wait is bounded (ptx.cuh); on expiry the CTA records
// SCA_ERR_TIMEOUT, drains in-flight copies/MMAs (bounded), frees tensor
// memory and returns.
#include <cuda.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "simt_launch.h"
#include "tmap.h"

namespace sca {
namespace bwdtc {

constexpr int BN = 128;           // keys per CTA
constexpr int BM = 128;           // query rows per tile
constexpr int PANEL = 128 * 128;  // bytes: 128 rows x 64 bf16, 128B swizzle
constexpr int kThreads = 320;

template <int D>
struct Layout {
  static constexpr int TILE = (D / 64) * PANEL;  // 128 rows x D bf16
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE;
  static constexpr int Q_OFF = V_OFF + TILE;          // 2 stages
  static constexpr int DO_OFF = Q_OFF + 2 * TILE;     // 2 stages
  static constexpr int DS_OFF = DO_OFF + 2 * TILE;    // dS^T: 128 keys x 128 queries, 2 panels
  static constexpr int LSE_OFF = DS_OFF + 2 * PANEL;  // 2 stages x (lse*log2e, delta) x 128 rows, fp32
  static constexpr int BAR_OFF = LSE_OFF + 2 * 2 * BM * 4;
  static constexpr int USED = BAR_OFF + 256;
  static constexpr int kMaxSmem = 232448;              // per-CTA limit (227 KB)
  // room to align the base to 1024 B when it fits; otherwise the kernel
  // checks at run time that the base is already aligned
  static constexpr int SMEM = USED + 1024 <= kMaxSmem ? (USED + 1024 > 120 * 1024 ? USED + 1024 : 120 * 1024)
                                                       : USED;
};

struct Bars {
  uint64_t kv_full;
  uint64_t q_full[2];        // Q tile landed, lse/delta staged
  uint64_t do_full[2];       // dO tile landed
  uint64_t q_empty[2];       // the MMAs of the stage's tile have completed
  uint64_t dq_staged[2];     // dQ of the stage's tile staged (dS panels + its dO) for the reduce
  uint64_t ds_free;          // the reduce has read the dQ half staged in the dS panels
  uint64_t epi_staged[2];    // warpgroup g staged dK (g=0) / dV (g=1) for the final TMA write
  uint64_t s_full, dp_full;   // S^T / dP^T of the current tile in tensor memory
  uint64_t p_half[2];        // P^T of query chunk c (32 per warpgroup) written by warps 0-7
  uint64_t ds_half[2];       // dS^T of query chunk c written (after chunk 1: dS in smem too)
  uint64_t dq_full, tmem_free;
  uint64_t k_conv, q_conv;   // K and V / the current Q tile converted to fp16
  uint64_t do_conv;          // the current dO tile converted to fp16
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// Items per launch: seven tensor maps per item must fit, with the rest of the
// arguments, in the 32764 bytes of kernel parameters.
constexpr int kItemsPerLaunch = 28;

struct TcArgs {
  // q, k, v, dO (bf16); dq, dk, dv (fp32, TMA reduce-add / store targets)
  CUtensorMap maps[kItemsPerLaunch][7];
  AttnArgs a;
  int32_t f16_inputs;   // SCA_F16_Q / SCA_F16_DOUT: those inputs arrive as fp16
};
static_assert(sizeof(TcArgs) <= 32764, "kernel parameters");

struct QTile {
  int64_t q0;
  int nq;
  int64_t qmin, qmax;
  bool visible, full;
};

SCA_INLINE QTile q_tile(const ItemGeom& g, int t, bool causal, int nk, int64_t kmin, int64_t kmax) {
  QTile q;
  q.q0 = static_cast<int64_t>(t) * BM;
  q.nq = static_cast<int>(min64(BM, g.Sq - q.q0));
  tile_pos_range(g.qs, q.q0, q.nq, q.qmin, q.qmax);
  q.visible = !causal || kmin <= q.qmax;
  q.full = q.nq == BM && nk == BN && (!causal || kmax <= q.qmin);
  return q;
}

SCA_INLINE void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// F16PV: P^T, V and dO in fp16 too, so dP^T and dV are fp16 MMAs (chosen for
// grouped-query attention, where dV sums over the group); otherwise those
// two products take the bf16 inputs as they are.
template <int D, bool F16PV>
__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ TcArgs ta) {
  using L = Layout<D>;
  const AttnArgs& a = ta.a;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  if (pad + L::USED > L::SMEM) {   // 128B-swizzled tiles need a 1024-aligned base
    if (threadIdx.x == 0) report(a.status, SCA_ERR_ALIGN);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  Bars* bars = reinterpret_cast<Bars*>(smem + L::BAR_OFF);
  float* lse_sm = reinterpret_cast<float*>(smem + L::LSE_OFF);   // [stage][lse2 | delta][row]

  const int item_idx = blockIdx.z;
  const Item& it = a.items[item_idx];
  const ItemGeom gm = item_geom(it);
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * BN;   // early keys (most queries) first
  if (k0 >= gm.Skv) return;
  // one key/value head; its query heads [h0, h0 + group) all read it
  const int b = blockIdx.y / a.Hkv, hk = blockIdx.y % a.Hkv;
  const int h0 = hk * a.group;
  const int nk = static_cast<int>(min64(BN, gm.Skv - k0));
  int64_t kmin, kmax;
  tile_pos_range(gm.ks, k0, nk, kmin, kmax);
  const bool causal = a.causal != 0;
  const int nqt = static_cast<int>((gm.Sq + BM - 1) / BM);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto qvis = [&](int t) { return q_tile(gm, t, causal, nk, kmin, kmax).visible; };
  // the same query tiles are visible for every query head of the group
  const int n_vis = count_tiles(nqt, lane, qvis) * a.group;
  float* dk_base = it.dk + b * a.dkv.b + hk * a.dkv.h;
  float* dv_base = it.dv + b * a.dkv.b + hk * a.dkv.h;

  if (n_vis == 0) {
    // no query sees these keys: overwrite mode still owes zeros
    if (!a.accumulate && threadIdx.x < nk) {
      const int64_t r = slab_row(gm.ks, a.dkv_by_pos, k0 + threadIdx.x);
      float* pk = dk_base + r * a.dkv.s;
      float* pv = dv_base + r * a.dkv.s;
      for (int c = 0; c < D; c += 4) {
        *reinterpret_cast<float4*>(pk + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4*>(pv + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->q_full[i], 1 + 32);   // TMA transaction + the producer warp's lse/delta stores
      mbar_init(&bars->do_full[i], 1);
      mbar_init(&bars->q_empty[i], 1);
      mbar_init(&bars->dq_staged[i], 256);
    }
    mbar_init(&bars->ds_free, 1);
    for (int i = 0; i < 2; ++i) mbar_init(&bars->epi_staged[i], 128);
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->p_half[i], 256);
      mbar_init(&bars->ds_half[i], 256);
    }
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->tmem_free, 256);
    mbar_init(&bars->k_conv, 256);
    mbar_init(&bars->q_conv, 256);
    mbar_init(&bars->do_conv, 256);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  int* status = a.status;
  const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;

  if (warp == 8) {
    // ---------------- TMA producer (lane 0), lse/delta staging, dq reduce-add
    const CUtensorMap* mq = &ta.maps[item_idx][0];
    const CUtensorMap* mo = &ta.maps[item_idx][3];
    const CUtensorMap* mdq = &ta.maps[item_idx][4];
    if (lane == 0) {
      const CUtensorMap* mk = &ta.maps[item_idx][1];
      const CUtensorMap* mv = &ta.maps[item_idx][2];
      tma_prefetch_map(mq);
      tma_prefetch_map(mo);
      tma_prefetch_map(mdq);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * L::TILE);
      for (int p = 0; p < D / 64; ++p) {
        const int krow0 = static_cast<int>(slab_row(gm.ks, a.kv_by_pos, k0));
        tma_load_4d(smem + L::K_OFF + p * PANEL, mk, &bars->kv_full, 64 * p, krow0, hk, b);
        tma_load_4d(smem + L::V_OFF + p * PANEL, mv, &bars->kv_full, 64 * p, krow0, hk, b);
      }
    }
    int q0_st0 = 0, q0_st1 = 0;   // first query row of the tile each stage holds
    int h_st0 = 0, h_st1 = 0;     // and its query head
    // dq[rows of the j-th visible tile] += its staged dQ, D/32 boxes of 32
    // fp32 columns: the first D/64 (warpgroup 0's half) from the dS panels,
    // the rest from the tile's dO stage.  Two bulk groups; once the first is
    // read the dS panels are released.
    auto reduce_tile = [&](int j) -> bool {
      const int sj = j & 1;
      const bool w = __all_sync(0xffffffffu, mbar_wait(&bars->dq_staged[sj], (j >> 1) & 1, abort, status));
      if (w && lane == 0) {
        const int row0 = sj ? q0_st1 : q0_st0, hq = sj ? h_st1 : h_st0;
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
          tma_reduce_add_4d(mdq, smem + L::DS_OFF + bx * PANEL, 32 * bx, row0, hq, b);
        bulk_commit();
#pragma unroll
        for (int bx = 0; bx < D / 64; ++bx)
          tma_reduce_add_4d(mdq, smem + L::DO_OFF + sj * L::TILE + bx * PANEL, D / 2 + 32 * bx, row0, hq, b);
        bulk_commit();
        bulk_wait_read<1>();
        mbar_arrive(&bars->ds_free);
      }
      return w;
    };
    int n = 0;
    bool ok = true;
    for (int h = h0; ok && h < h0 + a.group; ++h) {
      const float* lse_base = it.lse + b * a.lse_b + h * a.lse_h;
      const float* dl_base = it.delta + b * a.lse_b + h * a.lse_h;
      TileCursor cur;
      for (int t; (t = cur.next(nqt, lane, qvis)) >= 0;) {
        const QTile qt = q_tile(gm, t, causal, nk, kmin, kmax);
        const int st = n & 1;
        // tensor row of the tile's first query (a tile never straddles two
        // segments when rows are addressed by position)
        const int qrow0 = static_cast<int>(slab_row(gm.qs, a.q_by_pos, qt.q0));
        // lse/delta of this tile into registers while the stage drains
        float lse_r[BM / 32], dl_r[BM / 32];
#pragma unroll
        for (int k = 0; k < BM / 32; ++k) {
          const int i = lane + 32 * k;
          lse_r[k] = i < qt.nq ? lse_base[qrow0 + i] : -INFINITY;
          dl_r[k] = i < qt.nq ? dl_base[qrow0 + i] : 0.f;
        }
        // Q stage st (and its lse/delta slot) is free once the MMAs of tile
        // n-2 have completed
        if (n >= 2 && !__all_sync(0xffffffffu, mbar_wait(&bars->q_empty[st], ((n - 2) >> 1) & 1, abort, status))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->q_full[st], L::TILE);
          for (int p = 0; p < D / 64; ++p)
            tma_load_4d(smem + L::Q_OFF + st * L::TILE + p * PANEL, mq, &bars->q_full[st], 64 * p, qrow0, h, b);
        }
        float* l2s = lse_sm + st * 2 * BM;
#pragma unroll
        for (int k = 0; k < BM / 32; ++k) {
          // -lse*log2(e), or -inf where P must be 0 (row past the slab, or a
          // row that sees no key at all), so exp2(s*scale*log2e + it) is P;
          // -scale*delta, so scale*(dP - delta) is one FMA
          const int i = lane + 32 * k;
          l2s[i] = lse_r[k] == -INFINITY ? -INFINITY : -lse_r[k] * kLog2e;
          l2s[BM + i] = -a.scale * dl_r[k];
        }
        mbar_arrive(&bars->q_full[st]);
        // dO stage st still holds half of tile n-2's dQ until its reduce has
        // read it
        if (n >= 2) {
          if (!reduce_tile(n - 2)) { ok = false; break; }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
        if (st) {
          q0_st1 = qrow0;
          h_st1 = h;
        } else {
          q0_st0 = qrow0;
          h_st0 = h;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars->do_full[st], L::TILE);
          for (int p = 0; p < D / 64; ++p)
            tma_load_4d(smem + L::DO_OFF + st * L::TILE + p * PANEL, mo, &bars->do_full[st], 64 * p, qrow0, h, b);
        }
        ++n;
      }
    }
    // the last two tiles' reduces
    for (int j = (n > 2 ? n - 2 : 0); ok && j < n; ++j) ok = reduce_tile(j);
    if (lane == 0) {
      bulk_wait_all();   // every reduce has read shared memory and landed in dq
      if (*abort) {
        mbar_wait_drain(&bars->kv_full, 0);
        for (int j = (n > 2 ? n - 2 : 0); j < n; ++j) {
          mbar_wait_drain(&bars->q_full[j & 1], (j >> 1) & 1);
          mbar_wait_drain(&bars->do_full[j & 1], (j >> 1) & 1);
        }
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and its waits, so every operand is
    // warp-uniform; one elected lane issues each MMA and commit.  It needs
    // only the count of visible tiles, not their rows.
    {
      auto wait_all = [&](uint64_t* bar, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, abort, status));
      };
      constexpr uint32_t idesc_dp = F16PV ? idesc_f16_f32(BN, BM, false, false)    // dP^T: M=keys, N=queries
                                          : idesc_bf16_f32(BN, BM, false, false);
      constexpr uint32_t idesc_s = idesc_f16_f32(BN, BM, false, false);      // S^T (fp16 K, Q)
      constexpr uint32_t idesc_dv = F16PV ? idesc_f16_f32(BN, D, false, true)      // dV: M=keys, N=D
                                          : idesc_bf16_f32(BN, D, false, true);
      constexpr uint32_t idesc_dk = idesc_f16_f32(BN, D, false, true);       // dK (fp16 dS^T, Q)
      constexpr uint32_t idesc_dq = idesc_f16_f32(BM, D, true, true);        // dQ: M=queries, N=D
      const uint32_t sK = smem_u32(smem + L::K_OFF), sV = smem_u32(smem + L::V_OFF);
      const uint32_t sDS = smem_u32(smem + L::DS_OFF);
      bool ok = wait_all(&bars->kv_full, 0);
      for (int n = 0; ok && n < n_vis; ++n) {
        const int st = n & 1;
        const uint32_t sQ = smem_u32(smem + L::Q_OFF + st * L::TILE);
        const uint32_t sO = smem_u32(smem + L::DO_OFF + st * L::TILE);
        // S^T = K Q^T over the S^T columns (the previous dV has read P^T);
        // K and Q must have been converted to fp16
        if (!wait_all(&bars->q_full[st], (n >> 1) & 1)) { ok = false; break; }
        if (n == 0 && !wait_all(&bars->k_conv, 0)) { ok = false; break; }
        if (!wait_all(&bars->q_conv, n & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kdk = sdesc_sw128(sK, 16, 1024), qdk = sdesc_sw128(sQ, 16, 1024);
        const uint64_t vdk = sdesc_sw128(sV, 16, 1024), odk = sdesc_sw128(sO, 16, 1024);
        const uint64_t odm = sdesc_sw128(sO, PANEL, 1024), qdm = sdesc_sw128(sQ, PANEL, 1024);
        const uint64_t sdm = sdesc_sw128(sDS, PANEL, 1024), kdm = sdesc_sw128(sK, PANEL, 1024);
        const uint32_t acc0 = n > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;
          umma_ss_w(tS, sdesc_step(kdk, off), sdesc_step(qdk, off), idesc_s, kk > 0 ? 1u : 0u);
        }
        umma_commit_w(&bars->s_full);
        // dP^T = V dO^T over the dP^T columns, which hold the previous dQ
        // until it is read back
        if (n > 0 && !wait_all(&bars->tmem_free, (n - 1) & 1)) { ok = false; break; }
        if (F16PV ? !wait_all(&bars->do_conv, n & 1)      // V, dO converted to fp16
                  : !wait_all(&bars->do_full[st], (n >> 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;
          umma_ss_w(tdP, sdesc_step(vdk, off), sdesc_step(odk, off), idesc_dp, kk > 0 ? 1u : 0u);
        }
        umma_commit_w(&bars->dp_full);
        // dV += P^T dO, then dK += dS^T Q (A from tensor memory).  Query
        // K-step kk = 4g + 2c + e lives in warpgroup g's packed columns
        // 64g + 16c + 8e and is ready once chunk c of both warpgroups is:
        // each product runs as two halves, chunk 0's K-steps first.
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!wait_all(&bars->p_half[c], n & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 4 * (q >> 1) + 2 * c + (q & 1);
            const uint32_t acol = 64 * (kk >> 2) + 8 * (kk & 3);
            umma_ts_w(tdV, tS + acol, sdesc_step(odm, kk * 2048), idesc_dv, kk > 0 ? 1u : acc0);
          }
        }
        if (!ok) break;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          if (!wait_all(&bars->ds_half[c], n & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kk = 4 * (q >> 1) + 2 * c + (q & 1);
            const uint32_t acol = 64 * (kk >> 2) + 8 * (kk & 3);
            umma_ts_w(tdK, tdP + acol, sdesc_step(qdm, kk * 2048), idesc_dk, kk > 0 ? 1u : acc0);
          }
        }
        if (!ok) break;
        // dQ = dS K over the dP^T columns (dK has read dS^T), N = D: A = the
        // dS panels (complete after chunk 1), B = K tile, MN-major, its
        // 64-column panels LBO apart
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          umma_ss_w(tdP, sdesc_step(sdm, kk * 2048), sdesc_step(kdm, kk * 2048), idesc_dq, kk > 0 ? 1u : 0u);
        }
        umma_commit_w(&bars->q_empty[st]);
        umma_commit_w(&bars->dq_full);
      }
      if (!ok) {
        umma_commit_w(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    // ----------------------------------- elementwise + read-back (warps 0-7)
    const int wg = warp >> 2;                 // query-column half
    const int qw = warp & 3;                  // lane quadrant
    const int row = qw * 32 + lane;           // key row (S^T) / query row (dQ)
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const bool krow_valid = row < nk;
    const int64_t kpos = krow_valid ? seg_pos(gm.ks, k0 + row) : INT64_MAX;
    const float sl2 = a.scale_log2;
    uint8_t* sds = smem + L::DS_OFF + wg * PANEL + (row >> 3) * 1024 + (row & 7) * 128;
    int n = 0;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->kv_full, 0, abort, status));
    // a finite input beyond the fp16 range would become +-inf: recorded as
    // SCA_ERR_RANGE (the kernel still runs to completion)
    bool range_bad = false;
    if (ok) {   // K (and V) to fp16; the two tiles are contiguous
      range_bad |= smem_bf16_to_f16<(F16PV ? 2 : 1) * L::TILE, 256>(smem + L::K_OFF, threadIdx.x);
      fence_async_smem();
    }
    mbar_arrive(&bars->k_conv);
    // Q of the j-th visible tile to fp16, once its TMA load has landed
    // (unless the caller passed fp16 queries)
    const bool q_is_f16 = (ta.f16_inputs & SCA_F16_Q) != 0, do_is_f16 = (ta.f16_inputs & SCA_F16_DOUT) != 0;
    auto convert_q = [&](int j) -> bool {
      const bool w = __all_sync(0xffffffffu, mbar_wait(&bars->q_full[j & 1], (j >> 1) & 1, abort, status));
      if (w && !q_is_f16) {
        range_bad |= smem_bf16_to_f16<L::TILE, 256>(smem + L::Q_OFF + (j & 1) * L::TILE, threadIdx.x);
        fence_async_smem();
      }
      mbar_arrive(&bars->q_conv);
      return w;
    };
    // dO of the j-th visible tile to fp16 (F16PV only)
    auto convert_do = [&](int j) -> bool {
      const bool w = __all_sync(0xffffffffu, mbar_wait(&bars->do_full[j & 1], (j >> 1) & 1, abort, status));
      if (w && !do_is_f16) {
        range_bad |= smem_bf16_to_f16<L::TILE, 256>(smem + L::DO_OFF + (j & 1) * L::TILE, threadIdx.x);
        fence_async_smem();
      }
      mbar_arrive(&bars->do_conv);
      return w;
    };
    if (ok) ok = convert_q(0);
    if constexpr (F16PV) {
      if (ok) ok = convert_do(0);
    }
    for (int hq = 0; ok && hq < a.group; ++hq) {   // each query head of the group in turn
      TileCursor cur;
      for (int t; ok && (t = cur.next(nqt, lane, qvis)) >= 0;) {
        const QTile qt = q_tile(gm, t, causal, nk, kmin, kmax);
        // -lse*log2e and -scale*delta of this warpgroup's 64 query columns (staged by warp 8)
        const float* nl2 = lse_sm + (n & 1) * 2 * BM + 64 * wg;
        const float* dls = nl2 + BM;
        // phase 1: P^T = exp2(s * scale * log2(e) - lse * log2(e)), kept in fp32
        // for phase 2 and written to tensor memory as bf16 for the dV MMAs
        bool w = mbar_wait(&bars->s_full, n & 1, abort, status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        uint32_t pr[64];   // S^T, then P^T (fp32 bits)
        tmem_ld32(tS + lane_off + 64 * wg, pr);
        tmem_ld32(tS + lane_off + 64 * wg + 32, pr + 32);
        // tiles that may hold masked pairs or ragged rows: bit j set when query
        // column 64*wg + j is visible to this thread's key (rows past the slab
        // already have lse = -inf, so P = 0 there)
        uint64_t vis = ~0ull;
        if (!qt.full) vis = krow_valid ? query_runs(gm.qs, qt.q0, qt.nq, causal, kpos, 64 * wg) : 0ull;
        tmem_wait_ld32(pr);
        tmem_wait_ld32(pr + 32);
        auto exps = [&](auto masked) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              const float4 l4 = *reinterpret_cast<const float4*>(nl2 + 32 * c + i);   // broadcast reads
              const float2 lp[2] = {make_float2(l4.x, l4.y), make_float2(l4.z, l4.w)};
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int j = 32 * c + i + 2 * u;
                const float2 x = ffma2(make_float2(__uint_as_float(pr[j]), __uint_as_float(pr[j + 1])),
                                       make_float2(sl2, sl2), lp[u]);
                float p0 = ex2(x.x), p1 = ex2(x.y);
                if (decltype(masked)::value) {
                  p0 = (vis >> j) & 1 ? p0 : 0.f;
                  p1 = (vis >> (j + 1)) & 1 ? p1 : 0.f;
                }
                pr[j] = __float_as_uint(p0);
                pr[j + 1] = __float_as_uint(p1);
                pk[(i + 2 * u) >> 1] = F16PV ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
              }
            }
            // over S^T columns this thread has already read
            tmem_st16(tS + lane_off + 64 * wg + 16 * c, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&bars->p_half[c]);
          }
        };
        if (qt.full)
          exps(std::false_type{});
        else
          exps(std::true_type{});
        // phase 2: dS^T = scale P^T (dP^T - delta), fp16, to tensor memory (A of
        // the dK MMAs) and to this warpgroup's dS panel (A of the dQ MMAs)
        // the dS panels hold half of the previous tile's dQ until its reduce
        // has read them
        w = mbar_wait(&bars->dp_full, n & 1, abort, status);
        if (w && n > 0) w = mbar_wait(&bars->ds_free, (n - 1) & 1, abort, status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        const float2 sc2 = make_float2(a.scale, a.scale);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dr[32];
          tmem_ld32(tdP + lane_off + 64 * wg + 32 * c, dr);
          tmem_wait_ld32(dr);
          uint32_t dk[16];
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            const float4 d4 = *reinterpret_cast<const float4*>(dls + 32 * c + i);
            const float2 dp[2] = {make_float2(d4.x, d4.y), make_float2(d4.z, d4.w)};
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = i + 2 * u;
              const float2 pp = make_float2(__uint_as_float(pr[32 * c + j]), __uint_as_float(pr[32 * c + j + 1]));
              const float2 d = fmul2(pp, ffma2(make_float2(__uint_as_float(dr[j]), __uint_as_float(dr[j + 1])), sc2, dp[u]));
              dk[j >> 1] = pack_f16x2(d.x, d.y);
            }
          }
          tmem_st16(tdP + lane_off + 64 * wg + 16 * c, dk);
          // dS^T row into shared memory (MN-major, 128B swizzle): chunk j of
          // 16 bytes holds queries 8j..8j+7 of this warpgroup's panel
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = 4 * c + u;
            uint4 v = make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
            *reinterpret_cast<uint4*>(sds + ((j ^ (row & 7)) << 4)) = v;
          }
          tmem_wait_st();
          if (c == 1) fence_async_smem();   // the whole dS panel, for the dQ MMAs
          tc_fence_before();
          mbar_arrive(&bars->ds_half[c]);
        }
        // the next tile's Q conversion overlaps this tile's dK/dQ MMAs
        if (n + 1 < n_vis && !convert_q(n + 1)) { ok = false; break; }
        // dQ read-back from the dP^T columns: thread = query row, warpgroup wg
        // takes columns [wg*D/2, (wg+1)*D/2).  Tensor memory is released before
        // the reduces are issued, so the next tile's dP^T never waits on them.
        w = mbar_wait(&bars->dq_full, n & 1, abort, status);
        if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
        tc_fence_after();
        uint32_t r[D / 2];
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) tmem_ld32(tdP + lane_off + wg * (D / 2) + c, r + c);
#pragma unroll
        for (int c = 0; c < D / 2; c += 32) tmem_wait_ld32(r + c);
        tc_fence_before();
        mbar_arrive(&bars->tmem_free);
        // dQ (already scaled through dS) staged for the producer's TMA
        // reduce-add over the dS panels (warpgroup 0) or this tile's dO
        // (warpgroup 1), both free since the dQ MMA ran: 32-column boxes of
        // 128 rows, 128B-swizzled like the reduce's map
        uint8_t* stg = smem + (wg == 0 ? L::DS_OFF : L::DO_OFF + (n & 1) * L::TILE) + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t* x = r + 32 * sub + 4 * j;
            *reinterpret_cast<uint4*>(stg + sub * PANEL + ((j ^ (row & 7)) << 4)) = make_uint4(x[0], x[1], x[2], x[3]);
          }
        }
        fence_async_smem();
        mbar_arrive(&bars->dq_staged[n & 1]);
        if constexpr (F16PV) {   // after the dQ read-back, which the next dP^T waits for anyway
          if (n + 1 < n_vis && !convert_do(n + 1)) { ok = false; break; }
        }
        ++n;
      }
    }
    if (range_bad) report(status, SCA_ERR_RANGE);
    // dK (warpgroup 0, already scaled through dS) and dV (warpgroup 1): thread = key row,
    // staged fp32 in 32-column 128B-swizzled boxes over the K/V tiles (dK)
    // and the Q stages (dV), free since the last MMA completed; one thread
    // per warpgroup then has the TMA unit add them into (accumulate) or
    // store them to global memory.  Key rows past the slab are skipped by
    // the TMA bounds.
    const bool epi = __all_sync(0xffffffffu, ok) && n > 0;
    if (epi) {
      tc_fence_after();
      const uint32_t src = (wg == 0 ? tdK : tdV) + lane_off;
      uint8_t* stg = smem + (wg == 0 ? L::K_OFF : L::Q_OFF) + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(src + c, r);
        tmem_wait_ld32(r);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(stg + (c / 32) * PANEL + ((j ^ (row & 7)) << 4)) =
              make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
      }
      fence_async_smem();
      mbar_arrive(&bars->epi_staged[wg]);
      if ((threadIdx.x & 127) == 0 && mbar_wait(&bars->epi_staged[wg], 0, abort, status)) {
        const CUtensorMap* m = &ta.maps[item_idx][wg == 0 ? 5 : 6];
        const int dkrow0 = static_cast<int>(slab_row(gm.ks, a.dkv_by_pos, k0));
        const uint8_t* base = smem + (wg == 0 ? L::K_OFF : L::Q_OFF);
#pragma unroll
        for (int bx = 0; bx < D / 32; ++bx) {
          if (a.accumulate)
            tma_reduce_add_4d(m, base + bx * PANEL, 32 * bx, dkrow0, hk, b);
          else
            tma_store_4d(m, base + bx * PANEL, 32 * bx, dkrow0, hk, b);
        }
        bulk_commit();
        bulk_wait_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool F16PV>
static cudaError_t launch(TcArgs& ta, cudaStream_t st) {
  using L = Layout<D>;
  static std::once_flag once[64];
  static cudaError_t attr_err[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::call_once(once[dev & 63], [&] {
    attr_err[dev & 63] =
        cudaFuncSetAttribute(bwd_tc_kernel<D, F16PV>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  });
  if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
  dim3 grid(ta.a.max_k_tiles, ta.a.B * ta.a.Hkv, ta.a.n_items);   // one CTA per key tile of a key/value head
  bwd_tc_kernel<D, F16PV><<<grid, kThreads, L::SMEM, st>>>(ta);
  return cudaGetLastError();
}

}  // namespace bwdtc

cudaError_t tc_backward(AttnArgs& a, int f16_inputs, cudaStream_t st) {
  using namespace bwdtc;
  static TcArgs ta;
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  // dq gathers contributions from every key tile through TMA reduce-adds:
  // in overwrite mode it starts from zero
  if (!a.accumulate) {
    if (a.o.s != a.D) return cudaErrorNotSupported;
    for (int i = 0; i < a.n_items; ++i) {
      const Item& it = a.items[i];
      if (it.Sq == 0) continue;
      // the item's dq rows: its slab, or each segment at its positions
      const int parts = a.q_by_pos ? it.qs.n : 1;
      for (int sgm = 0; sgm < parts; ++sgm) {
        const int64_t row0 = a.q_by_pos ? (sgm == 0 ? it.qs.start0 : it.qs.start1) : 0;
        const int64_t nrows = a.q_by_pos ? it.qs.len : it.Sq;
        for (int bb = 0; bb < a.B; ++bb) {
          const size_t width = static_cast<size_t>(nrows * a.D) * 4;
          const size_t pitch = a.H > 1 ? static_cast<size_t>(a.o.h) * 4 : width;   // one head: pitch unused
          if (pitch < width) return cudaErrorNotSupported;
          cudaError_t e = cudaMemset2DAsync(it.o + bb * a.o.b + row0 * a.D, pitch, 0, width,
                                            static_cast<size_t>(a.H), st);
          if (e != cudaSuccess) return e;
        }
      }
    }
  }
  // items are independent: launch them in groups that fit the parameters
  for (int first = 0; first < a.n_items; first += kItemsPerLaunch) {
    const int cnt = a.n_items - first < kItemsPerLaunch ? a.n_items - first : kItemsPerLaunch;
    ta.a = a;
    ta.f16_inputs = f16_inputs;
    ta.a.n_items = cnt;
    int64_t mt = 0;
    for (int i = 0; i < cnt; ++i) {
      const Item& it = a.items[first + i];
      ta.a.items[i] = it;
      const int64_t t = (it.Skv + BN - 1) / BN;
      if (t > mt) mt = t;
      CUtensorMap* m = ta.maps[i];
      cudaError_t e;
      const int64_t qr = slab_extent(it.qs, a.q_by_pos), kr = slab_extent(it.ks, a.kv_by_pos),
                    dkr = slab_extent(it.ks, a.dkv_by_pos);
      if ((e = (f16_inputs & SCA_F16_Q ? make_tmap_f16 : make_tmap_bf16)(&m[0], it.q, a.D, qr, a.H, a.B, a.q, 64,
                                                                            BM)) != cudaSuccess)
        return e;
      if ((e = make_tmap_bf16(&m[1], it.k, a.D, kr, a.Hkv, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
      if ((e = make_tmap_bf16(&m[2], it.v, a.D, kr, a.Hkv, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
      if ((e = (f16_inputs & SCA_F16_DOUT ? make_tmap_f16 : make_tmap_bf16)(&m[3], it.dout, a.D, qr, a.H, a.B, a.q,
                                                                               64, BM)) != cudaSuccess)
        return e;
      if ((e = make_tmap_f32(&m[4], it.o, a.D, qr, a.H, a.B, a.o, 32, BM)) != cudaSuccess) return e;
      if ((e = make_tmap_f32(&m[5], it.dk, a.D, dkr, a.Hkv, a.B, a.dkv, 32, BN)) != cudaSuccess) return e;
      if ((e = make_tmap_f32(&m[6], it.dv, a.D, dkr, a.Hkv, a.B, a.dkv, 32, BN)) != cudaSuccess) return e;
    }
    if (mt == 0) continue;
    ta.a.max_k_tiles = static_cast<int>(mt);
    const bool f16pv = a.group > 1;
    const cudaError_t e = a.D == 64 ? (f16pv ? launch<64, true>(ta, st) : launch<64, false>(ta, st))
                                    : (f16pv ? launch<128, true>(ta, st) : launch<128, false>(ta, st));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace sca
