// Forward (o, lse) partial on the 5th-generation tensor cores (sm_103a).
//
// One CTA owns a tile of 128 query rows of one (item, batch, head) and walks
// the item's visible key/value tiles of 128 rows:
//
//   warp 8      TMA producer for Q (once) and the K ring (3 stages)
//   warp 10     TMA producer for the V ring (2 stages)
//   warp 9      tensor-memory allocation, and the MMA loop, run by the
//               whole warp with one elected lane issuing each tcgen05.mma
//               (issued under if (lane == 0) the same loop took ~85 clk
//               per MMA and set the tile period):
//                 S[n%2] = Q K_n^T           (A = Q from tensor memory)
//                 O     += P_n V_n           (A = P from tensor memory)
//               QK^T runs up to two tiles ahead of the softmax.  Keeping Q
//               in tensor memory halves QK^T's shared-memory operand
//               traffic (reading Q from shared memory too measured 2%
//               slower, and 7% slower even with a third S buffer).
//   warps 0-7   softmax, two warpgroups: warpgroup g owns columns
//               [64g, 64g+64) of every S row, thread t of the warpgroup owns
//               query row t (tensor-memory lane t).  The row maximum is
//               combined across the two warpgroups through shared memory
//               while the exponentials are already computed against the
//               current reference maximum (redone only when it moves); each
//               thread sums its exponentials as two interleaved partial sums
//               (one serial add chain was on the tile's critical path), and
//               each warpgroup writes its half of P (bf16) over its own S
//               columns.  O is rescaled when
//               the maximum grows by more than 2^8 (lazy rescale, exact
//               after the final division).
//               Epilogue: o = O / l, lse = m + ln l.  o goes through the
//               spent K stages: each thread writes its row (16-byte chunks,
//               chunk index XOR (row & 7), so no bank conflicts), then each
//               warp store instruction writes whole 512-byte rows.  Storing
//               straight from the thread-per-row registers touched 32 rows
//               per warp instruction and took ~5800 clk per CTA.
//
// Tensor memory: S0, S1 in columns [0,256), O in [256, 256+D), Q in
// [256+D, 256+D+D/2); all 512 columns are allocated (one CTA per SM:
// shared memory use is above half the SM).  Tiles with no visible (query,
// key) pair are skipped; in tiles that may hold masked pairs or ragged rows
// each query's visible columns (at most two runs) are masked by key_runs.  Every
// mbarrier wait is bounded (ptx.cuh); on expiry the CTA records
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
constexpr int SBUF = 2;        // S buffers in tensor memory
constexpr int PANEL = 128 * 128;  // bytes of 128 rows x 64 bf16 (one 128B-swizzle panel column)
constexpr int kThreads = 352;  // 8 softmax warps + 3 role warps
constexpr int kProdK = 8, kMma = 9, kProdV = 10;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (log2 units)

struct Bars {
  uint64_t q_full;
  uint64_t q_tmem;       // Q copied into tensor memory by the softmax warps
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[SBUF], p_full[SBUF];
  uint64_t pv_done[2];   // PV_j completes phase j/2 of pv_done[j%2]
  uint64_t o_full;       // every PV has completed
  uint64_t red_full[2];  // both warpgroups published their row maxima (per tile parity)
  uint64_t lsum_full;    // both warpgroups published their row sums
  uint64_t o_staged;     // both warpgroups staged their half of o for the row stores
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float red[2][2][BM];   // row-max exchange [tile parity][warpgroup][row]
  float lsum[2][BM];     // final row sums of the two warpgroups
};

template <int D>
struct Layout {
  static constexpr int TILE = (D / 64) * PANEL;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;
  static constexpr int V_OFF = K_OFF + KST * TILE;
  static constexpr int BAR_OFF = V_OFF + VST * TILE;
  static constexpr int USED = BAR_OFF + static_cast<int>(sizeof(Bars));
  // keep one CTA per SM (tensor memory is allocated whole): above half the SM
  static constexpr int SMEM = (USED + 1024 > 120 * 1024 ? USED + 1024 : 120 * 1024);
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

SCA_INLINE TileInfo tile_info(const ItemGeom& g, int kt, bool causal, int64_t qmin, int64_t qmax) {
  TileInfo t;
  t.k0 = static_cast<int64_t>(kt) * BN;
  t.nk = static_cast<int>(min64(BN, g.Skv - t.k0));
  int64_t kmin, kmax;
  tile_pos_range(g.ks, t.k0, t.nk, kmin, kmax);
  t.visible = !causal || kmin <= qmax;
  t.full = t.nk == BN && (!causal || kmax <= qmin);
  return t;
}

// Walks the visible tiles like TileCursor, and also returns whether each is
// fully visible: both flags come from one pair of ballots per 32 tiles.
struct InfoCursor {
  int base = -32;
  uint32_t mask = 0, fmask = 0;
  template <typename Info>
  __device__ __forceinline__ int next(int n, int lane, const Info& info, bool& full) {
    while (mask == 0) {
      base += 32;
      if (base >= n) return -1;
      bool vis = false, fl = false;
      if (base + lane < n) {
        const TileInfo t = info(base + lane);
        vis = t.visible;
        fl = t.full;
      }
      mask = __ballot_sync(0xffffffffu, vis);
      fmask = __ballot_sync(0xffffffffu, fl);
    }
    const int b = __ffs(mask) - 1;
    full = (fmask >> b) & 1u;
    mask &= mask - 1;
    return base + b;
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ TcArgs ta) {
  using L = Layout<D>;
  const AttnArgs& a = ta.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + L::BAR_OFF);

  const int item_idx = blockIdx.z;
  const Item& it = a.items[item_idx];
  const ItemGeom gm = item_geom(it);
  const int64_t q0 = static_cast<int64_t>(a.max_q_tiles - 1 - blockIdx.x) * BM;  // heavy tiles first
  if (q0 >= gm.Sq) return;
  const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
  const int hk = h / a.group;   // key/value head of this query head
  const int nq = static_cast<int>(min64(BM, gm.Sq - q0));
  int64_t qmin, qmax;
  tile_pos_range(gm.qs, q0, nq, qmin, qmax);
  const int nkt = static_cast<int>((gm.Skv + BN - 1) / BN);
  const bool causal = a.causal != 0;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto kvis = [&](int kt) { return tile_info(gm, kt, causal, qmin, qmax).visible; };
  const int n_vis = count_tiles(nkt, lane, kvis);
  if (n_vis == 0) {
    // no visible key: the empty partial
    if (warp < 8) {
      const int row = (warp & 3) * 32 + lane, g = warp >> 2;
      if (row < nq) {
        const int64_t orow = slab_row(gm.qs, a.q_by_pos, q0 + row);
        float* op = it.o + b * a.o.b + h * a.o.h + orow * a.o.s + g * (D / 2);
        for (int c = 0; c < D / 2; c += 4) *reinterpret_cast<float4*>(op + c) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g == 0) it.lse[b * a.lse_b + h * a.lse_h + orow] = -INFINITY;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_tmem, 2 * BM);
    for (int i = 0; i < KST; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < SBUF; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 2 * BM);
    }
    mbar_init(&bars->pv_done[0], 1);
    mbar_init(&bars->pv_done[1], 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->red_full[0], 2 * BM);
    mbar_init(&bars->red_full[1], 2 * BM);
    mbar_init(&bars->lsum_full, 2 * BM);
    mbar_init(&bars->o_staged, 2 * BM);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kMma) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tO = tmem + SBUF * 128;
  const uint32_t tQ = tO + D;   // Q as the A operand of QK^T (bf16, 2 per column)
  volatile int* abort = &bars->abort;
  int* status = a.status;

  const uint32_t sK = smem_u32(smem + L::K_OFF);
  const uint32_t sV = smem_u32(smem + L::V_OFF);

  if (warp == kProdK) {
    // ------------------------------------------------ Q + K producer
    // lane 0 waits and issues; the warp walks the tile list together
    const CUtensorMap* mq = &ta.maps[item_idx][0];
    const CUtensorMap* mk = &ta.maps[item_idx][1];
    if (lane == 0) {
      tma_prefetch_map(mq);
      tma_prefetch_map(mk);
      mbar_arrive_expect_tx(&bars->q_full, L::TILE);
      for (int p = 0; p < D / 64; ++p)
        tma_load_4d(smem + L::Q_OFF + p * PANEL, mq, &bars->q_full, 64 * p,
                    static_cast<int>(slab_row(gm.qs, a.q_by_pos, q0)), h, b);
    }
    int n = 0;
    TileCursor cur;
    for (int kt; (kt = cur.next(nkt, lane, kvis)) >= 0;) {
      const int st = n % KST;
      int w = 0;
      if (lane == 0 && mbar_wait(&bars->k_empty[st], ((n / KST) & 1) ^ 1, abort, status)) {
        w = 1;
        mbar_arrive_expect_tx(&bars->k_full[st], L::TILE);
        for (int p = 0; p < D / 64; ++p)
          tma_load_4d(smem + L::K_OFF + st * L::TILE + p * PANEL, mk, &bars->k_full[st], 64 * p,
                      static_cast<int>(slab_row(gm.ks, a.kv_by_pos, static_cast<int64_t>(kt) * BN)), hk, b);
      }
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      ++n;
    }
    if (lane == 0 && *abort) {  // let issued copies land before the CTA goes away
      mbar_wait_drain(&bars->q_full, 0);
      for (int j = (n > KST ? n - KST : 0); j < n; ++j) mbar_wait_drain(&bars->k_full[j % KST], (j / KST) & 1);
    }
  } else if (warp == kProdV) {
    // ------------------------------------------------------ V producer
    const CUtensorMap* mv = &ta.maps[item_idx][2];
    if (lane == 0) tma_prefetch_map(mv);
    int n = 0;
    TileCursor cur;
    for (int kt; (kt = cur.next(nkt, lane, kvis)) >= 0;) {
      const int st = n % VST;
      int w = 0;
      if (lane == 0 && mbar_wait(&bars->v_empty[st], ((n / VST) & 1) ^ 1, abort, status)) {
        w = 1;
        mbar_arrive_expect_tx(&bars->v_full[st], L::TILE);
        for (int p = 0; p < D / 64; ++p)
          tma_load_4d(smem + L::V_OFF + st * L::TILE + p * PANEL, mv, &bars->v_full[st], 64 * p,
                      static_cast<int>(slab_row(gm.ks, a.kv_by_pos, static_cast<int64_t>(kt) * BN)), hk, b);
      }
      if (!__shfl_sync(0xffffffffu, w, 0)) break;
      ++n;
    }
    if (lane == 0 && *abort) {
      for (int j = (n > VST ? n - VST : 0); j < n; ++j) mbar_wait_drain(&bars->v_full[j % VST], (j / VST) & 1);
    }
  } else if (warp == kMma) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and its waits, so every operand is
    // warp-uniform; one elected lane issues each MMA and commit.
    {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, D, false, true);
      auto wait_all = [&](uint64_t* bar, uint32_t par) {
        return __all_sync(0xffffffffu, mbar_wait(bar, par, abort, status));
      };
      bool ok = wait_all(&bars->q_tmem, 0);
      auto issue_qk = [&](int j) -> bool {   // S[j%2] = Q K_j^T, Q from tensor memory
        const int ks = j % KST;
        if (!wait_all(&bars->k_full[ks], (j / KST) & 1)) return false;
        tc_fence_after();
        const uint32_t tS = tmem + (j % SBUF) * 128;
        const uint64_t kd = sdesc_sw128(sK + ks * L::TILE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * PANEL + (kk & 3) * 32;   // K-major: panel, then 32 B steps
          umma_ts_w(tS, tQ + kk * 8, sdesc_step(kd, off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit_w(&bars->s_full[j % SBUF]);
        umma_commit_w(&bars->k_empty[ks]);
        return true;
      };
      for (int j = 0; ok && j < n_vis && j < SBUF; ++j) ok = issue_qk(j);
      for (int j = 0; ok && j < n_vis; ++j) {
        // O += P_j V_j  (B = V tile, MN-major: 64-column panels LBO apart, 8-key groups 1024 B apart)
        const int vs = j % VST;
        if (!wait_all(&bars->p_full[j % SBUF], (j / SBUF) & 1)) { ok = false; break; }
        if (!wait_all(&bars->v_full[vs], (j / VST) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tP = tmem + (j % SBUF) * 128;
        const uint64_t vd = sdesc_sw128(sV + vs * L::TILE, PANEL, 1024);
        const uint32_t acc0 = j > 0 ? 1u : 0u;
        // keys [16kk, 16kk+16) of P live in warpgroup kk/4's packed columns
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_ts_w(tO, tP + 64 * (kk >> 2) + 8 * (kk & 3), sdesc_step(vd, kk * 2048), idesc_pv, kk > 0 ? 1u : acc0);
        umma_commit_w(&bars->v_empty[vs]);
        umma_commit_w(&bars->pv_done[j & 1]);
        // S[j%2] is free once PV_j has read P_j (MMAs execute in order)
        if (j + SBUF < n_vis) ok = issue_qk(j + SBUF);
      }
      if (ok) umma_commit_w(&bars->o_full);
      if (!ok) {  // make sure no MMA still writes tensor memory
        umma_commit_w(&bars->drain);
        mbar_wait_drain(&bars->drain, 0);
      }
    }
  } else {
    // -------------------------------------------- softmax (warps 0..7)
    const int g = warp >> 2;                 // column half
    const int qw = warp & 3;                 // lane quadrant
    const int row = qw * 32 + lane;          // query row == tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>(qw * 32) << 16;
    const bool row_valid = row < nq;
    const int64_t qpos = row_valid ? seg_pos(gm.qs, q0 + row) : -1;   // -1: no key, causal
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    int n = 0;
    // Q into tensor memory (the A operand of QK^T, so the MMAs read only K
    // from shared memory): warpgroup g copies dims [g*D/2, (g+1)*D/2) of its
    // row out of the 128B-swizzled TMA panels, two bf16 per column.
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, abort, status));
    if (ok) {
      constexpr int W = D / 4;                 // 32-bit words per half row
      uint32_t qr[W];
#pragma unroll
      for (int c = 0; c < W / 4; ++c) {        // 16-byte chunks of 8 dims
        const int d0 = g * (D / 2) + 8 * c;
        const uint8_t* src = smem + L::Q_OFF + (d0 / 64) * PANEL + (row >> 3) * 1024 + (row & 7) * 128;
        const uint4 v = *reinterpret_cast<const uint4*>(src + ((((d0 % 64) / 8) ^ (row & 7)) << 4));
        qr[4 * c] = v.x; qr[4 * c + 1] = v.y; qr[4 * c + 2] = v.z; qr[4 * c + 3] = v.w;
      }
      if constexpr (W == 32) tmem_st32(tQ + lane_off + g * (D / 4), qr);
      else tmem_st16(tQ + lane_off + g * (D / 4), qr);
      tmem_wait_st();
    }
    tc_fence_before();
    mbar_arrive(&bars->q_tmem);
    InfoCursor cur;
    auto kinfo = [&](int t) { return tile_info(gm, t, causal, qmin, qmax); };
    bool full_tile = false;
    for (int kt; ok && (kt = cur.next(nkt, lane, kinfo, full_tile)) >= 0;) {
      TileInfo ti;
      ti.full = full_tile;
      ti.k0 = static_cast<int64_t>(kt) * BN;
      ti.nk = static_cast<int>(min64(BN, gm.Skv - ti.k0));
      const int sb = n % SBUF;
      bool w = mbar_wait(&bars->s_full[sb], (n / SBUF) & 1, abort, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[64];
      const uint32_t tS = tmem + lane_off + sb * 128;
      tmem_ld32(tS + 64 * g, sr);
      tmem_ld32(tS + 64 * g + 32, sr + 32);
      tmem_wait_ld32(sr);
      tmem_wait_ld32(sr + 32);
      float* s = reinterpret_cast<float*>(sr);
      if (!ti.full) {
        // at most two runs of visible columns; one bit test and select per
        // column (a position test per column here cost 9% of the forward)
        const uint64_t vis = key_runs(gm.ks, ti.k0, ti.nk, causal, qpos, 64 * g);
        const uint32_t v0 = static_cast<uint32_t>(vis), v1 = static_cast<uint32_t>(vis >> 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (!(v0 & (1u << i))) s[i] = -INFINITY;
          if (!(v1 & (1u << i))) s[32 + i] = -INFINITY;
        }
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < 64; c += 4) {
        mx0 = fmaxf(mx0, s[c]); mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]); mx3 = fmaxf(mx3, s[c + 3]);
      }
      const float mine = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      bars->red[n & 1][g][row] = mine;
      mbar_arrive(&bars->red_full[n & 1]);
      // Optimistic exponentials against the current reference maximum while
      // the other half's maximum arrives; redone only when the reference
      // has to move (rare after the first tile).
      const float2 sc2 = make_float2(sl2, sl2);
      float2 sum = make_float2(0.f, 0.f);
      uint32_t pk[32];
      auto exps = [&](float m_ref) {
        const float msub = (m_ref == -INFINITY) ? 0.f : m_ref;
        const float2 nm2 = make_float2(-msub, -msub);
        // two partial sums, two column pairs per step: the sum's add chain
        // sat on the tile's critical path (this order measured 5% faster)
        float2 s0 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          // two columns per packed instruction: p = 2^(s * scale * log2e - m)
          const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sc2, nm2);
          const float2 y = ffma2(make_float2(s[2 * i + 2], s[2 * i + 3]), sc2, nm2);
          const float2 p = make_float2(ex2(x.x), ex2(x.y));
          const float2 q = make_float2(ex2(y.x), ex2(y.y));
          s0 = fadd2(s0, p);
          s1 = fadd2(s1, q);
          pk[i] = pack_bf16x2(p.x, p.y);
          pk[i + 1] = pack_bf16x2(q.x, q.y);
        }
        sum = fadd2(s0, s1);
      };
      exps(m_used);
      w = mbar_wait(&bars->red_full[n & 1], (n >> 1) & 1, abort, status);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      const float mt = fmaxf(mine, bars->red[n & 1][g ^ 1][row]) * sl2;
      const float m_new = fmaxf(m_used, mt);
      const bool need = m_new > m_used + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = need ? ex2(m_used - m_new) : 1.f;   // m_used = -inf gives 0
        if (need) m_used = m_new;
        l *= alpha;
        if (n > 0) {
          // S_n is complete, so QK_n and the PV_{n-2} issued before it are:
          // the phase this parity names on pv_done[(n-1)%2] is PV_{n-1}'s
          const bool w1 = mbar_wait(&bars->pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort, status);
          if (!__all_sync(0xffffffffu, w1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 2; c += 32) {
            uint32_t r[32];
            const uint32_t ta_o = tO + lane_off + g * (D / 2) + c;
            tmem_ld32(ta_o, r);
            tmem_wait_ld32(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(ta_o, r);
          }
        }
        exps(m_used);   // against the moved reference
      }
      // P (bf16) over this half's own S columns [64g, 64g+32): no other
      // warpgroup reads them, so no ordering with the other half is needed
      tmem_st32(tS + 64 * g, pk);
      l += sum.x + sum.y;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[sb]);
      ++n;
    }
    // epilogue: every PV has completed
    if (ok) ok = mbar_wait(&bars->o_full, 0, abort, status);
    bars->lsum[g][row] = l;
    mbar_arrive(&bars->lsum_full);
    if (ok) ok = mbar_wait(&bars->lsum_full, 0, abort, status);
    const float l_tot = l + bars->lsum[g ^ 1][row];
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
      // o = O / l staged over the K stages (every QK^T has completed): row r
      // at r * D * 4 bytes, logical 16-byte chunk q at physical chunk
      // q ^ (r & 7)
      constexpr int CH = D / 4;                  // 16-byte chunks per row
      uint8_t* stg = smem + L::K_OFF;
      uint8_t* mine = stg + row * (D * 4);
#pragma unroll 1
      for (int c = 0; c < D / 2; c += 32) {
        uint32_t r[32];
        tmem_ld32(tO + lane_off + g * (D / 2) + c, r);
        tmem_wait_ld32(r);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int q = (g * (D / 2) + c) / 4 + j;
          const uint4 v = make_uint4(__float_as_uint(__uint_as_float(r[4 * j]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * j + 1]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * j + 2]) * inv),
                                     __float_as_uint(__uint_as_float(r[4 * j + 3]) * inv));
          *reinterpret_cast<uint4*>(mine + ((q ^ (row & 7)) << 4)) = v;
        }
      }
      if (row_valid && g == 0) {
        const int64_t orow = slab_row(gm.qs, a.q_by_pos, q0 + row);
        it.lse[b * a.lse_b + h * a.lse_h + orow] = l_tot > 0.f ? (m_used + log2f(l_tot)) * kLn2 : -INFINITY;
      }
      mbar_arrive(&bars->o_staged);
      // warp w stores rows [16w, 16w + 16): one whole row (D = 128) or two
      // (D = 64) per instruction
      if (__all_sync(0xffffffffu, mbar_wait(&bars->o_staged, 0, abort, status))) {
        constexpr int RPI = 32 / CH;
        const int sub = lane / CH, li = lane % CH;
        float* obase = it.o + b * a.o.b + h * a.o.h;
#pragma unroll 4
        for (int i = 0; i < 16; i += RPI) {
          const int r = 16 * warp + i + sub;
          if (r < nq) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + r * (D * 4) + ((li ^ (r & 7)) << 4));
            const int64_t orow = slab_row(gm.qs, a.q_by_pos, q0 + r);
            *reinterpret_cast<uint4*>(obase + orow * a.o.s + 4 * li) = v;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMma) {
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
  static TcArgs ta;  // large; filled per call on the host (the launch copies it)
  static std::mutex mu;
  std::lock_guard<std::mutex> g(mu);
  int64_t mt = 0;
  for (int i = 0; i < a.n_items; ++i) {
    const Item& it = a.items[i];
    const int64_t t = (it.Sq + BM - 1) / BM;
    if (t > mt) mt = t;
    cudaError_t e;
    const int64_t q_rows = slab_extent(it.qs, a.q_by_pos), kv_rows = slab_extent(it.ks, a.kv_by_pos);
    if ((e = make_tmap_bf16(&ta.maps[i][0], it.q, a.D, q_rows, a.H, a.B, a.q, 64, BM)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&ta.maps[i][1], it.k, a.D, kv_rows, a.Hkv, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
    if ((e = make_tmap_bf16(&ta.maps[i][2], it.v, a.D, kv_rows, a.Hkv, a.B, a.kv, 64, BN)) != cudaSuccess) return e;
  }
  a.max_q_tiles = static_cast<int>(mt);
  ta.a = a;
  return a.D == 64 ? launch<64>(ta, st) : launch<128>(ta, st);
}

}  // namespace sca
