// Shared device/host definitions of libsca: item parameters passed to the
// kernels, segment position arithmetic, status reporting.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "sca.h"

#define SCA_INLINE __device__ __forceinline__

namespace sca {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Segment map of a slab of rows (mirror of sca_segs, device friendly).
struct Segs {
  int64_t len;
  int64_t start0, start1;
  int32_t n;
};

inline Segs to_segs(const sca_segs& s) {
  Segs d;
  d.len = s.len;
  d.start0 = s.start[0];
  d.start1 = s.n > 1 ? s.start[1] : 0;
  d.n = s.n;
  return d;
}

// Global position of slab row i.
__host__ __device__ __forceinline__ int64_t seg_pos(const Segs& s, int64_t i) {
  return i < s.len ? s.start0 + i : s.start1 + (i - s.len);
}

// Tensor row of slab row i: i itself, or its global position when the
// tensor is addressed by position (natural order).
__host__ __device__ __forceinline__ int64_t slab_row(const Segs& s, bool by_pos, int64_t i) {
  return by_pos ? seg_pos(s, i) : i;
}

// Rows a tensor must span to hold a slab of n*len rows: n*len, or past the
// last global position when addressed by position.
__host__ __device__ __forceinline__ int64_t slab_extent(const Segs& s, bool by_pos) {
  if (!by_pos) return static_cast<int64_t>(s.n) * s.len;
  const int64_t e0 = s.start0 + s.len, e1 = s.n > 1 ? s.start1 + s.len : 0;
  return e0 > e1 ? e0 : e1;
}

// Positions of a tile of slab rows [r0, r0 + cnt) (cnt >= 1, at most two
// segment parts): min and max global position.
__host__ __device__ __forceinline__ void tile_pos_range(const Segs& s, int64_t r0, int64_t cnt,
                                                        int64_t& pmin, int64_t& pmax) {
  const int64_t r1 = r0 + cnt - 1;
  if (r1 < s.len || r0 >= s.len) {           // one part: positions increase
    pmin = seg_pos(s, r0);
    pmax = seg_pos(s, r1);
  } else {                                   // straddles the two segments
    const int64_t a0 = s.start0 + r0, a1 = s.start0 + s.len - 1;
    const int64_t b0 = s.start1, b1 = s.start1 + (r1 - s.len);
    pmin = a0 < b0 ? a0 : b0;
    pmax = a1 > b1 ? a1 : b1;
  }
}

// Bits [lo, hi) of a 64-bit word, the bounds clamped to [0, 64].
__host__ __device__ __forceinline__ uint64_t run_bits(int64_t lo, int64_t hi) {
  lo = lo < 0 ? 0 : (lo > 64 ? 64 : lo);
  hi = hi < 0 ? 0 : (hi > 64 ? 64 : hi);
  if (hi <= lo) return 0;
  const uint64_t below_hi = hi == 64 ? ~0ull : ((1ull << hi) - 1);
  return below_hi & ~((1ull << lo) - 1);
}

// Key columns c0 + j (j < 64) of the tile of slab rows [k0, k0 + nk) that a
// query at global position qpos (-1: none, under the causal mask) may see:
// bit j set when c0 + j < nk and, causal, the key's position <= qpos.  The
// tile's rows in segment part 0 are columns c < cb (position start0 + k0 + c),
// those in part 1 columns c >= cb (position start1 + k0 + c - len); positions
// rise within each part, so each part's visible columns form one run.
__host__ __device__ __forceinline__ uint64_t key_runs(const Segs& ks, int64_t k0, int64_t nk, bool causal,
                                                      int64_t qpos, int64_t c0) {
  const int64_t cb = ks.len - k0 < 0 ? 0 : min64(ks.len - k0, nk);
  int64_t a_hi = cb, b_hi = nk;
  if (causal) {
    a_hi = min64(a_hi, qpos - ks.start0 - k0 + 1);
    b_hi = min64(b_hi, qpos - ks.start1 - k0 + ks.len + 1);
  }
  return run_bits(-c0, a_hi - c0) | run_bits(cb - c0, b_hi - c0);
}

// Query columns c0 + j (j < 64) of the tile of slab rows [q0, q0 + nq) that
// a key at global position kpos may be seen by: bit j set when c0 + j < nq
// and, causal, the query's position >= kpos.  The mirror of key_runs: each
// segment part's visible columns form one run, here a suffix of the part.
__host__ __device__ __forceinline__ uint64_t query_runs(const Segs& qs, int64_t q0, int64_t nq, bool causal,
                                                        int64_t kpos, int64_t c0) {
  const int64_t cb = qs.len - q0 < 0 ? 0 : min64(qs.len - q0, nq);
  int64_t a_lo = 0, b_lo = cb;
  if (causal) {
    const int64_t a = kpos - qs.start0 - q0, b = kpos - qs.start1 - q0 + qs.len;
    a_lo = a > a_lo ? a : a_lo;
    b_lo = b > b_lo ? b : b_lo;
  }
  return run_bits(a_lo - c0, cb - c0) | run_bits(b_lo - c0, nq - c0);
}

// Walks, in order, the tiles t in [0, n) for which vis(t) holds, testing 32
// candidates per warp-wide ballot.  All 32 lanes of a warp call next()
// together with the same arguments; it returns -1 after the last tile.
struct TileCursor {
  int base = -32;
  uint32_t mask = 0;
  template <typename Vis>
  __device__ __forceinline__ int next(int n, int lane, const Vis& vis) {
    while (mask == 0) {
      base += 32;
      if (base >= n) return -1;
      mask = __ballot_sync(0xffffffffu, base + lane < n && vis(base + lane));
    }
    const int t = base + __ffs(mask) - 1;
    mask &= mask - 1;
    return t;
  }
};

// Number of t in [0, n) with vis(t), by warp-wide ballots (all lanes call).
template <typename Vis>
__device__ __forceinline__ int count_tiles(int n, int lane, const Vis& vis) {
  int c = 0;
  for (int base = 0; base < n; base += 32)
    c += __popc(__ballot_sync(0xffffffffu, base + lane < n && vis(base + lane)));
  return c;
}

// Per-item data of an attention launch (forward and backward share it).
struct Item {
  const void* q;
  const void* k;
  const void* v;
  const void* dout;   // backward only
  float* o;           // forward: o partial; backward: dq
  float* lse;         // forward: lse out; backward: final lse (read)
  const float* delta; // backward only
  float* dk;
  float* dv;
  Segs qs, ks;
  int64_t Sq, Skv;
};

struct View {
  int64_t b, h, s;
};

// The position geometry of one item, copied once per CTA out of the kernel
// parameters into registers: read in place, behind the dynamic item index,
// every use is a constant-cache load, and the tile loops make hundreds.
struct ItemGeom {
  Segs qs, ks;
  int64_t Sq, Skv;
};
SCA_INLINE ItemGeom item_geom(const Item& it) {
  ItemGeom g;
  g.qs = it.qs;
  g.ks = it.ks;
  g.Sq = it.Sq;
  g.Skv = it.Skv;
  return g;
}

struct AttnArgs {
  Item items[SCA_MAX_ITEMS];
  View q, kv, o, dkv;
  int64_t lse_b, lse_h;
  int32_t n_items, B, H, D;
  int32_t causal;
  int32_t accumulate; // backward: add into dq/dk/dv (1) or overwrite (0)
  float scale;        // natural-units score scale
  float scale_log2;   // scale * log2(e)
  int32_t max_q_tiles;
  int32_t max_k_tiles;
  int32_t q_by_pos, kv_by_pos, dkv_by_pos;   // row addressing (see sca_attn_dims)
  int32_t Hkv, group;   // key/value heads; query heads per key/value head
  int* status;
};

// First device-side failure wins; never traps.
SCA_INLINE void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Does either bf16 half of w hold a finite value beyond the fp16 range?
// bf16 magnitudes from 0x4780 (65536) up to 0x7f7f (the largest finite)
// round to +-inf in fp16; 0x477f (65280) and below convert exactly or to
// fp16 subnormals; +-inf and NaN stay what they are.
SCA_INLINE bool bf16x2_beyond_f16(uint32_t w) {
  const uint32_t lo = w & 0x7fffu, hi = (w >> 16) & 0x7fffu;
  return (lo - 0x4780u < 0x7f80u - 0x4780u) | (hi - 0x4780u < 0x7f80u - 0x4780u);
}

SCA_INLINE float to_f32(float x) { return x; }
SCA_INLINE float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

}  // namespace sca
