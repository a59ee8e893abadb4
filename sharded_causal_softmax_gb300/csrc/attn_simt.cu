// fp32-arithmetic (SIMT) attention kernels: the forward partial, and the
// backward split into a query-stationary dq kernel and a key-stationary
// dk/dv kernel (no atomics: every CTA owns its output rows).  They serve the
// fp32-input path, where tensor-core TF32 would be too coarse, and act as an
// independent cross-check of the tensor-core kernels.
//
// Thread layout: 4 threads ("quad") per row; thread ql of the quad owns the
// float4 columns ql, ql+4, ql+8, ... so that the quad's shared-memory reads
// of one key row hit distinct banks.
#include <cmath>

#include "common.cuh"
#include "simt_launch.h"

namespace sca {

constexpr int kSimtThreads = 128;
constexpr int kSimtRows = 32;   // rows per CTA (4 threads each)
constexpr int kSimtKeys = 32;   // rows per shared-memory tile

template <typename T>
SCA_INLINE float4 load4(const T* p);

template <>
SCA_INLINE float4 load4<float>(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

template <>
SCA_INLINE float4 load4<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  return make_float4(__low2float(a), __high2float(a), __low2float(b), __high2float(b));
}

SCA_INLINE float dot4(const float4 a, const float4 b) { return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w; }

SCA_INLINE void axpy4(float4& y, float a, const float4 x) {
  y.x += a * x.x; y.y += a * x.y; y.z += a * x.z; y.w += a * x.w;
}

SCA_INLINE float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  return v;
}

// Cooperative load of `n` (<= kSimtKeys) rows of D columns into shared
// memory as fp32; rows past n are zero.
template <int D, typename T>
SCA_INLINE void load_rows(float4 (*dst)[D / 4], const T* base, int64_t row_stride, int n) {
  for (int e = threadIdx.x; e < kSimtKeys * (D / 4); e += kSimtThreads) {
    const int j = e / (D / 4), f = e % (D / 4);
    dst[j][f] = j < n ? load4<T>(base + j * row_stride + 4 * f) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// ------------------------------------------------------------------ forward

template <int D, typename T>
__global__ void __launch_bounds__(kSimtThreads) fwd_simt_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NF = D / 16;  // float4 per thread
  __shared__ float4 Ks[kSimtKeys][D / 4];
  __shared__ float4 Vs[kSimtKeys][D / 4];
  const Item& it = a.items[blockIdx.z];
  const int64_t q0 = static_cast<int64_t>(a.max_q_tiles - 1 - blockIdx.x) * kSimtRows;
  if (q0 >= it.Sq) return;
  const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
  const int ql = threadIdx.x & 3, rr = threadIdx.x >> 2;
  const int64_t qrow = q0 + rr;
  const bool valid = qrow < it.Sq;
  const int64_t qpos = valid ? seg_pos(it.qs, qrow) : INT64_MIN;
  const int nq = static_cast<int>(min64(kSimtRows, it.Sq - q0));
  int64_t qmin, qmax;
  tile_pos_range(it.qs, q0, nq, qmin, qmax);

  float4 qv[NF], acc[NF];
  const int64_t qr = slab_row(it.qs, a.q_by_pos, valid ? qrow : 0);   // tensor row
  const T* qp = static_cast<const T*>(it.q) + b * a.q.b + h * a.q.h + qr * a.q.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    qv[t] = load4<T>(qp + 4 * (ql + 4 * t));
    acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;
  const int hk = h / a.group;   // key/value head of this query head
  const T* kb = static_cast<const T*>(it.k) + b * a.kv.b + hk * a.kv.h;
  const T* vb = static_cast<const T*>(it.v) + b * a.kv.b + hk * a.kv.h;
  const int nkt = static_cast<int>((it.Skv + kSimtKeys - 1) / kSimtKeys);
  for (int kt = 0; kt < nkt; ++kt) {
    const int64_t k0 = static_cast<int64_t>(kt) * kSimtKeys;
    const int nk = static_cast<int>(min64(kSimtKeys, it.Skv - k0));
    int64_t kmin, kmax;
    tile_pos_range(it.ks, k0, nk, kmin, kmax);
    if (a.causal && kmin > qmax) continue;
    const bool full = nk == kSimtKeys && (!a.causal || kmax <= qmin);
    __syncthreads();
    const int64_t kr0 = slab_row(it.ks, a.kv_by_pos, k0);   // a tile never straddles segments
    load_rows<D, T>(Ks, kb + kr0 * a.kv.s, a.kv.s, nk);
    load_rows<D, T>(Vs, vb + kr0 * a.kv.s, a.kv.s, nk);
    __syncthreads();
#pragma unroll 1
    for (int j0 = 0; j0 < kSimtKeys; j0 += 8) {
      float s[8];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int j = j0 + u;
        float d = 0.f;
#pragma unroll
        for (int t = 0; t < NF; ++t) d += dot4(qv[t], Ks[j][ql + 4 * t]);
        d = quad_sum(d) * a.scale_log2;
        if (!full) {
          const bool vis = j < nk && (!a.causal || seg_pos(it.ks, k0 + j) <= qpos);
          if (!vis) d = -INFINITY;
        }
        s[u] = d;
        mx = fmaxf(mx, d);
      }
      const float m_new = fmaxf(m, mx);
      if (m_new == -INFINITY) continue;
      const float alpha = exp2f(m - m_new);
      m = m_new;
      l *= alpha;
#pragma unroll
      for (int t = 0; t < NF; ++t) {
        acc[t].x *= alpha; acc[t].y *= alpha; acc[t].z *= alpha; acc[t].w *= alpha;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float p = exp2f(s[u] - m);
        l += p;
#pragma unroll
        for (int t = 0; t < NF; ++t) axpy4(acc[t], p, Vs[j0 + u][ql + 4 * t]);
      }
    }
  }
  if (!valid) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* op = it.o + b * a.o.b + h * a.o.h + qr * a.o.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    const float4 r = make_float4(acc[t].x * inv, acc[t].y * inv, acc[t].z * inv, acc[t].w * inv);
    *reinterpret_cast<float4*>(op + 4 * (ql + 4 * t)) = r;
  }
  if (ql == 0) it.lse[b * a.lse_b + h * a.lse_h + qr] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ----------------------------------------------------------- backward: dq

template <int D, typename T>
__global__ void __launch_bounds__(kSimtThreads) dq_simt_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NF = D / 16;
  __shared__ float4 Ks[kSimtKeys][D / 4];
  __shared__ float4 Vs[kSimtKeys][D / 4];
  const Item& it = a.items[blockIdx.z];
  const int64_t q0 = static_cast<int64_t>(a.max_q_tiles - 1 - blockIdx.x) * kSimtRows;
  if (q0 >= it.Sq) return;
  const int b = blockIdx.y / a.H, h = blockIdx.y % a.H;
  const int ql = threadIdx.x & 3, rr = threadIdx.x >> 2;
  const int64_t qrow = q0 + rr;
  const bool valid = qrow < it.Sq;
  const int64_t qr = slab_row(it.qs, a.q_by_pos, valid ? qrow : 0);   // tensor row
  const int64_t qpos = valid ? seg_pos(it.qs, qrow) : INT64_MIN;
  const int nq = static_cast<int>(min64(kSimtRows, it.Sq - q0));
  int64_t qmin, qmax;
  tile_pos_range(it.qs, q0, nq, qmin, qmax);

  float4 qv[NF], dov[NF], acc[NF];
  const T* qp = static_cast<const T*>(it.q) + b * a.q.b + h * a.q.h + qr * a.q.s;
  const T* dp = static_cast<const T*>(it.dout) + b * a.q.b + h * a.q.h + qr * a.q.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    qv[t] = load4<T>(qp + 4 * (ql + 4 * t));
    dov[t] = load4<T>(dp + 4 * (ql + 4 * t));
    acc[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float lse = it.lse[b * a.lse_b + h * a.lse_h + qr];
  const float lse2 = lse * kLog2e;
  const float dlt = it.delta[b * a.lse_b + h * a.lse_h + qr];
  const bool row_live = valid && lse != -INFINITY;
  const int hk = h / a.group;   // key/value head of this query head
  const T* kb = static_cast<const T*>(it.k) + b * a.kv.b + hk * a.kv.h;
  const T* vb = static_cast<const T*>(it.v) + b * a.kv.b + hk * a.kv.h;
  const int nkt = static_cast<int>((it.Skv + kSimtKeys - 1) / kSimtKeys);
  for (int kt = 0; kt < nkt; ++kt) {
    const int64_t k0 = static_cast<int64_t>(kt) * kSimtKeys;
    const int nk = static_cast<int>(min64(kSimtKeys, it.Skv - k0));
    int64_t kmin, kmax;
    tile_pos_range(it.ks, k0, nk, kmin, kmax);
    if (a.causal && kmin > qmax) continue;
    __syncthreads();
    const int64_t kr0 = slab_row(it.ks, a.kv_by_pos, k0);   // a tile never straddles segments
    load_rows<D, T>(Ks, kb + kr0 * a.kv.s, a.kv.s, nk);
    load_rows<D, T>(Vs, vb + kr0 * a.kv.s, a.kv.s, nk);
    __syncthreads();
#pragma unroll 2
    for (int j = 0; j < kSimtKeys; ++j) {
      float s = 0.f, dpv = 0.f;
#pragma unroll
      for (int t = 0; t < NF; ++t) {
        s += dot4(qv[t], Ks[j][ql + 4 * t]);
        dpv += dot4(dov[t], Vs[j][ql + 4 * t]);
      }
      s = quad_sum(s);
      dpv = quad_sum(dpv);
      const bool vis = row_live && j < nk && (!a.causal || seg_pos(it.ks, k0 + j) <= qpos);
      const float p = vis ? exp2f(s * a.scale_log2 - lse2) : 0.f;
      const float ds = p * (dpv - dlt);
#pragma unroll
      for (int t = 0; t < NF; ++t) axpy4(acc[t], ds, Ks[j][ql + 4 * t]);
    }
  }
  if (!valid) return;
  float* out = it.o + b * a.o.b + h * a.o.h + qr * a.o.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    float4* p4 = reinterpret_cast<float4*>(out + 4 * (ql + 4 * t));
    float4 r = a.accumulate ? *p4 : make_float4(0.f, 0.f, 0.f, 0.f);
    axpy4(r, a.scale, acc[t]);
    *p4 = r;
  }
}

// -------------------------------------------------------- backward: dk, dv

template <int D, typename T>
__global__ void __launch_bounds__(kSimtThreads) dkv_simt_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int NF = D / 16;
  __shared__ float4 Qs[kSimtKeys][D / 4];
  __shared__ float4 Ds[kSimtKeys][D / 4];
  __shared__ float Ls[kSimtKeys], Dl[kSimtKeys];
  __shared__ int64_t Ps[kSimtKeys];
  const Item& it = a.items[blockIdx.z];
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * kSimtRows;
  if (k0 >= it.Skv) return;
  const int b = blockIdx.y / a.Hkv, hk = blockIdx.y % a.Hkv;   // a key/value head
  const int ql = threadIdx.x & 3, rr = threadIdx.x >> 2;
  const int64_t krow = k0 + rr;
  const bool valid = krow < it.Skv;
  const int64_t kr = slab_row(it.ks, a.kv_by_pos, valid ? krow : 0);   // tensor rows of k/v and dk/dv
  const int64_t dkr = slab_row(it.ks, a.dkv_by_pos, valid ? krow : 0);
  const int64_t kpos = valid ? seg_pos(it.ks, krow) : INT64_MAX;
  const int nk = static_cast<int>(min64(kSimtRows, it.Skv - k0));
  int64_t kmin, kmax;
  tile_pos_range(it.ks, k0, nk, kmin, kmax);

  float4 kv4[NF], vv4[NF], dk[NF], dv[NF];
  const T* kp = static_cast<const T*>(it.k) + b * a.kv.b + hk * a.kv.h + kr * a.kv.s;
  const T* vp = static_cast<const T*>(it.v) + b * a.kv.b + hk * a.kv.h + kr * a.kv.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    kv4[t] = load4<T>(kp + 4 * (ql + 4 * t));
    vv4[t] = load4<T>(vp + 4 * (ql + 4 * t));
    dk[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    dv[t] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int nqt = static_cast<int>((it.Sq + kSimtKeys - 1) / kSimtKeys);
  // every query head that reads this key/value head contributes
  for (int h = hk * a.group; h < (hk + 1) * a.group; ++h) {
    const T* qb = static_cast<const T*>(it.q) + b * a.q.b + h * a.q.h;
    const T* db = static_cast<const T*>(it.dout) + b * a.q.b + h * a.q.h;
    const float* lb = it.lse + b * a.lse_b + h * a.lse_h;
    const float* dlb = it.delta + b * a.lse_b + h * a.lse_h;
    for (int qt = 0; qt < nqt; ++qt) {
      const int64_t r0 = static_cast<int64_t>(qt) * kSimtKeys;
      const int nq = static_cast<int>(min64(kSimtKeys, it.Sq - r0));
      int64_t qmin, qmax;
      tile_pos_range(it.qs, r0, nq, qmin, qmax);
      if (a.causal && kmin > qmax) continue;
      __syncthreads();
      const int64_t qr0 = slab_row(it.qs, a.q_by_pos, r0);   // a tile never straddles segments
      load_rows<D, T>(Qs, qb + qr0 * a.q.s, a.q.s, nq);
      load_rows<D, T>(Ds, db + qr0 * a.q.s, a.q.s, nq);
      if (threadIdx.x < kSimtKeys) {
        const int i = threadIdx.x;
        const bool ok = i < nq;
        Ls[i] = ok ? lb[qr0 + i] : -INFINITY;
        Dl[i] = ok ? dlb[qr0 + i] : 0.f;
        Ps[i] = ok ? seg_pos(it.qs, r0 + i) : INT64_MIN;
      }
      __syncthreads();
#pragma unroll 2
      for (int i = 0; i < kSimtKeys; ++i) {
        float s = 0.f, dpv = 0.f;
#pragma unroll
        for (int t = 0; t < NF; ++t) {
          s += dot4(Qs[i][ql + 4 * t], kv4[t]);
          dpv += dot4(Ds[i][ql + 4 * t], vv4[t]);
        }
        s = quad_sum(s);
        dpv = quad_sum(dpv);
        const float lse = Ls[i];
        const bool vis = valid && lse != -INFINITY && (!a.causal || kpos <= Ps[i]);
        const float p = vis ? exp2f(s * a.scale_log2 - lse * kLog2e) : 0.f;
        const float ds = p * (dpv - Dl[i]);
#pragma unroll
        for (int t = 0; t < NF; ++t) {
          axpy4(dv[t], p, Ds[i][ql + 4 * t]);
          axpy4(dk[t], ds, Qs[i][ql + 4 * t]);
        }
      }
    }
  }
  if (!valid) return;
  float* dkp = it.dk + b * a.dkv.b + hk * a.dkv.h + dkr * a.dkv.s;
  float* dvp = it.dv + b * a.dkv.b + hk * a.dkv.h + dkr * a.dkv.s;
#pragma unroll
  for (int t = 0; t < NF; ++t) {
    float4* pk = reinterpret_cast<float4*>(dkp + 4 * (ql + 4 * t));
    float4* pv = reinterpret_cast<float4*>(dvp + 4 * (ql + 4 * t));
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 rk = a.accumulate ? *pk : z, rv = a.accumulate ? *pv : z;
    axpy4(rk, a.scale, dk[t]);
    axpy4(rv, 1.f, dv[t]);
    *pk = rk;
    *pv = rv;
  }
}

// ----------------------------------------------------------------- launch

static int max_tiles(const AttnArgs& a, bool keys, int tile) {
  int64_t m = 0;
  for (int i = 0; i < a.n_items; ++i) {
    const int64_t n = keys ? a.items[i].Skv : a.items[i].Sq;
    const int64_t t = (n + tile - 1) / tile;
    if (t > m) m = t;
  }
  return static_cast<int>(m);
}

template <int D, typename T>
static cudaError_t launch_fwd(AttnArgs& a, cudaStream_t st) {
  a.max_q_tiles = max_tiles(a, false, kSimtRows);
  dim3 grid(a.max_q_tiles, a.B * a.H, a.n_items);
  fwd_simt_kernel<D, T><<<grid, kSimtThreads, 0, st>>>(a);
  return cudaGetLastError();
}

template <int D, typename T>
static cudaError_t launch_bwd(AttnArgs& a, cudaStream_t st) {
  a.max_q_tiles = max_tiles(a, false, kSimtRows);
  a.max_k_tiles = max_tiles(a, true, kSimtRows);
  dim3 gq(a.max_q_tiles, a.B * a.H, a.n_items);
  dq_simt_kernel<D, T><<<gq, kSimtThreads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gk(a.max_k_tiles, a.B * a.Hkv, a.n_items);
  dkv_simt_kernel<D, T><<<gk, kSimtThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t simt_forward(AttnArgs& a, int dtype, cudaStream_t st) {
  if (dtype == SCA_BF16) return a.D == 64 ? launch_fwd<64, __nv_bfloat16>(a, st) : launch_fwd<128, __nv_bfloat16>(a, st);
  return a.D == 64 ? launch_fwd<64, float>(a, st) : launch_fwd<128, float>(a, st);
}

cudaError_t simt_backward(AttnArgs& a, int dtype, cudaStream_t st) {
  if (dtype == SCA_BF16) return a.D == 64 ? launch_bwd<64, __nv_bfloat16>(a, st) : launch_bwd<128, __nv_bfloat16>(a, st);
  return a.D == 64 ? launch_bwd<64, float>(a, st) : launch_bwd<128, float>(a, st);
}

}  // namespace sca
