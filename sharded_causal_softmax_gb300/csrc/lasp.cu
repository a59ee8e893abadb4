// Causal linear attention over P contiguous shards (linear attention
// sequence parallelism: "Effiziente Parallelisierung linearer
// Aufmerksamkeitssequenzen fuer skalierbare Sprachmodelle" - intermediate
// states exchanged point to point between shards, the right-product trick).
//
//   o_t = scale * sum_{s <= t} (q_t . k_s) v_s
//
// The sequence is taken in blocks of kBlk = 64 rows.  Forward:
//   1. lasp_block_states: st_j = K_j^T V_j (D x D fp32) for every block j.
//   2. lasp_scan: within each shard, st_j := sum of st_i over the shard's
//      blocks before j (exclusive prefix); the shard's total is written out.
//   3. lasp_exchange: the point-to-point pass, hop by hop along the ring:
//      in_r = in_{r-1} + total_{r-1}.
//   4. lasp_fwd: o_j = scale * (Q_j (st_j + in_r) + tril(Q_j K_j^T) V_j).
// Backward: the same with st'_j = Q_j^T dO_j, suffix scan and the reverse
// pass, then dq from the forward states and dk, dv from the backward ones.
//
// Everything is fp32 arithmetic on the CUDA cores: without normalisation
// the outputs grow like sqrt(t) and a state rounded to a tensor-core input
// type would cost ~2^-9 of them.  Shared-memory matrices keep an odd row
// stride (cols + 1), and a thread (ti, tj) of the 16 x 16 grid owns rows
// ti*RM .. ti*RM+RM-1 and columns tj, tj+16, ...: row-wise and column-wise
// operand reads are then free of bank conflicts.
#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "lasp_tc.h"

namespace sca {
namespace lasp {

constexpr int kBlk = 64;
constexpr int kThreads = 256;

template <typename T>
SCA_INLINE float ld(const T* p) { return to_f32(*p); }

// fp32 rows [rows][cols] of a row-contiguous tensor into shared memory with
// row stride cols + 1.
template <int COLS, typename T>
SCA_INLINE void load_block(float* dst, const T* src, int rows) {
  for (int e = threadIdx.x; e < rows * COLS; e += kThreads) {
    const int r = e / COLS, c = e % COLS;
    dst[r * (COLS + 1) + c] = ld(src + static_cast<int64_t>(r) * COLS + c);
  }
}

// a D x D state (optionally the sum of two) into shared memory, stride D + 1
template <int D>
SCA_INLINE void load_state(float* dst, const float* a, const float* b) {
  for (int e = threadIdx.x; e < D * D; e += kThreads) {
    const int r = e / D, c = e % D;
    dst[r * (D + 1) + c] = a[e] + (b ? b[e] : 0.f);
  }
}

// acc[i][u] += sum_k A(m0 + i, k) * B(k, tj + 16 u), A and B in shared
// memory, each read row-major (X[row * ld + col]) or transposed.
template <int RM, int RN, bool AT, bool BT>
SCA_INLINE void gemm_acc(float (&acc)[RM][RN], const float* A, int lda, const float* B, int ldb, int K, int m0,
                         int tj) {
#pragma unroll 4
  for (int k = 0; k < K; ++k) {
    float a[RM], b[RN];
#pragma unroll
    for (int i = 0; i < RM; ++i) a[i] = AT ? A[k * lda + m0 + i] : A[(m0 + i) * lda + k];
#pragma unroll
    for (int u = 0; u < RN; ++u) {
      const int n = tj + 16 * u;
      b[u] = BT ? B[n * ldb + k] : B[k * ldb + n];
    }
#pragma unroll
    for (int i = 0; i < RM; ++i)
#pragma unroll
      for (int u = 0; u < RN; ++u) acc[i][u] = fmaf(a[i], b[u], acc[i][u]);
  }
}

template <int RM, int RN>
SCA_INLINE void zero(float (&acc)[RM][RN]) {
#pragma unroll
  for (int i = 0; i < RM; ++i)
#pragma unroll
    for (int u = 0; u < RN; ++u) acc[i][u] = 0.f;
}

// the masked kBlk x kBlk product (row t, column s kept when s <= t) into
// shared memory, stride kBlk + 1
template <int D, bool BT>
SCA_INLINE void masked_product(float* out, const float* A, const float* B, int ti, int tj) {
  float c[4][4];
  zero(c);
  gemm_acc<4, 4, false, BT>(c, A, D + 1, B, D + 1, D, 4 * ti, tj);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = 4 * ti + i, s = tj + 16 * u;
      out[t * (kBlk + 1) + s] = s <= t ? c[i][u] : 0.f;
    }
}

template <int RN>
SCA_INLINE void store_rows(float* dst, const float (&acc)[4][RN], int m0, int tj, float mul, int D) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int u = 0; u < RN; ++u) dst[static_cast<int64_t>(m0 + i) * D + tj + 16 * u] = mul * acc[i][u];
}

// ------------------------------------------------------------------ kernels

// st[bh][j] = A_j^T B_j over the kBlk rows of block j.
template <int D, typename T>
__global__ void __launch_bounds__(kThreads) states_kernel(const T* a, const T* b, float* st, int64_t S) {
  extern __shared__ float sm[];
  float* As = sm;
  float* Bs = sm + kBlk * (D + 1);
  const int j = blockIdx.x, bh = blockIdx.y;
  const int64_t row0 = static_cast<int64_t>(bh) * S + static_cast<int64_t>(j) * kBlk;
  load_block<D>(As, a + row0 * D, kBlk);
  load_block<D>(Bs, b + row0 * D, kBlk);
  __syncthreads();
  constexpr int R = D / 16;
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  float c[R][R];
  zero(c);
  gemm_acc<R, R, true, false>(c, As, D + 1, Bs, D + 1, kBlk, R * ti, tj);   // A^T: element (i, r) = A[r][i]
  float* out = st + (static_cast<int64_t>(bh) * (S / kBlk) + j) * D * D;
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int u = 0; u < R; ++u) out[(R * ti + i) * D + tj + 16 * u] = c[i][u];
}

// Exclusive prefix (reverse: suffix) of the states over each shard's blocks,
// in place; the shard's total into tot[bh][r].
__global__ void scan_kernel(float* st, float* tot, int64_t nblk, int DD, int P, int reverse) {
  const int e4 = blockIdx.x * blockDim.x + threadIdx.x;   // four consecutive entries per thread
  const int DD4 = DD / 4;
  if (e4 >= DD4) return;
  const int bh = blockIdx.y, r = blockIdx.z;
  const int64_t nb = nblk / P;
  float4* base = reinterpret_cast<float4*>(st + (static_cast<int64_t>(bh) * nblk + r * nb) * DD) + e4;
  float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
  // eight independent 16-byte loads in flight, then their exclusive prefix
  for (int64_t i0 = 0; i0 < nb; i0 += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u, j = reverse ? nb - 1 - i : i;
      v[u] = i < nb ? base[j * DD4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t i = i0 + u, j = reverse ? nb - 1 - i : i;
      if (i < nb) base[j * DD4] = run;
      run.x += v[u].x;
      run.y += v[u].y;
      run.z += v[u].z;
      run.w += v[u].w;
    }
  }
  reinterpret_cast<float4*>(tot + (static_cast<int64_t>(bh) * P + r) * DD)[e4] = run;
}

// The pass of states along the ring of shards, one hop at a time.
__global__ void exchange_kernel(const float* tot, float* in, int DD, int P, int reverse) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= DD) return;
  const int64_t bh = blockIdx.y;
  float run = 0.f;   // what the current shard receives from its neighbour
  for (int i = 0; i < P; ++i) {
    const int r = reverse ? P - 1 - i : i;
    in[(bh * P + r) * DD + e] = run;
    run += tot[(bh * P + r) * DD + e];
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) fwd_kernel(const T* q, const T* k, const T* v, const float* st,
                                                       const float* sin, float* o, int64_t S, int P, float scale) {
  extern __shared__ float sm[];
  float* Ss = sm;                           // [D][D + 1]
  float* Qs = Ss + D * (D + 1);             // [kBlk][D + 1]
  float* Ks = Qs + kBlk * (D + 1);
  float* Vs = Ks + kBlk * (D + 1);
  float* Ms = Vs + kBlk * (D + 1);          // [kBlk][kBlk + 1]
  const int j = blockIdx.x, bh = blockIdx.y;
  const int64_t nblk = S / kBlk;
  const int r = static_cast<int>(j / (nblk / P));
  const int64_t row0 = static_cast<int64_t>(bh) * S + static_cast<int64_t>(j) * kBlk;
  load_state<D>(Ss, st + (static_cast<int64_t>(bh) * nblk + j) * D * D, sin + (static_cast<int64_t>(bh) * P + r) * D * D);
  load_block<D>(Qs, q + row0 * D, kBlk);
  load_block<D>(Ks, k + row0 * D, kBlk);
  load_block<D>(Vs, v + row0 * D, kBlk);
  __syncthreads();
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  constexpr int RN = D / 16;
  float acc[4][RN];
  zero(acc);
  gemm_acc<4, RN, false, false>(acc, Qs, D + 1, Ss, D + 1, D, 4 * ti, tj);   // Q (state before the block)
  masked_product<D, true>(Ms, Qs, Ks, ti, tj);                                // tril(Q K^T)
  __syncthreads();
  gemm_acc<4, RN, false, false>(acc, Ms, kBlk + 1, Vs, D + 1, kBlk, 4 * ti, tj);
  store_rows(o + row0 * D, acc, 4 * ti, tj, scale, D);
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) dq_kernel(const T* k, const T* v, const T* dout, const float* st,
                                                      const float* sin, float* dq, int64_t S, int P, float scale) {
  extern __shared__ float sm[];
  float* Ss = sm;
  float* Os = Ss + D * (D + 1);             // dO
  float* Ks = Os + kBlk * (D + 1);
  float* Vs = Ks + kBlk * (D + 1);
  float* Ms = Vs + kBlk * (D + 1);
  const int j = blockIdx.x, bh = blockIdx.y;
  const int64_t nblk = S / kBlk;
  const int r = static_cast<int>(j / (nblk / P));
  const int64_t row0 = static_cast<int64_t>(bh) * S + static_cast<int64_t>(j) * kBlk;
  load_state<D>(Ss, st + (static_cast<int64_t>(bh) * nblk + j) * D * D, sin + (static_cast<int64_t>(bh) * P + r) * D * D);
  load_block<D>(Os, dout + row0 * D, kBlk);
  load_block<D>(Ks, k + row0 * D, kBlk);
  load_block<D>(Vs, v + row0 * D, kBlk);
  __syncthreads();
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  constexpr int RN = D / 16;
  float acc[4][RN];
  zero(acc);
  gemm_acc<4, RN, false, true>(acc, Os, D + 1, Ss, D + 1, D, 4 * ti, tj);     // dO (state)^T
  masked_product<D, true>(Ms, Os, Vs, ti, tj);                                // tril(dO V^T)
  __syncthreads();
  gemm_acc<4, RN, false, false>(acc, Ms, kBlk + 1, Ks, D + 1, kBlk, 4 * ti, tj);
  store_rows(dq + row0 * D, acc, 4 * ti, tj, scale, D);
}

template <int D, typename T>
__global__ void __launch_bounds__(kThreads) dkdv_kernel(const T* q, const T* k, const T* v, const T* dout,
                                                        const float* st, const float* sin, float* dk, float* dv,
                                                        int64_t S, int P, float scale) {
  extern __shared__ float sm[];
  float* Gs = sm;                           // backward state: sum of q^T dO after the block
  float* Qs = Gs + D * (D + 1);
  float* Ks = Qs + kBlk * (D + 1);
  float* Vs = Ks + kBlk * (D + 1);
  float* Os = Vs + kBlk * (D + 1);
  float* Ms = Os + kBlk * (D + 1);
  const int j = blockIdx.x, bh = blockIdx.y;
  const int64_t nblk = S / kBlk;
  const int r = static_cast<int>(j / (nblk / P));
  const int64_t row0 = static_cast<int64_t>(bh) * S + static_cast<int64_t>(j) * kBlk;
  load_state<D>(Gs, st + (static_cast<int64_t>(bh) * nblk + j) * D * D, sin + (static_cast<int64_t>(bh) * P + r) * D * D);
  load_block<D>(Qs, q + row0 * D, kBlk);
  load_block<D>(Ks, k + row0 * D, kBlk);
  load_block<D>(Vs, v + row0 * D, kBlk);
  load_block<D>(Os, dout + row0 * D, kBlk);
  __syncthreads();
  const int ti = threadIdx.x / 16, tj = threadIdx.x % 16;
  constexpr int RN = D / 16;
  float ak[4][RN], av[4][RN];
  zero(ak);
  zero(av);
  gemm_acc<4, RN, false, true>(ak, Vs, D + 1, Gs, D + 1, D, 4 * ti, tj);      // V G^T
  gemm_acc<4, RN, false, false>(av, Ks, D + 1, Gs, D + 1, D, 4 * ti, tj);     // K G
  masked_product<D, true>(Ms, Os, Vs, ti, tj);                                // tril(dO V^T): (t, s)
  __syncthreads();
  gemm_acc<4, RN, true, false>(ak, Ms, kBlk + 1, Qs, D + 1, kBlk, 4 * ti, tj); // its transpose times Q
  __syncthreads();
  masked_product<D, true>(Ms, Qs, Ks, ti, tj);                                // tril(Q K^T): (t, s)
  __syncthreads();
  gemm_acc<4, RN, true, false>(av, Ms, kBlk + 1, Os, D + 1, kBlk, 4 * ti, tj); // its transpose times dO
  store_rows(dk + row0 * D, ak, 4 * ti, tj, scale, D);
  store_rows(dv + row0 * D, av, 4 * ti, tj, scale, D);
}

template <int D>
constexpr int smem_bytes(int blocks) {   // one D x D state and `blocks` kBlk x D tiles, one kBlk^2 matrix
  return (D * (D + 1) + blocks * kBlk * (D + 1) + kBlk * (kBlk + 1)) * 4;
}

template <typename K>
static cudaError_t allow_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Fixed state workspace of lasp_fwd_noalloc: 8M floats (32 MB) per device,
// part of the module image, so that call allocates nothing.
constexpr int64_t kScratchFloats = int64_t(8) << 20;
__device__ __align__(256) float g_scratch[kScratchFloats];

// Device address of g_scratch on the current device.  A successful lookup
// is kept per device (at most kMaxDevices); a failed one (for instance made
// inside a stream capture) is not, so a later call retries it.  The first
// call on a device should come before any stream capture.
constexpr int kMaxDevices = 64;
static float* scratch_ptr(cudaError_t* err) {
  static std::mutex mu;
  static float* ptr[kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_scratch);
    if (*err != cudaSuccess) {
      cudaGetLastError();   // not sticky: leave no error behind for the next launch check
      return nullptr;
    }
    ptr[dev] = static_cast<float*>(p);
  }
  return ptr[dev];
}

}  // namespace lasp
}  // namespace sca

using namespace sca;
using namespace sca::lasp;

// block: 64 = the fp32 CUDA-core kernels below; a multiple of 128 (up to
// 4096) = the tensor-core kernels of lasp_tc.cu (bf16, D = 128)
static int lasp_check(int64_t BH, int64_t S, int D, int P, int dtype, int block, const char* who) {
  SCA_REQUIRE(BH >= 1 && BH <= 65535, SCA_ERR_ARG, "%s: BH=%lld outside [1, 65535]", who, static_cast<long long>(BH));
  SCA_REQUIRE(D == 64 || D == 128, SCA_ERR_UNSUPPORTED, "%s: D=%d: only 64 and 128", who, D);
  SCA_REQUIRE(dtype == SCA_BF16 || dtype == SCA_F32, SCA_ERR_ARG, "%s: dtype=%d unknown", who, dtype);
  const bool tc = block != kBlk;
  SCA_REQUIRE(!tc || (block > 0 && block % kLaspTcSub == 0 && block <= kLaspTcMaxBlock), SCA_ERR_ARG,
              "%s: block=%d: %d, or a multiple of %d up to %d", who, block, kBlk, kLaspTcSub, kLaspTcMaxBlock);
  SCA_REQUIRE(!tc || (dtype == SCA_BF16 && D == 128), SCA_ERR_UNSUPPORTED,
              "%s: blocks of a multiple of %d rows (tensor cores) need bf16 inputs and D = 128", who, kLaspTcSub);
  SCA_REQUIRE(P >= 1 && S > 0 && S % (static_cast<int64_t>(block) * P) == 0, SCA_ERR_ARG,
              "%s: S=%lld must be a positive multiple of %d*P (P=%d)", who, static_cast<long long>(S), block, P);
  return SCA_OK;
}

#define SCA_LASP_DISPATCH(D_, DT_, CALL)                        \
  do {                                                          \
    if ((D_) == 64 && (DT_) == SCA_BF16) { CALL(64, __nv_bfloat16); } \
    else if ((D_) == 64) { CALL(64, float); }                  \
    else if ((DT_) == SCA_BF16) { CALL(128, __nv_bfloat16); }  \
    else { CALL(128, float); }                                 \
  } while (0)

extern "C" int lasp_block_states(const void* a, const void* b, int dtype, float* st, int64_t BH, int64_t S, int D,
                                 int block, int* dev_status, void* stream) {
  int rc;
  if ((rc = lasp_check(BH, S, D, 1, dtype, block, "lasp_block_states")) != SCA_OK) return rc;
  SCA_REQUIRE(a && b && st, SCA_ERR_ARG, "lasp_block_states: NULL pointer");
  if (block != kBlk) return lasp_tc_states(a, b, st, BH, S, block, dev_status, as_stream(stream));
  const dim3 grid(static_cast<unsigned>(S / kBlk), static_cast<unsigned>(BH));
  cudaError_t e = cudaSuccess;
#define SCA_STATES(DD, TT)                                                                               \
  {                                                                                                     \
    constexpr int bytes = 2 * kBlk * (DD + 1) * 4;                                                      \
    e = allow_smem(states_kernel<DD, TT>, bytes);                                                       \
    if (e == cudaSuccess)                                                                               \
      states_kernel<DD, TT><<<grid, kThreads, bytes, as_stream(stream)>>>(static_cast<const TT*>(a),    \
                                                                          static_cast<const TT*>(b), st, S); \
  }
  SCA_LASP_DISPATCH(D, dtype, SCA_STATES);
#undef SCA_STATES
  if (e != cudaSuccess) return cuda_status(e, "lasp_block_states");
  return cuda_status(cudaGetLastError(), "lasp_block_states launch");
}

extern "C" int lasp_scan(float* st, float* shard_total, int64_t BH, int64_t S, int D, int P, int block, int reverse,
                         void* stream) {
  int rc;
  if ((rc = lasp_check(BH, S, D, P, block == kBlk ? SCA_F32 : SCA_BF16, block, "lasp_scan")) != SCA_OK) return rc;
  SCA_REQUIRE(st && shard_total, SCA_ERR_ARG, "lasp_scan: NULL pointer");
  SCA_REQUIRE(reinterpret_cast<uintptr_t>(st) % 16 == 0 && reinterpret_cast<uintptr_t>(shard_total) % 16 == 0,
              SCA_ERR_ALIGN, "lasp_scan: st and shard_total must be 16-byte aligned");
  const int DD = D * D;
  const dim3 grid((DD / 4 + 255) / 256, static_cast<unsigned>(BH), static_cast<unsigned>(P));
  scan_kernel<<<grid, 256, 0, as_stream(stream)>>>(st, shard_total, S / block, DD, P, reverse ? 1 : 0);
  return cuda_status(cudaGetLastError(), "lasp_scan launch");
}

extern "C" int lasp_exchange(const float* shard_total, float* shard_in, int64_t BH, int D, int P, int reverse,
                             void* stream) {
  SCA_REQUIRE(shard_total && shard_in, SCA_ERR_ARG, "lasp_exchange: NULL pointer");
  SCA_REQUIRE(BH >= 1 && BH <= 65535 && P >= 1 && (D == 64 || D == 128), SCA_ERR_ARG,
              "lasp_exchange: BH=%lld, D=%d, P=%d", static_cast<long long>(BH), D, P);
  const int DD = D * D;
  const dim3 grid((DD + 255) / 256, static_cast<unsigned>(BH));
  exchange_kernel<<<grid, 256, 0, as_stream(stream)>>>(shard_total, shard_in, DD, P, reverse ? 1 : 0);
  return cuda_status(cudaGetLastError(), "lasp_exchange launch");
}

extern "C" int lasp_fwd(const void* q, const void* k, const void* v, int dtype, const float* st,
                        const float* shard_in, float* o, int64_t BH, int64_t S, int D, int P, int block, float scale,
                        int* dev_status, void* stream) {
  int rc;
  if ((rc = lasp_check(BH, S, D, P, dtype, block, "lasp_fwd")) != SCA_OK) return rc;
  SCA_REQUIRE(q && k && v && st && shard_in && o, SCA_ERR_ARG, "lasp_fwd: NULL pointer");
  if (block != kBlk) return lasp_tc_fwd(q, k, v, st, shard_in, o, BH, S, P, block, scale, dev_status, as_stream(stream));
  const dim3 grid(static_cast<unsigned>(S / kBlk), static_cast<unsigned>(BH));
  cudaError_t e = cudaSuccess;
#define SCA_FWD(DD, TT)                                                                                    \
  {                                                                                                       \
    constexpr int bytes = smem_bytes<DD>(3);                                                              \
    e = allow_smem(fwd_kernel<DD, TT>, bytes);                                                            \
    if (e == cudaSuccess)                                                                                 \
      fwd_kernel<DD, TT><<<grid, kThreads, bytes, as_stream(stream)>>>(                                   \
          static_cast<const TT*>(q), static_cast<const TT*>(k), static_cast<const TT*>(v), st, shard_in, o, S, \
          P, scale);                                                                                      \
  }
  SCA_LASP_DISPATCH(D, dtype, SCA_FWD);
#undef SCA_FWD
  if (e != cudaSuccess) return cuda_status(e, "lasp_fwd");
  return cuda_status(cudaGetLastError(), "lasp_fwd launch");
}

extern "C" int lasp_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype,
                        const float* st_fwd, const float* in_fwd, const float* st_bwd, const float* in_bwd, float* dq,
                        float* dk, float* dv, int64_t BH, int64_t S, int D, int P, int block, float scale,
                        int* dev_status, void* stream) {
  int rc;
  if ((rc = lasp_check(BH, S, D, P, dtype, block, "lasp_bwd")) != SCA_OK) return rc;
  SCA_REQUIRE(q && k && v && dout && st_fwd && in_fwd && st_bwd && in_bwd && dq && dk && dv, SCA_ERR_ARG,
              "lasp_bwd: NULL pointer");
  if (block != kBlk)
    return lasp_tc_bwd(q, k, v, dout, st_fwd, in_fwd, st_bwd, in_bwd, dq, dk, dv, BH, S, P, block, scale, dev_status,
                       as_stream(stream));
  const dim3 grid(static_cast<unsigned>(S / kBlk), static_cast<unsigned>(BH));
  cudaError_t e = cudaSuccess;
#define SCA_BWD(DD, TT)                                                                                     \
  {                                                                                                        \
    constexpr int b1 = smem_bytes<DD>(3), b2 = smem_bytes<DD>(4);                                          \
    e = allow_smem(dq_kernel<DD, TT>, b1);                                                                 \
    if (e == cudaSuccess) e = allow_smem(dkdv_kernel<DD, TT>, b2);                                         \
    if (e == cudaSuccess) {                                                                                \
      dq_kernel<DD, TT><<<grid, kThreads, b1, as_stream(stream)>>>(                                        \
          static_cast<const TT*>(k), static_cast<const TT*>(v), static_cast<const TT*>(dout), st_fwd, in_fwd, dq, \
          S, P, scale);                                                                                    \
      dkdv_kernel<DD, TT><<<grid, kThreads, b2, as_stream(stream)>>>(                                      \
          static_cast<const TT*>(q), static_cast<const TT*>(k), static_cast<const TT*>(v),                 \
          static_cast<const TT*>(dout), st_bwd, in_bwd, dk, dv, S, P, scale);                              \
    }                                                                                                      \
  }
  SCA_LASP_DISPATCH(D, dtype, SCA_BWD);
#undef SCA_BWD
  if (e != cudaSuccess) return cuda_status(e, "lasp_bwd");
  return cuda_status(cudaGetLastError(), "lasp_bwd launch");
}

extern "C" int lasp_fwd_noalloc(const void* q, const void* k, const void* v, int dtype, float* o, int64_t BH,
                                int64_t S, int D, int P, float scale, void* stream) {
  int rc;
  if ((rc = lasp_check(BH, S, D, P, dtype, kBlk, "lasp_fwd_noalloc")) != SCA_OK) return rc;
  SCA_REQUIRE(q && k && v && o, SCA_ERR_ARG, "lasp_fwd_noalloc: NULL pointer");
  const int64_t nblk = S / kBlk, DD = static_cast<int64_t>(D) * D;
  const int64_t need = BH * nblk * DD + 2 * BH * P * DD;   // block states, shard totals, shard inputs
  SCA_REQUIRE(need <= kScratchFloats, SCA_ERR_UNSUPPORTED,
              "lasp_fwd_noalloc: needs %lld floats of state, the fixed workspace holds %lld",
              static_cast<long long>(need), static_cast<long long>(kScratchFloats));
  cudaError_t e;
  float* st = scratch_ptr(&e);
  if (!st) return cuda_status(e, "lasp_fwd_noalloc workspace address");
  float* tot = st + BH * nblk * DD;
  float* in = tot + BH * P * DD;
  // every state is written before it is read: nothing needs clearing
  if ((rc = lasp_block_states(k, v, dtype, st, BH, S, D, kBlk, nullptr, stream)) != SCA_OK) return rc;
  if ((rc = lasp_scan(st, tot, BH, S, D, P, kBlk, 0, stream)) != SCA_OK) return rc;
  if ((rc = lasp_exchange(tot, in, BH, D, P, 0, stream)) != SCA_OK) return rc;
  return lasp_fwd(q, k, v, dtype, st, in, o, BH, S, D, P, kBlk, scale, nullptr, stream);
}
