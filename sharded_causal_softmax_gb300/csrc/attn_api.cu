// C-ABI entry points attn_fwd_shard / attn_bwd_shard: argument validation
// on the host, then dispatch to the tensor-core (bf16) or fp32-arithmetic
// kernels.  Nothing is launched when validation fails.
#include <cmath>

#include "common.cuh"
#include "host_common.h"
#include "simt_launch.h"

namespace sca {

static int check_segs(const sca_segs& s, const char* what, int idx) {
  SCA_REQUIRE(s.n == 1 || s.n == 2, SCA_ERR_ARG, "item %d: %s.n=%d must be 1 or 2", idx, what, s.n);
  SCA_REQUIRE(s.len >= 0 && s.len < (1LL << 31), SCA_ERR_ARG, "item %d: %s.len=%lld out of range", idx, what,
              static_cast<long long>(s.len));
  return SCA_OK;
}

static int check_view(const sca_view& v, int elem_mult, const char* what) {
  SCA_REQUIRE(v.b >= 0 && v.h >= 0 && v.s >= 0, SCA_ERR_ARG, "%s: negative stride", what);
  SCA_REQUIRE(v.b % elem_mult == 0 && v.h % elem_mult == 0 && v.s % elem_mult == 0, SCA_ERR_ALIGN,
              "%s: strides must be multiples of %d elements", what, elem_mult);
  return SCA_OK;
}

static int check_dims(const sca_attn_dims* d, bool bwd) {
  SCA_REQUIRE(d != nullptr, SCA_ERR_ARG, "dims is NULL");
  SCA_REQUIRE(d->B >= 1 && d->H >= 1 && static_cast<int64_t>(d->B) * d->H <= 65535, SCA_ERR_ARG,
              "B=%d, H=%d: need B, H >= 1 and B*H <= 65535", d->B, d->H);
  SCA_REQUIRE(d->D == 64 || d->D == 128, SCA_ERR_UNSUPPORTED, "D=%d: only 64 and 128 are supported", d->D);
  SCA_REQUIRE(d->dtype == SCA_BF16 || d->dtype == SCA_F32, SCA_ERR_ARG, "dtype=%d unknown", d->dtype);
  SCA_REQUIRE(d->algo >= SCA_ALGO_AUTO && d->algo <= SCA_ALGO_TC, SCA_ERR_ARG, "algo=%d unknown", d->algo);
  SCA_REQUIRE(std::isfinite(d->scale), SCA_ERR_ARG, "scale is not finite");
  SCA_REQUIRE(d->dtype == SCA_BF16 || d->algo != SCA_ALGO_TC, SCA_ERR_UNSUPPORTED,
              "the tensor-core kernels take bf16 inputs only");
  const int in_mult = d->dtype == SCA_BF16 ? 8 : 4;
  int rc;
  if ((rc = check_view(d->q, in_mult, "q view")) != SCA_OK) return rc;
  if ((rc = check_view(d->kv, in_mult, "kv view")) != SCA_OK) return rc;
  if ((rc = check_view(d->o, 4, bwd ? "dq view" : "o view")) != SCA_OK) return rc;
  if (bwd && (rc = check_view(d->dkv, 4, "dkv view")) != SCA_OK) return rc;
  SCA_REQUIRE(d->q.s >= d->D && d->kv.s >= d->D && d->o.s >= d->D && (!bwd || d->dkv.s >= d->D), SCA_ERR_ARG,
              "row strides must be >= D");
  SCA_REQUIRE(d->lse_b >= 0 && d->lse_h >= 0, SCA_ERR_ARG, "negative lse stride");
  SCA_REQUIRE((d->q_by_pos == 0 || d->q_by_pos == 1) && (d->kv_by_pos == 0 || d->kv_by_pos == 1) &&
                  (d->dkv_by_pos == 0 || d->dkv_by_pos == 1),
              SCA_ERR_ARG, "q_by_pos, kv_by_pos, dkv_by_pos must be 0 or 1");
  SCA_REQUIRE(bwd || d->dkv_by_pos == 0, SCA_ERR_ARG, "dkv_by_pos applies to the backward only");
  SCA_REQUIRE(d->kv_heads >= 0 && (d->kv_heads == 0 || d->H % d->kv_heads == 0), SCA_ERR_ARG,
              "kv_heads=%d must be 0 or divide H=%d", d->kv_heads, d->H);
  SCA_REQUIRE((d->f16_inputs & ~(SCA_F16_Q | SCA_F16_DOUT)) == 0, SCA_ERR_ARG, "f16_inputs=%d has unknown bits",
              d->f16_inputs);
  SCA_REQUIRE(d->f16_inputs == 0 || (bwd && d->dtype == SCA_BF16 && d->algo != SCA_ALGO_SIMT), SCA_ERR_ARG,
              "f16_inputs applies to the bf16 tensor-core backward only");
  SCA_REQUIRE(!(d->f16_inputs & SCA_F16_DOUT) || (d->kv_heads > 0 && d->kv_heads < d->H), SCA_ERR_ARG,
              "f16_inputs: fp16 dout needs grouped key/value heads (0 < kv_heads < H)");
  return SCA_OK;
}

// A by-position slab is read and written in 128-row tiles that must not
// straddle two segments.
static int check_by_pos(const sca_segs& s, bool by_pos, const char* what, int idx) {
  SCA_REQUIRE(!by_pos || s.len % 128 == 0, SCA_ERR_UNSUPPORTED,
              "item %d: %s addressed by position needs segments of a multiple of 128 rows (len=%lld)", idx, what,
              static_cast<long long>(s.len));
  for (int i = 0; by_pos && i < s.n; ++i)
    SCA_REQUIRE(s.start[i] >= 0, SCA_ERR_ARG, "item %d: %s addressed by position has a negative start", idx, what);
  return SCA_OK;
}

static void fill_common(AttnArgs& a, const sca_attn_dims* d, int n_items, int* dev_status) {
  a.n_items = n_items;
  a.B = d->B;
  a.H = d->H;
  a.D = d->D;
  a.causal = d->causal ? 1 : 0;
  a.accumulate = d->accumulate ? 1 : 0;
  a.scale = d->scale;
  a.scale_log2 = d->scale * kLog2e;
  a.q = {d->q.b, d->q.h, d->q.s};
  a.kv = {d->kv.b, d->kv.h, d->kv.s};
  a.o = {d->o.b, d->o.h, d->o.s};
  a.dkv = {d->dkv.b, d->dkv.h, d->dkv.s};
  a.lse_b = d->lse_b;
  a.lse_h = d->lse_h;
  a.status = dev_status;
  a.max_q_tiles = a.max_k_tiles = 0;
  a.q_by_pos = d->q_by_pos;
  a.kv_by_pos = d->kv_by_pos;
  a.dkv_by_pos = d->dkv_by_pos;
  a.Hkv = d->kv_heads > 0 ? d->kv_heads : d->H;
  a.group = d->H / a.Hkv;
}

static bool use_tc(const sca_attn_dims* d) {
  return d->algo == SCA_ALGO_TC || (d->algo == SCA_ALGO_AUTO && d->dtype == SCA_BF16);
}

}  // namespace sca

using namespace sca;

extern "C" int attn_fwd_shard(const sca_fwd_item* items, int n_items, const sca_attn_dims* dims,
                              int* dev_status, void* stream) {
  SCA_REQUIRE(items != nullptr, SCA_ERR_ARG, "attn_fwd_shard: items is NULL");
  SCA_REQUIRE(n_items >= 1 && n_items <= SCA_MAX_ITEMS, SCA_ERR_ARG, "attn_fwd_shard: n_items=%d outside [1, %d]",
              n_items, SCA_MAX_ITEMS);
  int rc;
  if ((rc = check_dims(dims, false)) != SCA_OK) return rc;
  AttnArgs a;
  fill_common(a, dims, n_items, dev_status);
  const uintptr_t in_align = 16;
  int64_t rows = 0;
  for (int i = 0; i < n_items; ++i) {
    const sca_fwd_item& x = items[i];
    if ((rc = check_segs(x.q_pos, "q_pos", i)) != SCA_OK) return rc;
    if ((rc = check_segs(x.kv_pos, "kv_pos", i)) != SCA_OK) return rc;
    if ((rc = check_by_pos(x.q_pos, dims->q_by_pos, "q", i)) != SCA_OK) return rc;
    if ((rc = check_by_pos(x.kv_pos, dims->kv_by_pos, "k/v", i)) != SCA_OK) return rc;
    SCA_REQUIRE(x.q && x.k && x.v && x.o && x.lse, SCA_ERR_ARG, "item %d: NULL pointer", i);
    SCA_REQUIRE(aligned(x.q, in_align) && aligned(x.k, in_align) && aligned(x.v, in_align) && aligned(x.o, 16) &&
                    aligned(x.lse, 4),
                SCA_ERR_ALIGN, "item %d: q/k/v/o must be 16-byte aligned, lse 4-byte", i);
    Item& it = a.items[i];
    it = Item{};
    it.q = x.q;
    it.k = x.k;
    it.v = x.v;
    it.o = x.o;
    it.lse = x.lse;
    it.qs = to_segs(x.q_pos);
    it.ks = to_segs(x.kv_pos);
    it.Sq = static_cast<int64_t>(x.q_pos.n) * x.q_pos.len;
    it.Skv = static_cast<int64_t>(x.kv_pos.n) * x.kv_pos.len;
    rows += it.Sq;
  }
  if (rows == 0) return SCA_OK;
  cudaStream_t st = as_stream(stream);
  cudaError_t e;
  if (use_tc(dims)) {
    e = tc_forward(a, st);
    if (e == cudaErrorNotSupported)
      return fail(SCA_ERR_ALIGN, "attn_fwd_shard: layout not expressible as a TMA tensor map");
  } else {
    e = simt_forward(a, dims->dtype, st);
  }
  return cuda_status(e, "attn_fwd_shard launch");
}

extern "C" int attn_bwd_shard(const sca_bwd_item* items, int n_items, const sca_attn_dims* dims,
                              int* dev_status, void* stream) {
  SCA_REQUIRE(items != nullptr, SCA_ERR_ARG, "attn_bwd_shard: items is NULL");
  SCA_REQUIRE(n_items >= 1 && n_items <= SCA_MAX_ITEMS, SCA_ERR_ARG, "attn_bwd_shard: n_items=%d outside [1, %d]",
              n_items, SCA_MAX_ITEMS);
  int rc;
  if ((rc = check_dims(dims, true)) != SCA_OK) return rc;
  AttnArgs a;
  fill_common(a, dims, n_items, dev_status);
  int64_t rows = 0;
  for (int i = 0; i < n_items; ++i) {
    const sca_bwd_item& x = items[i];
    if ((rc = check_segs(x.q_pos, "q_pos", i)) != SCA_OK) return rc;
    if ((rc = check_segs(x.kv_pos, "kv_pos", i)) != SCA_OK) return rc;
    if ((rc = check_by_pos(x.q_pos, dims->q_by_pos, "q", i)) != SCA_OK) return rc;
    if ((rc = check_by_pos(x.kv_pos, dims->kv_by_pos, "k/v", i)) != SCA_OK) return rc;
    if ((rc = check_by_pos(x.kv_pos, dims->dkv_by_pos, "dk/dv", i)) != SCA_OK) return rc;
    SCA_REQUIRE(x.q && x.k && x.v && x.dout && x.lse && x.delta && x.dq && x.dk && x.dv, SCA_ERR_ARG,
                "item %d: NULL pointer", i);
    SCA_REQUIRE(aligned(x.q, 16) && aligned(x.k, 16) && aligned(x.v, 16) && aligned(x.dout, 16) &&
                    aligned(x.dq, 16) && aligned(x.dk, 16) && aligned(x.dv, 16) && aligned(x.lse, 4) &&
                    aligned(x.delta, 4),
                SCA_ERR_ALIGN, "item %d: tensors must be 16-byte aligned, lse/delta 4-byte", i);
    Item& it = a.items[i];
    it = Item{};
    it.q = x.q;
    it.k = x.k;
    it.v = x.v;
    it.dout = x.dout;
    it.lse = const_cast<float*>(x.lse);
    it.delta = x.delta;
    it.o = x.dq;
    it.dk = x.dk;
    it.dv = x.dv;
    it.qs = to_segs(x.q_pos);
    it.ks = to_segs(x.kv_pos);
    it.Sq = static_cast<int64_t>(x.q_pos.n) * x.q_pos.len;
    it.Skv = static_cast<int64_t>(x.kv_pos.n) * x.kv_pos.len;
    rows += it.Sq * it.Skv;
  }
  if (rows == 0) return SCA_OK;
  cudaStream_t st = as_stream(stream);
  cudaError_t e;
  if (use_tc(dims)) {
    e = tc_backward(a, dims->f16_inputs, st);
    if (e == cudaErrorNotSupported)
      return fail(SCA_ERR_ALIGN, "attn_bwd_shard: layout not expressible as a TMA tensor map "
                                 "(or dq rows not contiguous in overwrite mode)");
  } else {
    e = simt_backward(a, dims->dtype, st);
  }
  return cuda_status(e, "attn_bwd_shard launch");
}
