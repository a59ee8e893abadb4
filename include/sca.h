/*
 * sca.h - C ABI of the sharded causal softmax attention library (libsca.so).
 *
 * The library computes causal softmax attention over a sequence split into P
 * context shards, one (query shard, key/value block) pair at a time, as an
 * (o, lse) partial, and merges the partials exactly by log-sum-exp
 * rescaling.  The operation is the unit O = f(A B) C of "METP:
 * memory-efficient tensor parallelism" (FITEE 10.1631/FITEE.2400602,
 * abstract) with A B = Q K^T, f = causal row softmax of the scores times
 * `scale`, C = V:
 *
 *     s_ij  = scale * q_i . k_j   if pos(k_j) <= pos(q_i), else -inf
 *     lse_i = ln sum_j exp(s_ij)                  (natural log)
 *     o_i   = sum_j exp(s_ij - lse_i) v_j
 *
 * A query row that sees no key of the block gives o = 0, lse = -inf.
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller
 *     owns all memory.  No entry point allocates device memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and returns an sca_status.  Arguments are validated on
 *     the host before anything is launched; on a non-OK return nothing was
 *     launched and sca_last_error() gives a message.
 *   - `dev_status` (may be NULL) is a device int32 the caller zeroes once;
 *     kernels record the first device-side failure in it (a bounded wait that
 *     gave up: SCA_ERR_TIMEOUT).  Kernels never trap.  sca_read_status()
 *     reads it back.
 *   - Tensors are [B, H, rows, D] views with D contiguous; element strides
 *     for batch, head and row are given explicitly (sca_view).  Base pointers
 *     must be 16-byte aligned and row strides multiples of 8 elements (bf16)
 *     or 4 elements (fp32).
 *   - Errors are return codes only; no C++ exception crosses this boundary.
 */
#ifndef SCA_H
#define SCA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SCA_OK = 0,
  SCA_ERR_ARG = -1,          /* invalid argument (size, pointer, stride, alias) */
  SCA_ERR_UNSUPPORTED = -2,  /* valid but not implemented (e.g. D not 64/128)  */
  SCA_ERR_CUDA = -3,         /* a CUDA runtime/driver call failed              */
  SCA_ERR_TIMEOUT = -4,      /* device-side bounded wait gave up (dev_status)  */
  SCA_ERR_ALIGN = -5,        /* pointer or stride misaligned                   */
  SCA_ERR_RANGE = -6         /* an fp16 conversion met a finite value beyond
                                the fp16 range, |x| >= 65536 (dev_status)    */
} sca_status;

typedef enum { SCA_BF16 = 0, SCA_F32 = 1 } sca_dtype;

/* Kernel choice for attn_fwd_shard / attn_bwd_shard.  AUTO picks the
 * tcgen05 tensor-core kernel for bf16 and the fp32 SIMT kernel for fp32.
 * SIMT forces the fp32-arithmetic kernel for either input dtype (used as an
 * independent cross-check of the tensor-core kernel). */
typedef enum { SCA_ALGO_AUTO = 0, SCA_ALGO_SIMT = 1, SCA_ALGO_TC = 2 } sca_algo;

/* Row-position map of a slab of rows (a shard's queries or a key/value
 * block): n (1 or 2) segments of `len` consecutive global positions; slab
 * row i (0 <= i < n*len) sits at global position start[i / len] + i % len.
 * A zigzag shard r of a sequence cut into 2P chunks of c rows is
 * {n=2, len=c, start={r*c, (2P-1-r)*c}}; a contiguous shard is n=1.
 * Causal visibility compares these global positions. */
typedef struct {
  int32_t n;
  int32_t reserved;
  int64_t len;
  int64_t start[2];
} sca_segs;

/* Element strides (batch, head, row) of a [B, H, rows, D] tensor view; the
 * D stride is 1. */
typedef struct {
  int64_t b, h, s;
} sca_view;

/* Shapes and layouts shared by all items of one attention call. */
typedef struct {
  int32_t B, H, D;     /* batch, heads, head dim (64 or 128)                 */
  int32_t dtype;       /* sca_dtype of q, k, v (and dO in the backward)      */
  int32_t causal;      /* 1: mask pos(k) > pos(q); 0: every key visible       */
  int32_t algo;        /* sca_algo                                           */
  float scale;         /* score scale, normally 1/sqrt(D)                    */
  int32_t accumulate;  /* backward: 1 adds into dq/dk/dv, 0 overwrites them  */
  sca_view q;          /* q (and dO) view                                    */
  sca_view kv;         /* k and v view                                       */
  sca_view o;          /* fp32 o (forward) / dq (backward) view              */
  sca_view dkv;        /* fp32 dk, dv view (backward only)                   */
  int64_t lse_b, lse_h;/* fp32 lse (and delta) strides; row stride is 1       */
  /* Row addressing.  0: slab row i of an item is row i of the tensor
   * (shard-major slabs).  1: it is row pos(i) of the tensor, its global
   * position from the item's segment map (natural order: the zigzag map
   * folded into the addressing, no permuted copy).  By-position segments
   * must be multiples of 128 rows (SCA_ERR_UNSUPPORTED otherwise). */
  int32_t q_by_pos;    /* q, o, lse (forward); q, dout, dq, lse, delta (bwd) */
  int32_t kv_by_pos;   /* k, v                                               */
  int32_t dkv_by_pos;  /* dk, dv (backward only)                             */
  /* Key/value heads (grouped-query attention, "Avances en la capacitacion
   * de LLMs de secuencia larga", section "Comprendiendo la Arquitectura de
   * los LLMs": query heads in groups share one key/value head).  0 or H:
   * one per query head.  Otherwise H must be a multiple of it and query
   * head h reads key/value head h / (H / kv_heads); k, v (and dk, dv, which
   * then sum over the group) have kv_heads heads in the kv / dkv views. */
  int32_t kv_heads;
  /* Backward, bf16 on the tensor cores only (SCA_ERR_ARG otherwise): inputs
   * the caller has already converted to fp16 with cast_bf16_to_f16, so the
   * kernel skips converting them tile by tile.  Bit 0 (SCA_F16_Q): each
   * item's q holds fp16.  Bit 1 (SCA_F16_DOUT): each item's dout holds
   * fp16; only with grouped key/value heads (0 < kv_heads < H), the one
   * case where the backward runs dP and dV as fp16 products.  0: bf16. */
  int32_t f16_inputs;
} sca_attn_dims;

#define SCA_F16_Q 1
#define SCA_F16_DOUT 2

/* One (query shard, key/value block) work item of the forward. */
typedef struct {
  const void* q;       /* [B,H,Sq,D] with Sq = q_pos.n * q_pos.len           */
  const void* k;       /* [B,H,Skv,D] with Skv = kv_pos.n * kv_pos.len        */
  const void* v;       /* same view as k                                     */
  float* o;            /* fp32 [B,H,Sq,D] partial output (normalised)        */
  float* lse;          /* fp32 [B,H,Sq] partial lse (natural log)            */
  sca_segs q_pos;
  sca_segs kv_pos;
} sca_fwd_item;

#define SCA_MAX_ITEMS 32

/* attn_fwd_shard - (o, lse) partials of causal attention for n_items
 * independent (query shard, key block) pairs in one launch.
 * Defined by: the unit O = f(A B) C of the METP abstract (above); the
 * per-block partial and its lse are what lets a shard's output be built one
 * ring step at a time ("Avances en la capacitacion de LLMs de secuencia
 * larga", section "Limitaciones de los Enfoques Existentes").
 * Items must not share output rows.  o is written (not accumulated), in
 * fp32, already divided by the row's softmax denominator; lse is natural
 * log.  Rows with no visible key: o = 0, lse = -inf.
 * Errors: SCA_ERR_ARG for n_items outside [1, SCA_MAX_ITEMS], segment
 * counts outside {1, 2}, non-positive sizes; SCA_ERR_UNSUPPORTED for D not
 * in {64, 128}; SCA_ERR_ALIGN for misaligned bases or strides. */
int attn_fwd_shard(const sca_fwd_item* items, int n_items, const sca_attn_dims* dims,
                   int* dev_status, void* stream);

/* attn_merge_lse - exact merge of n (o, lse) partials of the same rows:
 *   M = max_i lse_i, w_i = exp(lse_i - M),
 *   lse = M + ln sum_i w_i,  o = sum_i w_i o_i / sum_i w_i.
 * Defined by: the pages print no merge.  They keep one partial per key
 * block so that a shard's output can be assembled as blocks arrive ("Avances
 * en la capacitacion de LLMs de secuencia larga", section "Limitaciones de
 * los Enfoques Existentes"); with each partial normalised and carrying its
 * natural-log lse (attn_fwd_shard), the formula above is the exact way to
 * combine them (the textbook log-sum-exp rescaling), so the merged row is
 * the softmax over the union of the blocks' keys.
 * Rows whose partials are all -inf give o = 0, lse = -inf.
 * Layout: o_parts[p * o_part_stride + row * D + d] (fp32),
 * lse_parts[p * lse_part_stride + row] (fp32), rows contiguous.
 * Outputs: o_out fp32 [rows, D], lse_out fp32 [rows], o_bf16_out optional
 * bf16 copy (NULL to skip).  Without unpermuting, o_out may be exactly one
 * partial's o rows (o_parts + p * o_part_stride) and lse_out exactly one
 * partial's lse rows; every other overlap of an output with an input or
 * with another output is rejected (SCA_ERR_ARG).
 * If `unpermute_P` > 0 the rows are taken as `rows / S` sequences of S
 * rows in zigzag shard-major order over unpermute_P shards, and each output
 * row is written at its natural position (fused inverse zigzag permute; the
 * outputs must then not overlap the inputs at all).
 * Errors: SCA_ERR_ARG for n < 1 or n > 64, rows < 0, D not a positive
 * multiple of 4, S not divisible by 2*unpermute_P, overlaps as above;
 * SCA_ERR_ALIGN. */
int attn_merge_lse(const float* o_parts, const float* lse_parts, int n, int64_t rows, int D,
                   int64_t o_part_stride, int64_t lse_part_stride,
                   float* o_out, float* lse_out, void* o_bf16_out,
                   int unpermute_P, int64_t S, void* stream);

/* zigzag_permute - reorder the sequence axis of a [outer, S, row_bytes]
 * byte tensor into zigzag shard-major order: the sequence is cut into 2P
 * chunks of S/(2P) rows and shard r's slab holds chunk r followed by chunk
 * 2P-1-r (TSP page, "Zyphra presenta el paralelismo de secuencia y tensor
 * (TSP)", section "Lo que realmente significa plegar": K/V are reordered in
 * zigzag before FlashAttention to balance causal work).  inverse = 1 undoes
 * it.  A pure copy (bit exact).  src and dst must not overlap.  When both
 * pointers and the chunk size (S/(2P) * row_bytes) are multiples of 16
 * bytes, the chunks move by bulk copies through shared memory (the TMA
 * unit); a bounded wait that gives up records SCA_ERR_TIMEOUT in
 * *dev_status (may be NULL).  Otherwise a vectorised copy kernel moves them.
 * Errors: SCA_ERR_ARG for S % (2P) != 0, P < 1, row_bytes not a positive
 * multiple of 4, overlapping buffers; SCA_ERR_ALIGN if pointers are not
 * 4-byte aligned. */
int zigzag_permute(const void* src, void* dst, int64_t outer, int64_t S, int64_t row_bytes,
                   int P, int inverse, int* dev_status, void* stream);

/* ring_stage_block - one ring step's key/value hand-off emulated on one GPU:
 * copy rows [row0, row0 + rows) of every (b, h) of a [outer, S_src, row]
 * tensor into a contiguous [outer, rows, row] staging buffer, so the next
 * ring step's block is staged while the current one is computed (double
 * buffering of the METP abstract; point-to-point passing of key/value
 * blocks, "Avances en la capacitacion de LLMs de secuencia larga", section
 * "Limitaciones de los Enfoques Existentes").  When addresses and row sizes
 * are multiples of 16 bytes the copy is a small kernel (one 64-thread block
 * per SM, few registers) that runs beside the attention kernels; otherwise
 * it is one strided 2-D runtime copy.  Issue it on a stream of its own (of
 * high priority, so its blocks are dispatched first) to overlap it with
 * compute.  Errors: SCA_ERR_ARG for out-of-range rows. */
int ring_stage_block(const void* src, void* dst, int64_t outer, int64_t S_src, int64_t row0,
                     int64_t rows, int64_t row_bytes, void* stream);

/* ring_stage_segments - the same hand-off for a block kept in natural order:
 * its rows are the `seg->n` segments of `seg->len` rows starting at rows
 * seg->start[i] of every (b, h) of a [outer, S_src, row] tensor (a zigzag
 * shard: chunks r and 2P-1-r), gathered in segment order into a contiguous
 * [outer, seg->n * seg->len, row] staging slab, one strided 2-D copy per
 * segment (the copy kernel of ring_stage_block, under the same conditions;
 * double buffering of the METP abstract; block passing of "Avances en la
 * capacitacion de LLMs de secuencia larga", section "Limitaciones de los
 * Enfoques Existentes").  The caller owns both buffers;
 * they must not overlap.  Errors: SCA_ERR_ARG for NULL pointers, segment
 * counts outside {1, 2}, rows outside [0, S_src). */
int ring_stage_segments(const void* src, void* dst, int64_t outer, int64_t S_src, const sca_segs* seg,
                        int64_t row_bytes, void* stream);

/* One strided 2-D copy of a ring hand-off: `height` rows of `width` bytes,
 * row r from src + r * src_pitch to dst + r * dst_pitch (pitches in bytes). */
typedef struct {
  const void* src;
  void* dst;
  int64_t height, width, src_pitch, dst_pitch;
} sca_copy;

#define SCA_MAX_COPIES 128

/* ring_stage_copies - every copy of one ring hand-off (the blocks all ranks
 * receive for the next step, gathered from home rows or passed on from a
 * neighbour's staging buffer) in one launch of the hand-off copy kernel (one
 * 64-thread block per SM, few registers: it runs beside the attention
 * kernels; double buffering of the METP abstract).  Up to SCA_MAX_COPIES
 * copies; pointers 16-byte aligned, widths and pitches multiples of 16
 * bytes, pitches at least the width; no copy's source may overlap its own
 * destination, and no copy may write what another copy of the call reads or
 * writes (they run concurrently).  Issue it on a stream of its own, of high
 * priority, to overlap it with compute.  Errors: SCA_ERR_ARG (count, NULL,
 * sizes, overlap), SCA_ERR_ALIGN. */
int ring_stage_copies(const sca_copy* copies, int n, void* stream);

/* One (query shard, key/value block) work item of the backward.  dq, dk, dv
 * are fp32: with dims->accumulate = 1 the item ADDS its contribution, with 0
 * it overwrites them (every row of dq and of dk/dv is written, also rows
 * that see no key of the block).  lse and delta are the FINAL (merged)
 * values of the query rows. */
typedef struct {
  const void* q;       /* [B,H,Sq,D], dims->q view                           */
  const void* k;       /* [B,H,Skv,D], dims->kv view                         */
  const void* v;
  const void* dout;    /* dO, [B,H,Sq,D], dims->q view                       */
  const float* lse;    /* fp32 [B,H,Sq], natural log, dims->lse_* strides    */
  const float* delta;  /* fp32 [B,H,Sq], delta_i = dO_i . O_i                */
  float* dq;           /* fp32 [B,H,Sq,D], dims->o view                      */
  float* dk;           /* fp32 [B,H,Skv,D], dims->dkv view                   */
  float* dv;
  sca_segs q_pos;
  sca_segs kv_pos;
} sca_bwd_item;

/* attn_bwd_shard - gradient contributions of n_items (query shard, key
 * block) pairs, recomputing P_ij = exp(s_ij - lse_i) from the saved lse:
 *   dP_ij = dO_i . v_j,  dS_ij = P_ij (dP_ij - delta_i),
 *   dq_i += scale sum_j dS_ij k_j,  dk_j += scale sum_i dS_ij q_i,
 *   dv_j += sum_i P_ij dO_i.
 * (Textbook softmax-attention backward; the pages describe only storing
 * less and recomputing, "Avances en la capacitacion de LLMs de secuencia
 * larga", section "Escalabilidad y Gestion de Memoria".)
 * Items in one call must not share dq rows nor dk/dv rows.
 * With bf16 inputs the tensor-core kernel computes S, dK and dQ as fp16
 * products (q and k are converted to fp16 inside the kernel, dS is rounded
 * to fp16), and with grouped-query heads dP and dV too (v and dout
 * converted, P rounded to fp16): |q|, |k| (and |v|, |dout|) must stay below
 * 65536.  A finite input at or above that would become +-inf in fp16; the
 * kernel records SCA_ERR_RANGE in dev_status when it converts one (as does
 * cast_bf16_to_f16 for the inputs the caller converted), so such a call
 * cannot pass for a good one.  dims->f16_inputs lets the caller pass q (and, grouped, dout)
 * already converted by cast_bf16_to_f16: the same values, converted once
 * per call instead of once per key tile that reads them.  dq is summed over key tiles
 * by fp32 reduce-adds in no fixed order, so it is reproducible only up to
 * rounding order; dk and dv have one writer per row.  The tensor-core path
 * needs dq, dk, dv rows 16-byte aligned with strides that are multiples of
 * 16 bytes (SCA_ERR_ALIGN otherwise), and in overwrite mode dq rows
 * contiguous (dims->o.s == D).  Errors as attn_fwd_shard. */
int attn_bwd_shard(const sca_bwd_item* items, int n_items, const sca_attn_dims* dims,
                   int* dev_status, void* stream);

/* cast_bf16_to_f16 - dst[i] = src[i] rounded from bf16 to fp16 (round to
 * nearest even), for i < n: exact for |x| in [2^-14, 65280] (every bf16
 * value up to the largest below 65536), fp16 subnormals below 2^-14 (an
 * absolute error under 2^-25), +-inf for finite |x| >= 65536.  Meeting such
 * a value records SCA_ERR_RANGE in *dev_status (may be NULL); the
 * conversion still completes.  +-inf and NaN inputs stay +-inf and NaN.
 * No counterpart on the pages: the staging step that gives attn_bwd_shard
 * (dims->f16_inputs) its fp16 queries once per call.  src and dst may not
 * overlap; n a multiple of 8 and both pointers 16-byte aligned (whole
 * 16-byte vectors).
 * Errors: SCA_ERR_ARG for NULL pointers, n < 0, n % 8 != 0, overlap;
 * SCA_ERR_ALIGN for misaligned pointers. */
int cast_bf16_to_f16(const void* src, void* dst, int64_t n, int* dev_status, void* stream);

/* attn_bwd_delta - delta_i = sum_d dO_id * O_id for `rows` contiguous rows:
 * o fp32 [rows, D], dout [rows, D] of dtype `dout_dtype`, delta fp32 [rows].
 * Errors: SCA_ERR_ARG, SCA_ERR_ALIGN. */
int attn_bwd_delta(const float* o, const void* dout, int dout_dtype, float* delta,
                   int64_t rows, int D, void* stream);

/* ---- Linear attention sequence parallelism (LASP) --------------------
 * Causal linear attention (identity feature map, no normalisation):
 *   o_t = scale * sum_{s <= t} (q_t . k_s) v_s
 * over P contiguous shards of the sequence, which exchange D x D states
 * point to point: the k^T v of earlier shards in the forward, the q^T dO of
 * later shards in the backward, and use the right product q . state
 * ("Effiziente Parallelisierung linearer Aufmerksamkeitssequenzen fuer
 * skalierbare Sprachmodelle", the LASP summary; it prints no formula, this
 * is the plain reading).  Tensors q, k, v, dout are row-contiguous
 * [BH, S, D] (BH = batch x heads, at most 65535) of dtype bf16 or fp32,
 * 16-byte aligned; o, dq, dk, dv are fp32 [BH, S, D], overwritten.
 *
 * Rows go in blocks of `block` rows, which also selects the kernels:
 *   SCA_LASP_BLOCK_F32 (64): fp32 arithmetic on the CUDA cores; bf16 or
 *     fp32 inputs, D 64 or 128;
 *   a multiple of SCA_LASP_BLOCK_TC (128) up to 4096: tcgen05 tensor cores
 *     with fp32 accumulation, each block taken as sub-blocks of 128 rows
 *     with the state carried from one to the next inside the kernel; bf16
 *     inputs and D = 128 only (else SCA_ERR_UNSUPPORTED).  The fp32
 *     operands (states, masked block products) are split into two bf16
 *     parts and multiplied twice, keeping about fp32 accuracy.
 * S must be a multiple of block * P, and every call of one pass uses the
 * same block.  States are fp32 D x D, row index the first factor's
 * column: per block st [BH, S/block, D, D], per shard [BH, P, D, D]; the
 * caller owns every buffer (no allocation).  `dev_status` (may be NULL) is
 * the device status word the tensor-core kernels report a timed-out wait
 * in (SCA_ERR_TIMEOUT); the CUDA-core kernels never wait.  Errors:
 * SCA_ERR_ARG (NULL pointers, sizes, block), SCA_ERR_UNSUPPORTED (D not 64
 * or 128, block 128 without bf16 and D = 128), SCA_ERR_ALIGN (an input the
 * tensor-core path cannot address by TMA), SCA_ERR_CUDA. */
#define SCA_LASP_BLOCK_F32 64
#define SCA_LASP_BLOCK_TC 128

/* lasp_block_states - st[bh][j] = A_j^T B_j over the rows of block j:
 * (A, B) = (k, v) for the forward, (q, dout) for the backward. */
int lasp_block_states(const void* a, const void* b, int dtype, float* st, int64_t BH, int64_t S, int D, int block,
                      int* dev_status, void* stream);

/* lasp_scan - within each of the P shards (contiguous runs of blocks),
 * replaces st[bh][j] by the sum over the shard's blocks before j
 * (reverse = 0) or after j (reverse = 1), in place, and writes the sum over
 * all the shard's blocks to shard_total[bh][r]. */
int lasp_scan(float* st, float* shard_total, int64_t BH, int64_t S, int D, int P, int block, int reverse,
              void* stream);

/* lasp_exchange - the point-to-point pass of shard states, one hop at a
 * time along the ring: shard_in[bh][r] = sum of shard_total[bh][s] over
 * s < r (reverse = 0: shard r-1 sends to r) or s > r (reverse = 1: shard r+1
 * sends to r). */
int lasp_exchange(const float* shard_total, float* shard_in, int64_t BH, int D, int P, int reverse,
                  void* stream);

/* lasp_fwd - for every block j of shard r:
 *   o_j = scale * (q_j (st[j] + shard_in[r]) + tril(q_j k_j^T) v_j)
 * with st, shard_in from lasp_block_states(k, v) / lasp_scan(reverse = 0) /
 * lasp_exchange(reverse = 0). */
int lasp_fwd(const void* q, const void* k, const void* v, int dtype, const float* st, const float* shard_in,
             float* o, int64_t BH, int64_t S, int D, int P, int block, float scale, int* dev_status, void* stream);

/* lasp_bwd - for every block j of shard r, with F = st_fwd[j] + in_fwd[r]
 * (the forward states) and G = st_bwd[j] + in_bwd[r] (from
 * lasp_block_states(q, dout), lasp_scan and lasp_exchange with reverse = 1):
 *   dq_j = scale * (dout_j F^T + tril(dout_j v_j^T) k_j)
 *   dk_j = scale * (v_j G^T + tril(dout_j v_j^T)^T q_j)
 *   dv_j = scale * (k_j G + tril(q_j k_j^T)^T dout_j) */
int lasp_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype, const float* st_fwd,
             const float* in_fwd, const float* st_bwd, const float* in_bwd, float* dq, float* dk, float* dv,
             int64_t BH, int64_t S, int D, int P, int block, float scale, int* dev_status, void* stream);

/* lasp_fwd_noalloc - the whole LASP forward (lasp_block_states,
 * lasp_scan, lasp_exchange, lasp_fwd, blocks of SCA_LASP_BLOCK_F32 rows on
 * the CUDA cores) in one call, with its states in a
 * fixed device array inside the library instead of caller buffers: the call
 * allocates nothing.  The pages have no counterpart of this call; it exists
 * for callers that cannot provide a workspace (e.g. a captured graph that
 * must not allocate).  Limit: BH * (S / 64) * D^2 + 2 * BH * P * D^2
 * floats of state must fit the 8M-float (32 MB) array, else
 * SCA_ERR_UNSUPPORTED before anything runs.  The array's device address is
 * looked up on the first call on each device and kept once the lookup
 * succeeds (a failed lookup returns SCA_ERR_CUDA and is retried by the next
 * call); make that first call outside any stream capture.  Devices with an
 * ordinal above 63 get SCA_ERR_CUDA.  All calls share the array: two calls in
 * flight at once (other streams or threads, same device) race and must be
 * serialised by the caller.  Nothing in the array must start at zero (every
 * state is written before it is read).  o: fp32 [BH, S, D], overwritten. */
int lasp_fwd_noalloc(const void* q, const void* k, const void* v, int dtype, float* o, int64_t BH, int64_t S,
                     int D, int P, float scale, void* stream);

/* sca_selftest_wait_timeout - runs, on one thread, the bounded mbarrier
 * wait every tensor-core kernel uses, on a barrier nothing completes.  After
 * the library's wait limit (2 s) it gives up and records SCA_ERR_TIMEOUT in
 * *dev_status, exactly as a kernel whose pipeline stalled would; the kernel
 * returns and the context stays usable.  For testing the failure path; the
 * pages have no counterpart.  Errors: SCA_ERR_ARG (NULL status word),
 * SCA_ERR_CUDA. */
int sca_selftest_wait_timeout(int* dev_status, void* stream);

/* Message of the last non-OK return on the calling thread ("" if none). */
const char* sca_last_error(void);

/* Synchronises `stream`, copies *dev_status to the host and returns it
 * (SCA_OK if no kernel recorded a failure), or SCA_ERR_CUDA. */
int sca_read_status(const int* dev_status, void* stream);

/* Library version as major*10000 + minor*100 + patch. */
int sca_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SCA_H */
