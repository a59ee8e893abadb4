"""P virtual context shards of causal softmax attention on one GPU.

The schedule (host logic only; every byte is moved or computed by libsca):

* Partition.  Zigzag (TSP page, "Zyphra presenta el paralelismo de secuencia
  y tensor (TSP)", section "Lo que realmente significa plegar"): the sequence
  is cut into 2P chunks of c rows and shard r owns chunks r and 2P-1-r, which
  balances causal work.  Contiguous: shard r owns rows [r S/P, (r+1) S/P).
* Addressing.  "position" (the default when every chunk is a multiple of 128
  rows): the kernels read and write a shard's rows at their global positions
  in the natural-order tensors, so the zigzag map lives in the TMA
  coordinates and no permuted copy is made.  "permuted": ``zigzag_permute``
  lays Q, K, V (and dO, lse, delta) out shard-major so a shard is one
  contiguous slab, and the merge and the gradients undo it.
* 2D split ("Avances en la capacitacion de LLMs de secuencia larga", section
  "Introduciendo la Atencion 2D"): G head groups x P context shards give
  G*P virtual ranks; rank (g, r) holds heads [g H/G, (g+1) H/G) of shard r.
* Ring (same page, section "Limitaciones de los Enfoques Existentes"): at
  step t rank (g, r) holds key/value block (r - t) mod P and computes the
  (o, lse) partial of its queries against it.  With the "ring" schedule the
  blocks move like a ring pass: before step t+1, each rank's staging buffer
  receives the block its left neighbour holds at step t, copied by a small
  copy kernel on a high-priority side stream into a spare staging buffer
  while the steps before it compute (the double buffer of the METP
  abstract, FITEE 10.1631/FITEE.2400602; three buffers from P = 4 on, so
  each copy overlaps two steps).  The "direct" schedule reads every block from its
  home rows (the K/V all-gather reading of the TSP page); its forward
  partials of all P steps are independent and go out together, up to
  SCA_MAX_ITEMS (query shard, block) items per launch.
* Double ring (same page, section "Mejorando la Eficiencia de Comunicacion
  con la Atencion de Doble Anillo"; the page gives no layout): with
  visit="double_ring" the P shards form P / inner groups of `inner`
  consecutive shards.  Shard r = g * inner + i first passes blocks around
  the inner ring of its group (inner steps: blocks of group g, places
  i, i-1, ...), then the outer ring moves every group on to the blocks of
  the group before it, and the inner ring runs again.  At step
  t = u * inner + v shard r holds block ((g - u) mod outer) * inner +
  (i - v) mod inner.  Each staging copy takes a rank's next block from the
  rank that held it at the step before: a neighbour in the group on an
  inner hop, a rank of the previous group on an outer hop.
* Merge: the P partials of every row are combined exactly by log-sum-exp
  rescaling (``attn_merge_lse``), fused with the inverse permute when the
  partials are shard-major.
* "fused" schedule: all shards in one launch per direction.  Each CTA keeps
  its running (m, l, O) over every key/value block, so there are no partials
  and no merge; the backward writes each dK/dV row once.  One GPU holds
  every block, so nothing is staged.
* "auto" (the default): "fused" when a shard holds at most
  AUTO_FUSED_MAX_ROWS rows (a ring step's CTAs would then walk at most 32 key
  tiles each, too few to amortise a CTA's fixed cost of set-up, first loads
  and epilogue), "ring" otherwise or when the double ring is asked for.
* Backward: delta = rowsum(dO * O), then the same ring of steps; each step
  recomputes P from the final lse and adds into dQ of the rank's rows and
  into dK/dV of the block's rows (step 0 overwrites, so no zeroing pass is
  needed).

PyTorch supplies device memory, streams and events only.
"""
from __future__ import annotations

import math

import torch

from . import capi

_DT = {torch.bfloat16: capi.SCA_BF16, torch.float32: capi.SCA_F32}


def f16_input_flags(stage: bool, dtype, algo: int, H: int, Hkv: int) -> int:
    """sca_attn_dims.f16_inputs of a backward that stages its fp16 inputs:
    the queries whenever the tensor-core kernel runs (bf16, not forced onto
    the CUDA cores), and dO too under grouped key/value heads, where that
    kernel also takes dO in fp16."""
    if not stage or dtype != torch.bfloat16 or algo == capi.SCA_ALGO_SIMT:
        return 0
    return capi.SCA_F16_Q | (capi.SCA_F16_DOUT if Hkv < H else 0)


def launch_groups(n_items: int, per_launch: int = capi.SCA_MAX_ITEMS):
    """[lo, hi) ranges that send n_items independent items in as few
    launches as the per-launch limit allows."""
    return [(lo, min(lo + per_launch, n_items)) for lo in range(0, n_items, per_launch)]


def ring_block(r: int, t: int, P: int) -> int:
    """Key/value block held by shard r at ring step t."""
    return (r - t) % P


def double_ring_block(r: int, t: int, P: int, inner: int) -> int:
    """Key/value block held by shard r at step t of the double ring over
    P / inner groups of `inner` shards (see the module docstring)."""
    outer = P // inner
    g, i = divmod(r, inner)
    u, v = divmod(t, inner)
    return ((g - u) % outer) * inner + (i - v) % inner


def hop_senders(block_of, t_next: int, P: int):
    """senders[r]: the shard whose block at step t_next - 1 shard r holds at
    step t_next (every step's map from shards to blocks is one-to-one)."""
    held = {block_of(r, t_next - 1): r for r in range(P)}
    return [held[block_of(r, t_next)] for r in range(P)]


def copy_runs(senders):
    """(dst0, src0, n) runs of consecutive destinations whose senders are
    consecutive too: each run is one contiguous copy of staged slabs."""
    runs = []
    for r, s in enumerate(senders):
        if runs and runs[-1][0] + runs[-1][2] == r and runs[-1][1] + runs[-1][2] == s:
            runs[-1] = (runs[-1][0], runs[-1][1], runs[-1][2] + 1)
        else:
            runs.append((r, s, 1))
    return runs


def shard_segs(S: int, P: int, layout: str, r: int) -> capi.sca_segs:
    """Global positions of shard r's rows, in the shard's row order."""
    if layout == "zigzag":
        c = S // (2 * P)
        return capi.segs(2, c, (r * c, (2 * P - 1 - r) * c))
    n = S // P
    return capi.segs(1, n, (r * n, 0))


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


AUTO_FUSED_MAX_ROWS = 4096


def resolve_schedule(schedule, S, P, visit="ring"):
    """The schedule "auto" stands for at these sizes; others unchanged."""
    if schedule != "auto":
        return schedule
    if visit == "ring" and (P == 1 or S // P <= AUTO_FUSED_MAX_ROWS):
        return "fused"
    return "ring"


class ShardedCausalAttention:
    """Buffers and launch schedule of one sharded attention configuration.

    Create once, then call ``forward`` (and ``backward``) per step; nothing is
    allocated per call.  Inputs are [B, H, S, D] tensors in natural order, of
    ``dtype`` (bf16 or fp32), contiguous, on the current CUDA device.
    Outputs are fp32 [B, H, S, D] (and lse [B, H, S], natural log).
    ``backward`` reads the q, k, v of the last ``forward`` (kept by
    reference) unless they are passed again.  With ``kv_heads`` < H
    (grouped-query attention) k and v, and dk and dv, have kv_heads heads;
    query head h reads key/value head h // (H // kv_heads).
    """

    def __init__(self, B, H, S, D, P, layout="zigzag", dtype=torch.bfloat16, head_groups=1,
                 schedule="auto", scale=None, causal=True, algo=capi.SCA_ALGO_AUTO, backward=False,
                 bf16_out=False, device=None, addressing="auto", kv_heads=None, f16_staging=True,
                 visit="ring", inner=None, group_steps=True):
        if layout not in ("zigzag", "contiguous"):
            raise ValueError(f"layout {layout!r}")
        if schedule not in ("auto", "ring", "direct", "fused"):
            raise ValueError(f"schedule {schedule!r}")
        if visit == "ring":
            inner = P
        elif visit == "double_ring":
            if inner is None or inner < 1 or P % inner:
                raise ValueError(f"double_ring needs an inner ring size dividing P={P} (got {inner})")
        else:
            raise ValueError(f"visit {visit!r}")
        self.schedule_requested = schedule
        schedule = resolve_schedule(schedule, S, P, visit)
        if addressing not in ("auto", "position", "permuted"):
            raise ValueError(f"addressing {addressing!r}")
        if dtype not in _DT:
            raise ValueError(f"dtype {dtype}")
        if S % (2 * P if layout == "zigzag" else P):
            raise ValueError(f"S={S} not divisible into {P} {layout} shards")
        Hkv = H if kv_heads is None else int(kv_heads)
        if Hkv < 1 or H % Hkv:
            raise ValueError(f"kv_heads={kv_heads} must divide H={H}")
        if H % head_groups or Hkv % head_groups:
            raise ValueError("head_groups must divide H and kv_heads")
        if head_groups * P > capi.SCA_MAX_ITEMS:
            raise ValueError(f"{head_groups * P} virtual ranks > {capi.SCA_MAX_ITEMS}")
        zig = layout == "zigzag"
        seg_len = S // (2 * P) if zig else S // P
        if addressing == "auto":
            addressing = "position" if seg_len % 128 == 0 else "permuted"
        if addressing == "position" and seg_len % 128:
            raise ValueError(f"position addressing needs shard segments of a multiple of 128 rows ({seg_len})")
        self.B, self.H, self.S, self.D, self.P = B, H, S, D, P
        self.G, self.Hg = head_groups, H // head_groups
        self.Hkv, self.Hkvg = Hkv, Hkv // head_groups   # key/value heads: all, per head group
        self.layout, self.schedule, self.dtype = layout, schedule, dtype
        self.visit, self.inner = visit, inner
        # direct schedule: the forward's partials of all steps in as few
        # launches as possible, or (False) one launch per step as the ring
        # sends them, only without staging copies
        self.group_steps = group_steps
        self.addressing = addressing
        self.pos = addressing == "position"
        fused = schedule == "fused"
        self.perm = zig and not self.pos and not fused   # shard-major permuted copies
        self.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        self.causal, self.algo, self.backward_enabled = causal, algo, backward
        self.n_r = S // P                       # rows per shard
        self.eb = torch.tensor([], dtype=dtype).element_size()
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.device = dev
        z = lambda *shape, dt=torch.float32: torch.empty(shape, dtype=dt, device=dev)
        self.qp = z(B, H, S, D, dt=dtype) if self.perm else None
        self.kp = z(B, Hkv, S, D, dt=dtype) if self.perm else None
        self.vp = z(B, Hkv, S, D, dt=dtype) if self.perm else None
        self.o_parts = z(P, B, H, S, D) if not fused else None
        self.lse_parts = z(P, B, H, S) if not fused else None
        self.o = z(B, H, S, D)
        self.lse = z(B, H, S)
        self.o_bf16 = z(B, H, S, D, dt=torch.bfloat16) if bf16_out else None
        ring = schedule == "ring" and P > 1
        # staging buffers: step t reads buffer t % n_stage, and the copy that
        # fills it for step t+1 may start once step t+1-n_stage is done.  With
        # three, each hand-off has two steps of compute to hide behind.
        self.n_stage = 3 if P > 3 else 2
        self.stage_k = [z(self.G, P, B, self.Hkvg, self.n_r, D, dt=dtype) for _ in range(self.n_stage)] if ring else None
        self.stage_v = [z(self.G, P, B, self.Hkvg, self.n_r, D, dt=dtype) for _ in range(self.n_stage)] if ring else None
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if backward:
            self.delta = z(B, H, S)
            self.dq = z(B, H, S, D)
            self.dk = z(B, Hkv, S, D)
            self.dv = z(B, Hkv, S, D)
            self.dop = z(B, H, S, D, dt=dtype) if self.perm else None
            self.lse_p = z(B, H, S) if self.perm else None
            self.delta_p = z(B, H, S) if self.perm else None
            self.dq_p = z(B, H, S, D) if self.perm else None
            self.dk_p = z(B, Hkv, S, D) if self.perm else None
            self.dv_p = z(B, Hkv, S, D) if self.perm else None
        # the tensor-core backward runs S, dK, dQ (and, grouped, dP, dV) as
        # fp16 products: its fp16 queries (and grouped dO) are cast once per
        # backward here rather than tile by tile in every key-tile CTA
        self.f16_in = f16_input_flags(backward and f16_staging, dtype, algo, H, Hkv)
        self.q16 = z(B, H, S, D, dt=torch.float16) if self.f16_in else None
        self.do16 = z(B, H, S, D, dt=torch.float16) if self.f16_in & capi.SCA_F16_DOUT else None
        # the hand-offs run on a stream of their own, at high priority: their
        # small copy blocks are dispatched ahead of attention CTAs and fit
        # beside them on the SMs
        self.copy_stream = torch.cuda.Stream(device=dev, priority=-1) if ring else None
        self.ev_ready = torch.cuda.Event()
        self.ev_staged = [torch.cuda.Event() for _ in range(P)]
        self.ev_done = [torch.cuda.Event() for _ in range(P)]
        self._inputs = None
        self.launches = 0   # kernels + copies issued by the last forward/backward
        self.kernels = 0    # kernels alone
        self.staged_bytes = 0   # bytes copied into staging buffers by the last forward/backward
        # when set to a list, each staging pass of a ring step appends its
        # (start, end) events, recorded on the copy stream
        self.stage_events = None

    # ------------------------------------------------------------ helpers

    def _permute(self, src, dst, row_bytes, inverse, stream):
        capi.zigzag_permute(_ptr(src), _ptr(dst), src.numel() // (self.S * (row_bytes // src.element_size())),
                            self.S, row_bytes, self.P, inverse, _ptr(self.status), stream)
        self.launches += 1
        self.kernels += 1

    def _rows(self, g, r):
        """Element offset (in rows of one head's sequence) of rank (g, r)'s
        slab: the head group's first row, plus the shard's slab offset when
        the tensors are shard-major (position addressing finds the rows by
        their positions instead)."""
        off = g * self.Hg * self.S
        return off if self.pos else off + r * self.n_r

    def _kv_rows(self, g, j):
        """The same for key/value-side tensors (kv_heads heads)."""
        off = g * self.Hkvg * self.S
        return off if self.pos else off + j * self.n_r

    # ------------------------------------------------- kernel descriptions

    def uses_tensor_cores(self, kind: str) -> bool:
        return self.dtype == torch.bfloat16 and self.algo != capi.SCA_ALGO_SIMT

    def kernel_name(self, kind: str) -> str:
        tc = self.uses_tensor_cores(kind)
        if kind == "fwd":
            return "fwd_tc_kernel" if tc else "fwd_simt_kernel"
        return "bwd_tc_kernel" if tc else "dq_simt_kernel+dkv_simt_kernel"

    def kernel_sources(self, kind: str):
        tc = self.uses_tensor_cores(kind)
        if kind == "fwd":
            return ["fwd_tc.cu", "ptx.cuh", "common.cuh"] if tc else ["attn_simt.cu", "common.cuh"]
        return ["bwd_tc.cu", "ptx.cuh", "common.cuh"] if tc else ["attn_simt.cu", "common.cuh"]

    def kernels_per_attn_call(self, kind: str) -> int:
        return 2 if (kind == "bwd" and not self.uses_tensor_cores("bwd")) else 1

    def _dims(self, kv_view, backward=False, accumulate=0, q_by_pos=0, kv_by_pos=0, dkv_by_pos=0):
        d = capi.sca_attn_dims()
        d.B, d.H, d.D = self.B, self.Hg, self.D
        d.kv_heads = self.Hkvg
        d.dtype = _DT[self.dtype]
        d.causal = 1 if self.causal else 0
        d.algo = self.algo
        d.scale = self.scale
        d.accumulate = accumulate
        S, D, H = self.S, self.D, self.H
        d.q = capi.view(H * S * D, S * D, D)
        d.kv = kv_view
        d.o = capi.view(H * S * D, S * D, D)
        d.dkv = capi.view(self.Hkv * S * D, S * D, D)
        d.lse_b, d.lse_h = H * S, S
        d.q_by_pos, d.kv_by_pos, d.dkv_by_pos = int(q_by_pos), int(kv_by_pos), int(dkv_by_pos)
        d.f16_inputs = self.f16_in if backward else 0
        return d

    def _home_kv_view(self):
        return capi.view(self.Hkv * self.S * self.D, self.S * self.D, self.D)

    def _stage_kv_view(self):
        return capi.view(self.Hkvg * self.n_r * self.D, self.n_r * self.D, self.D)

    def block(self, r: int, t: int) -> int:
        """Key/value block shard r holds (visits) at step t."""
        if self.visit == "double_ring":
            return double_ring_block(r, t, self.P, self.inner)
        return ring_block(r, t, self.P)

    def _kv_ptrs(self, k_home, v_home, t, g, r):
        """(k, v) base pointers of the block rank (g, r) holds at step t."""
        if self.stage_k is None or t == 0:
            off = self._kv_rows(g, self.block(r, t)) * self.D * self.eb
            return _ptr(k_home) + off, _ptr(v_home) + off
        buf = t % self.n_stage
        return _ptr(self.stage_k[buf][g, r]), _ptr(self.stage_v[buf][g, r])

    def _stage(self, k_home, v_home, t_next):
        """Hand-off into the spare buffer: rank (g, r) receives the block it
        visits at step t_next from the rank that holds it at step t_next - 1
        (its left neighbour on the ring; on the double ring a neighbour in
        its group, or a rank of the previous group on an outer hop).  Every
        copy of the hand-off goes out in one ring_stage_copies launch."""
        P, B, Hg, n_r, D, eb = self.P, self.B, self.Hkvg, self.n_r, self.D, self.eb
        cs = self.copy_stream.cuda_stream
        ns = self.n_stage
        dst_k, dst_v = self.stage_k[t_next % ns], self.stage_v[t_next % ns]
        row = D * eb
        blk = B * Hg * n_r
        copies = []
        for g in range(self.G):
            if t_next == 1:   # the senders' blocks are still at home
                for r in range(P):
                    segs = shard_segs(self.S, P, self.layout, self.block(r, 1))
                    for b in range(B):
                        off = ((b * self.Hkv + g * Hg) * self.S) * row
                        for home, dst in ((k_home, dst_k), (v_home, dst_v)):
                            if self.pos:   # gather the block's chunks from natural order
                                w = segs.len * row
                                for i in range(segs.n):
                                    copies.append(capi.copy2d(_ptr(home) + off + segs.start[i] * row,
                                                              _ptr(dst[g, r, b]) + i * w, Hg, w, self.S * row,
                                                              segs.n * w))
                            else:
                                w = n_r * row
                                copies.append(capi.copy2d(_ptr(home) + off + self.block(r, 1) * w,
                                                          _ptr(dst[g, r, b]), Hg, w, self.S * row, w))
            else:             # the senders' staged blocks: one copy per run of consecutive ranks
                src_k, src_v = self.stage_k[(t_next - 1) % ns], self.stage_v[(t_next - 1) % ns]
                for r0, s0, n in copy_runs(hop_senders(self.block, t_next, P)):
                    for src, dst in ((src_k, dst_k), (src_v, dst_v)):
                        w = n * blk * row
                        copies.append(capi.copy2d(_ptr(src[g, s0]), _ptr(dst[g, r0]), 1, w, w, w))
        for lo in range(0, len(copies), capi.SCA_MAX_COPIES):
            capi.ring_stage_copies(copies[lo:lo + capi.SCA_MAX_COPIES], cs)
            self.launches += 1
        self.staged_bytes += sum(c.height * c.width for c in copies)

    def _ring(self, k_home, v_home, launch_step):
        """Run launch_step(t, kv_ptrs(g, r), kv_view, home) for t = 0..P-1
        with the staging copies of step t+1 overlapped on the copy stream;
        `home` says whether the blocks are read from their home rows.

        Step t's kernel is enqueued before the copies of step t+1: those
        copies wait only for the step that last read the buffer they
        overwrite (t+1-n_stage), so the host's time spent issuing them
        overlaps step t on the GPU instead of delaying its launch."""
        cur = torch.cuda.current_stream(self.device)
        ring = self.stage_k is not None
        if ring:
            self.ev_ready.record(cur)
            self.copy_stream.wait_event(self.ev_ready)
        for t in range(self.P):
            if ring and t >= 1:
                cur.wait_event(self.ev_staged[t])
            home = not ring or t == 0
            view = self._home_kv_view() if home else self._stage_kv_view()
            launch_step(t, lambda g, r: self._kv_ptrs(k_home, v_home, t, g, r), view, home)
            self.ev_done[t].record(cur)
            if ring and t + 1 < self.P:
                with torch.cuda.stream(self.copy_stream):
                    # the buffer this copy fills was last read by step
                    # t+1-n_stage (step 0 reads home rows, no buffer)
                    if t + 1 - self.n_stage >= 1:
                        self.copy_stream.wait_event(self.ev_done[t + 1 - self.n_stage])
                    if self.stage_events is not None:
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(self.copy_stream)
                    self._stage(k_home, v_home, t + 1)
                    if self.stage_events is not None:
                        e1.record(self.copy_stream)
                        self.stage_events.append((e0, e1))
                    self.ev_staged[t + 1].record(self.copy_stream)
        if ring:  # the staging buffers are reused by the next call
            cur.wait_stream(self.copy_stream)

    # ------------------------------------------------------------ forward

    def forward(self, q, k, v):
        self._check_inputs(q)
        self._check_inputs(k, v, heads=self.Hkv)
        self.launches = self.kernels = self.staged_bytes = 0
        self._inputs = (q, k, v)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        if self.schedule == "fused":
            return self._forward_fused(q, k, v, stream)
        row = self.D * self.eb
        if self.perm:
            self._permute(q, self.qp, row, 0, stream)
            self._permute(k, self.kp, row, 0, stream)
            self._permute(v, self.vp, row, 0, stream)
            qh, kh, vh = self.qp, self.kp, self.vp
        else:
            qh, kh, vh = q, k, v
        S, D, H, P = self.S, self.D, self.H, self.P
        eb = self.eb
        st_ptr = _ptr(self.status)

        def step_items(t, kv_ptrs):
            items = []
            for g in range(self.G):
                for r in range(P):
                    it = capi.sca_fwd_item()
                    rows = self._rows(g, r)
                    it.q = _ptr(qh) + rows * D * eb
                    it.k, it.v = kv_ptrs(g, r)
                    it.o = _ptr(self.o_parts[t]) + rows * D * 4
                    it.lse = _ptr(self.lse_parts[t]) + rows * 4
                    it.q_pos = shard_segs(S, P, self.layout, r)
                    it.kv_pos = shard_segs(S, P, self.layout, self.block(r, t))
                    items.append(it)
            return items

        def step(t, kv_ptrs, kv_view, home):
            dims = self._dims(kv_view, q_by_pos=self.pos, kv_by_pos=self.pos and home)
            capi.attn_fwd_shard(step_items(t, kv_ptrs), dims, st_ptr, stream)
            self.launches += 1
            self.kernels += 1

        if self.schedule == "direct" and self.group_steps:
            # every block is read from its home rows (the all-gather reading),
            # so the partials of all P steps are independent: they go out
            # together, up to SCA_MAX_ITEMS items per launch
            items = []
            for t in range(P):
                items += step_items(t, lambda g, r, t=t: self._kv_ptrs(kh, vh, t, g, r))
            dims = self._dims(self._home_kv_view(), q_by_pos=self.pos, kv_by_pos=self.pos)
            for lo, hi in launch_groups(len(items)):
                capi.attn_fwd_shard(items[lo:hi], dims, st_ptr, stream)
                self.launches += 1
                self.kernels += 1
        else:
            self._ring(kh, vh, step)
        rows = self.B * H * S
        capi.attn_merge_lse(_ptr(self.o_parts), _ptr(self.lse_parts), P, rows, D, rows * D, rows,
                            _ptr(self.o), _ptr(self.lse), _ptr(self.o_bf16) if self.o_bf16 is not None else 0,
                            P if self.perm else 0, S, stream)
        self.launches += 1
        self.kernels += 1
        return self.o, self.lse

    def _forward_fused(self, q, k, v, stream):
        """Every shard in one launch: each head group is one item over the
        whole sequence, so every CTA's online softmax runs over all blocks
        and writes the final O and lse."""
        S, D, eb = self.S, self.D, self.eb
        items = []
        for g in range(self.G):
            rows, kv_rows = g * self.Hg * S, g * self.Hkvg * S
            it = capi.sca_fwd_item()
            it.q, it.k, it.v = _ptr(q) + rows * D * eb, _ptr(k) + kv_rows * D * eb, _ptr(v) + kv_rows * D * eb
            it.o = _ptr(self.o) + rows * D * 4
            it.lse = _ptr(self.lse) + rows * 4
            it.q_pos = capi.segs(1, S, (0, 0))
            it.kv_pos = capi.segs(1, S, (0, 0))
            items.append(it)
        capi.attn_fwd_shard(items, self._dims(self._home_kv_view()), _ptr(self.status), stream)
        self.launches += 1
        self.kernels += 1
        if self.o_bf16 is not None:   # a one-partial merge is the bf16 rounding pass
            rows = self.B * self.H * S
            capi.attn_merge_lse(_ptr(self.o), _ptr(self.lse), 1, rows, D, rows * D, rows, _ptr(self.o),
                                _ptr(self.lse), _ptr(self.o_bf16), 0, S, stream)
            self.launches += 1
            self.kernels += 1
        return self.o, self.lse

    # ----------------------------------------------------------- backward

    def backward(self, do, q=None, k=None, v=None):
        """Gradients (dq, dk, dv) fp32 natural order for the inputs of the
        last ``forward``."""
        if not self.backward_enabled:
            raise RuntimeError("plan built without backward=True")
        if q is None:
            if self._inputs is None:
                raise RuntimeError("backward before forward")
            q, k, v = self._inputs
        self._check_inputs(do, q)
        self._check_inputs(k, v, heads=self.Hkv)
        self.launches = self.kernels = self.staged_bytes = 0
        stream = torch.cuda.current_stream(self.device).cuda_stream
        S, D, H, P, B = self.S, self.D, self.H, self.P, self.B
        eb = self.eb
        rows_all = B * H * S
        capi.attn_bwd_delta(_ptr(self.o), _ptr(do), _DT[self.dtype], _ptr(self.delta), rows_all, D, stream)
        self.launches += 1
        self.kernels += 1
        if self.schedule == "fused":
            q, do = self._cast_f16(q, do, stream)
            return self._backward_fused(do, q, k, v, stream)
        if self.perm:
            self._permute(do, self.dop, D * eb, 0, stream)
            self._permute(self.lse, self.lse_p, 4, 0, stream)
            self._permute(self.delta, self.delta_p, 4, 0, stream)
            qh, kh, vh, doh = self.qp, self.kp, self.vp, self.dop
            lse_h, dl_h = self.lse_p, self.delta_p
            dq, dk, dv = self.dq_p, self.dk_p, self.dv_p
        else:
            qh, kh, vh, doh = q, k, v, do
            lse_h, dl_h = self.lse, self.delta
            dq, dk, dv = self.dq, self.dk, self.dv
        qh, doh = self._cast_f16(qh, doh, stream)
        st_ptr = _ptr(self.status)

        def step(t, kv_ptrs, kv_view, home):
            items = []
            for g in range(self.G):
                for r in range(P):
                    j = self.block(r, t)
                    qo, ko = self._rows(g, r), self._kv_rows(g, j)
                    it = capi.sca_bwd_item()
                    it.q = _ptr(qh) + qo * D * eb
                    it.dout = _ptr(doh) + qo * D * eb
                    it.k, it.v = kv_ptrs(g, r)
                    it.lse = _ptr(lse_h) + qo * 4
                    it.delta = _ptr(dl_h) + qo * 4
                    it.dq = _ptr(dq) + qo * D * 4
                    it.dk = _ptr(dk) + ko * D * 4
                    it.dv = _ptr(dv) + ko * D * 4
                    it.q_pos = shard_segs(S, P, self.layout, r)
                    it.kv_pos = shard_segs(S, P, self.layout, j)
                    items.append(it)
            dims = self._dims(kv_view, backward=True, accumulate=1 if t > 0 else 0, q_by_pos=self.pos,
                              kv_by_pos=self.pos and home, dkv_by_pos=self.pos)
            capi.attn_bwd_shard(items, dims, st_ptr, stream)
            self.launches += 1
            self.kernels += self.kernels_per_attn_call("bwd")

        self._ring(kh, vh, step)
        if self.perm:
            self._permute(dq, self.dq, D * 4, 1, stream)
            self._permute(dk, self.dk, D * 4, 1, stream)
            self._permute(dv, self.dv, D * 4, 1, stream)
        return self.dq, self.dk, self.dv

    def _cast_f16(self, q, do, stream):
        """The backward's query (and grouped dO) tensors: fp16 copies when the
        plan stages them, else the inputs themselves."""
        if self.f16_in & capi.SCA_F16_Q:
            capi.cast_bf16_to_f16(_ptr(q), _ptr(self.q16), q.numel(), _ptr(self.status), stream)
            q = self.q16
            self.launches += 1
            self.kernels += 1
        if self.f16_in & capi.SCA_F16_DOUT:
            capi.cast_bf16_to_f16(_ptr(do), _ptr(self.do16), do.numel(), _ptr(self.status), stream)
            do = self.do16
            self.launches += 1
            self.kernels += 1
        return q, do

    def _backward_fused(self, do, q, k, v, stream):
        """Every shard in one launch: each head group is one item over the
        whole sequence; every key tile's dK/dV is complete in its CTA and
        written once, dQ is summed over key tiles."""
        S, D, eb = self.S, self.D, self.eb
        items = []
        for g in range(self.G):
            rows, kv_rows = g * self.Hg * S, g * self.Hkvg * S
            it = capi.sca_bwd_item()
            it.q, it.k, it.v = _ptr(q) + rows * D * eb, _ptr(k) + kv_rows * D * eb, _ptr(v) + kv_rows * D * eb
            it.dout = _ptr(do) + rows * D * eb
            it.lse, it.delta = _ptr(self.lse) + rows * 4, _ptr(self.delta) + rows * 4
            it.dq = _ptr(self.dq) + rows * D * 4
            it.dk, it.dv = _ptr(self.dk) + kv_rows * D * 4, _ptr(self.dv) + kv_rows * D * 4
            it.q_pos = capi.segs(1, S, (0, 0))
            it.kv_pos = capi.segs(1, S, (0, 0))
            items.append(it)
        capi.attn_bwd_shard(items, self._dims(self._home_kv_view(), backward=True), _ptr(self.status), stream)
        self.launches += 1
        self.kernels += self.kernels_per_attn_call("bwd")
        return self.dq, self.dk, self.dv

    def read_status(self) -> int:
        """Synchronise and return the device status word (0 = OK)."""
        return capi.sca_read_status(_ptr(self.status), torch.cuda.current_stream(self.device).cuda_stream)

    def _check_inputs(self, *ts, heads=None):
        H = self.H if heads is None else heads
        for t in ts:
            if t.dtype != self.dtype or t.device != self.device or not t.is_contiguous() or \
                    tuple(t.shape) != (self.B, H, self.S, self.D):
                raise ValueError(f"expected contiguous {self.dtype} [{self.B},{H},{self.S},{self.D}] "
                                 f"on {self.device}, got {t.dtype} {tuple(t.shape)} on {t.device}")
