"""P virtual shards of causal linear attention on one GPU (linear attention
sequence parallelism: "Effiziente Parallelisierung linearer
Aufmerksamkeitssequenzen fuer skalierbare Sprachmodelle" - intermediate
states exchanged point to point between shards, the right-product trick).

    o_t = scale * sum_{s <= t} (q_t . k_s) v_s

Forward: every shard sums k^T v over its blocks (``lasp_block_states`` then
``lasp_scan``, which leaves each block the state of the shard's blocks
before it), the shard totals travel from shard to shard
(``lasp_exchange``: shard r receives the sum of everything before it from
shard r-1), and ``lasp_fwd`` combines, per block, the masked left product
inside the block with the right product of its queries and the state.
Backward: the same with q^T dO states travelling from later shards to
earlier ones.  The shards are contiguous (linear attention costs the same
per row, so no zigzag).  bf16 inputs with D = 128 run on the tensor-core
kernels (blocks of up to 4096 rows, carried through in sub-blocks of 128);
fp32 inputs and D = 64 on the fp32 CUDA-core kernels (blocks of 64 rows).
PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import math

import torch

from . import capi

_DT = {torch.bfloat16: capi.SCA_BF16, torch.float32: capi.SCA_F32}


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def default_block(B: int, H: int, S: int, D: int, P: int, dtype) -> int:
    """Rows per stored state: 64 on the CUDA-core path (fp32 inputs or
    D = 64); on the tensor cores the largest block (up to 4096 rows) that
    tiles every shard and still gives at least 128 blocks to spread over
    the SMs (the smallest that tiles, else 128)."""
    if dtype != torch.bfloat16 or D != 128:
        return capi.SCA_LASP_BLOCK_F32
    fits = [b for b in (4096, 2048, 1024, 512, 256, 128) if S % (b * P) == 0]
    return next((b for b in fits if B * H * (S // b) >= 128), fits[-1] if fits else capi.SCA_LASP_BLOCK_TC)


class ShardedLinearAttention:
    """Buffers and launch schedule of one LASP configuration; inputs are
    contiguous [B, H, S, D] tensors of ``dtype``, outputs fp32."""

    def __init__(self, B, H, S, D, P, dtype=torch.bfloat16, scale=None, backward=False, device=None,
                 block=None):
        if dtype not in _DT:
            raise ValueError(f"dtype {dtype}")
        if D not in (64, 128):
            raise ValueError(f"D={D}: only 64 and 128")
        tc_ok = dtype == torch.bfloat16 and D == 128
        sub = capi.SCA_LASP_BLOCK_TC
        if block is None:
            block = default_block(B, H, S, D, P, dtype)
        tc = block != capi.SCA_LASP_BLOCK_F32
        if tc and (block % sub or not sub <= block <= 4096 or not tc_ok):
            raise ValueError(f"block={block}: 64, or a multiple of {sub} up to 4096 for bf16 inputs with D = 128")
        blk = self.block = block
        self.tensor_cores = tc
        if S % (blk * P):
            raise ValueError(f"S={S} must be a multiple of {blk}*P={blk * P}")
        self.B, self.H, self.S, self.D, self.P, self.dtype = B, H, S, D, P, dtype
        self.BH = B * H
        self.scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
        self.backward_enabled = backward
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.device = dev
        z = lambda *shape: torch.empty(shape, dtype=torch.float32, device=dev)
        nblk = S // blk
        self.st_f = z(self.BH, nblk, D, D)       # per block: k^T v of the shard's blocks before it
        self.tot_f = z(self.BH, P, D, D)
        self.in_f = z(self.BH, P, D, D)          # what each shard receives from the one before
        self.o = z(B, H, S, D)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        if backward:
            self.st_b = z(self.BH, nblk, D, D)   # per block: q^T dO of the shard's blocks after it
            self.tot_b = z(self.BH, P, D, D)
            self.in_b = z(self.BH, P, D, D)
            self.dq, self.dk, self.dv = z(B, H, S, D), z(B, H, S, D), z(B, H, S, D)
        self._inputs = None
        self.kernels = 0

    def forward(self, q, k, v):
        self._check(q, k, v)
        self._inputs = (q, k, v)
        st = torch.cuda.current_stream(self.device).cuda_stream
        dt, BH, S, D, P = _DT[self.dtype], self.BH, self.S, self.D, self.P
        blk, sp = self.block, _ptr(self.status)
        capi.lasp_block_states(_ptr(k), _ptr(v), dt, _ptr(self.st_f), BH, S, D, blk, sp, st)
        capi.lasp_scan(_ptr(self.st_f), _ptr(self.tot_f), BH, S, D, P, blk, 0, st)
        capi.lasp_exchange(_ptr(self.tot_f), _ptr(self.in_f), BH, D, P, 0, st)
        capi.lasp_fwd(_ptr(q), _ptr(k), _ptr(v), dt, _ptr(self.st_f), _ptr(self.in_f), _ptr(self.o), BH, S, D, P,
                      blk, self.scale, sp, st)
        self.kernels = 4
        return self.o

    def backward(self, do):
        if not self.backward_enabled:
            raise RuntimeError("plan built without backward=True")
        if self._inputs is None:
            raise RuntimeError("backward before forward")
        q, k, v = self._inputs
        self._check(do)
        st = torch.cuda.current_stream(self.device).cuda_stream
        dt, BH, S, D, P = _DT[self.dtype], self.BH, self.S, self.D, self.P
        blk, sp = self.block, _ptr(self.status)
        capi.lasp_block_states(_ptr(q), _ptr(do), dt, _ptr(self.st_b), BH, S, D, blk, sp, st)
        capi.lasp_scan(_ptr(self.st_b), _ptr(self.tot_b), BH, S, D, P, blk, 1, st)
        capi.lasp_exchange(_ptr(self.tot_b), _ptr(self.in_b), BH, D, P, 1, st)
        capi.lasp_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), dt, _ptr(self.st_f), _ptr(self.in_f), _ptr(self.st_b),
                      _ptr(self.in_b), _ptr(self.dq), _ptr(self.dk), _ptr(self.dv), BH, S, D, P, blk, self.scale,
                      sp, st)
        self.kernels = 6 if self.tensor_cores else 5
        return self.dq, self.dk, self.dv

    # ---- the interface the benchmark reads (mirrors ShardedCausalAttention)

    @property
    def addressing(self):
        return "contiguous shards, blocks of %d rows" % self.block

    def roofline_bound(self, kind: str) -> str:
        """The tensor-core kernels do six 128x128x128 MMA groups per 128-row
        sub-block (25 MFLOP) against ~180 KB moved (input and output rows,
        a share of the block state): ~140 FLOP per byte, under the bf16
        ridge (~290 FLOP/B), so bytes bound.  The CUDA-core kernels are
        bound by fp32 FMA issue."""
        return "hbm" if self.tensor_cores else "alu"

    def algorithmic_bytes(self, kind: str) -> int:
        """Bytes one lasp_fwd / lasp_bwd call must move: its input rows
        (bf16), per block its fp32 D x D state(s), and its fp32 output rows
        (the per-shard inputs are shared by a shard's blocks and stay in
        L2)."""
        nb = self.BH * (self.S // self.block)
        rows, D = self.block, self.D
        if kind == "fwd":
            return nb * (3 * rows * D * 2 + D * D * 4 + rows * D * 4)
        return nb * (4 * rows * D * 2 + 2 * D * D * 4 + 3 * rows * D * 4)

    def uses_tensor_cores(self, kind: str) -> bool:
        return self.tensor_cores

    def kernel_name(self, kind: str) -> str:
        if self.tensor_cores:
            return "block_kernel<kFwd>" if kind == "fwd" else "block_kernel<kDq,kDk,kDv>"
        return "fwd_kernel" if kind == "fwd" else "dq_kernel+dkdv_kernel"

    def kernel_sources(self, kind: str):
        if self.tensor_cores:
            return ["lasp_tc.cu", "lasp.cu", "ptx.cuh", "common.cuh"]
        return ["lasp.cu", "common.cuh"]

    def read_status(self) -> int:
        """Synchronise and return the device status word (0 = OK; the
        tensor-core kernels record a timed-out wait there)."""
        return capi.sca_read_status(_ptr(self.status), torch.cuda.current_stream(self.device).cuda_stream)

    def _check(self, *ts):
        for t in ts:
            if t.dtype != self.dtype or t.device != self.device or not t.is_contiguous() or \
                    tuple(t.shape) != (self.B, self.H, self.S, self.D):
                raise ValueError(f"expected contiguous {self.dtype} [{self.B},{self.H},{self.S},{self.D}] "
                                 f"on {self.device}, got {t.dtype} {tuple(t.shape)} on {t.device}")
