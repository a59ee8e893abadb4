"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module holds no arithmetic of the attention method: it only draws
normally distributed tensors from a seeded CPU generator, rounds them to the
storage dtype, and picks seeded row samples.  Both the fp64 oracle and the
GPU path read their inputs from here, so the two compute on identical values.

Workloads (shapes, dtypes, seeds, shard counts) are the synthetic cases this
library is checked and measured on; head dim 128 matches the 7B decoder
(h=4096, 32 heads) that the TSP news page ("Zyphra presenta el paralelismo de
secuencia y tensor (TSP)", section "Resultados de memoria y rendimiento")
uses as its reference model.  The grouped-query case stands for the 7B-GQA
model of "Avances en la capacitacion de LLMs de secuencia larga" (section
"Evaluacion y Comparacion con Sistemas Existentes"): 32 query heads; the page
gives no key/value head count, 8 is the reading taken.  The linear-attention
case (LASP, "Effiziente Parallelisierung linearer Aufmerksamkeitssequenzen
fuer skalierbare Sprachmodelle") takes the training shape of the softmax one.

Recipe (fixed, so a reader can regenerate any case):
  g = torch.Generator('cpu').manual_seed(seed)
  draw torch.randn in the order Q [B,H,S,D], K, V [B,Hkv,S,D] (Hkv = H
  unless grouped-query), dO [B,H,S,D], all float32
  round to the storage dtype (bf16 round-to-nearest-even) when it is bf16
  Q *= q_mult (exact in bf16 for q_mult = 2)
Sampled rows: torch.Generator('cpu').manual_seed(10_000 + seed), per (b, h)
randperm(S)[:n] sorted ascending.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str            # "f32" or "bf16": storage/input dtype
    seed: int
    P: int                # context shards
    layout: str           # "contiguous" or "zigzag"
    q_mult: float = 1.0
    head_groups: int = 1  # 2D head x context split
    backward: bool = False
    schedule: str = "auto"      # "auto", "ring" (staged KV blocks), "direct" or "fused"
    sample_rows: int = 0        # 0: oracle checks every row
    description: str = ""
    kv_heads: int | None = None  # grouped-query attention: key/value heads
    method: str = "softmax"      # "softmax" attention, or "lasp" (causal linear attention)


WORKLOADS = {
    "tiny_f32": Workload(
        "tiny_f32", B=1, H=2, S=256, D=64, dtype="f32", seed=0, P=2,
        layout="contiguous",
        description="tiny fp32 case: B1 H2 S256 D64, P=2 contiguous shards"),
    "fwd_s8k": Workload(
        "fwd_s8k", B=1, H=16, S=8192, D=128, dtype="bf16", seed=1, P=4,
        layout="zigzag",
        description="causal forward B1 H16 S8192 D128 bf16, P=4 zigzag shards"),
    "ring_s128k": Workload(
        "ring_s128k", B=1, H=8, S=131072, D=128, dtype="bf16", seed=2, P=8,
        layout="zigzag", schedule="ring", sample_rows=256,
        description="ring emulation B1 H8 S131072 D128 bf16, P=8 zigzag, "
                    "KV blocks of 8192 in ring order, double-buffered staging"),
    "2d_s32k": Workload(
        "2d_s32k", B=2, H=32, S=32768, D=128, dtype="bf16", seed=3, P=4,
        layout="zigzag", q_mult=2.0, head_groups=4, sample_rows=256,
        description="2D head x context split B2 H32 S32768 D128 bf16, Q*2, "
                    "4 head groups x 4 zigzag shards"),
    "train_s32k": Workload(
        "train_s32k", B=1, H=16, S=32768, D=128, dtype="bf16", seed=4, P=4,
        layout="zigzag", backward=True, sample_rows=256,
        description="training step fwd+bwd B1 H16 S32768 D128 bf16, P=4 zigzag"),
    "gqa_s32k": Workload(
        "gqa_s32k", B=1, H=32, S=32768, D=128, dtype="bf16", seed=5, P=4,
        layout="zigzag", backward=True, sample_rows=256, kv_heads=8,
        description="grouped-query training step fwd+bwd B1 H32 (8 key/value heads) S32768 D128 bf16, "
                    "P=4 zigzag"),
    "lasp_s32k": Workload(
        "lasp_s32k", B=1, H=16, S=32768, D=128, dtype="bf16", seed=6, P=4, layout="contiguous",
        backward=True, sample_rows=256, method="lasp",
        description="linear attention (LASP) training step fwd+bwd B1 H16 S32768 D128 bf16, "
                    "P=4 contiguous shards passing states point to point"),
}


def _round(x: torch.Tensor, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        return x.to(torch.bfloat16)
    if dtype == "f32":
        return x
    raise ValueError(f"unknown dtype {dtype!r}")


def make_inputs(B: int, H: int, S: int, D: int, dtype: str, seed: int,
                q_mult: float = 1.0, with_do: bool = False, kv_heads: int | None = None):
    """Return (q, k, v[, do]) CPU tensors in the storage dtype: q, do
    [B,H,S,D]; k, v [B,kv_heads,S,D] (kv_heads = H by default)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    names = ["q", "k", "v"] + (["do"] if with_do else [])
    out = []
    for name in names:
        heads = H if (kv_heads is None or name in ("q", "do")) else kv_heads
        x = torch.randn([B, heads, S, D], generator=g, dtype=torch.float32)
        x = _round(x, dtype)
        if name == "q" and q_mult != 1.0:
            x = x * q_mult
        out.append(x)
    return tuple(out)


def workload_inputs(w: Workload, S: int | None = None, H: int | None = None):
    """Inputs of a named workload (optionally with fewer rows/heads for quick
    runs; a grouped-query workload keeps its query heads per key/value head)."""
    Hq = H or w.H
    kv = None if w.kv_heads is None else max(1, Hq * w.kv_heads // w.H)
    return make_inputs(w.B, Hq, S or w.S, w.D, w.dtype, w.seed,
                       q_mult=w.q_mult, with_do=w.backward, kv_heads=kv)


def sample_rows(B: int, H: int, S: int, n: int, seed: int) -> torch.Tensor:
    """Seeded sorted row indices, [B,H,n] int64 (one independent draw per (b,h))."""
    g = torch.Generator(device="cpu").manual_seed(10_000 + seed)
    out = torch.empty([B, H, n], dtype=torch.int64)
    for b in range(B):
        for h in range(H):
            out[b, h] = torch.sort(torch.randperm(S, generator=g)[:n]).values
    return out
