"""Sharded causal softmax attention for GB300 (sm_103a).

The computation - causal softmax attention split into P context shards, each
(query shard, key/value block) partial kept as an (o, lse) pair and merged
exactly by log-sum-exp rescaling - runs in the CUDA kernels of libsca.so
behind the C ABI of ``include/sca.h``.  ``capi`` is the ctypes binding of
that ABI (same function names); ``ShardedCausalAttention`` is the host-side
schedule of P virtual shards (zigzag or contiguous, ring visiting order with
multi-buffered staging, head groups; or the double ring) on one GPU; ``ShardedLinearAttention``
the schedule of causal linear attention over P contiguous shards that pass
their states point to point (LASP).
"""
from . import capi
from .capi import (ScaError, attn_bwd_delta, attn_bwd_shard, attn_fwd_shard, attn_merge_lse,
                   ring_stage_block, sca_read_status, sca_version, zigzag_permute)
from .lasp import ShardedLinearAttention
from .sharded import ShardedCausalAttention, ring_block, shard_segs

__all__ = ["capi", "ScaError", "attn_fwd_shard", "attn_bwd_shard", "attn_merge_lse", "zigzag_permute",
           "ring_stage_block", "attn_bwd_delta", "sca_read_status", "sca_version", "ShardedCausalAttention",
           "ring_block", "shard_segs", "ShardedLinearAttention"]
