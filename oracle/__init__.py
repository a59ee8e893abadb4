"""fp64 CPU oracle for sharded causal softmax attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
``__graft_entry__`` and the ``cpu_baseline`` / reference leg of ``bench.py``
may import or run anything in this package.  The library (the CUDA kernels,
the C ABI and the Python binding in ``sharded_causal_softmax_gb300``) never
imports it and shares no code with it; the two meet only in the seeded input
generator ``seeded_inputs``, which holds no arithmetic of the method.

What it computes, and where that comes from:

* ``attention`` - the causal softmax attention unit O = f(A B) C that METP
  splits ("METP: memory-efficient tensor parallelism", FITEE
  10.1631/FITEE.2400602, abstract), with A B = Q K^T, f = row softmax of the
  scores times 1/sqrt(d) under the causal mask, C = V.  The pages do not print
  the formula; the oracle writes out the textbook definition.  It also returns
  the natural-log log-sum-exp of each row's scores, so that any (query shard,
  key block) result is an (o, lse) pair.
* ``merge_lse`` - the exact combination of such pairs by log-sum-exp
  rescaling.
* ``shards`` - contiguous and zigzag context partitions (the zigzag map of the
  TSP page, "Zyphra presenta el paralelismo de secuencia y tensor (TSP)",
  section "Lo que realmente significa plegar": shard r owns chunks r and
  2P-1-r of 2P equal chunks), ring and double-ring visiting orders
  ("Avances en la capacitacion de LLMs de secuencia larga", sections
  "Limitaciones de los Enfoques Existentes" and "Mejorando la Eficiencia de
  Comunicacion con la Atencion de Doble Anillo") and the sharded forward that
  merges per-block partials.
* ``attention_backward`` - gradients of the same unit, with P recomputed from
  the saved lse (textbook softmax-attention backward).
* ``attention_gqa`` / ``attention_backward_gqa`` - grouped-query attention:
  query heads in consecutive groups share one key/value head ("Avances en la
  capacitacion de LLMs de secuencia larga", section "Comprendiendo la
  Arquitectura de los LLMs"); the key/value gradients sum over the group.
* ``linear`` - causal linear attention and its sequence-parallel form
  (LASP: states passed point to point between contiguous shards; "Effiziente
  Parallelisierung linearer Aufmerksamkeitssequenzen fuer skalierbare
  Sprachmodelle").

Everything is float64 numpy; matmul is the only library primitive used.
"""
from .attention import (attention, attention_rows, attention_backward, attention_backward_block,
                        attention_backward_gqa, attention_gqa, backward_query_rows, backward_key_columns,
                        kv_head_of, merge_lse, softmax_matrix)
from .linear import (lasp_backward, lasp_forward, linear_attention, linear_attention_backward,
                     linear_attention_rows, linear_dkv_rows, linear_dq_rows, shard_bounds)
from .shards import (chunk_len, zigzag_order, contiguous_order, shard_order,
                     shard_positions, permute_rows, ring_visit_order,
                     double_ring_visit_order, sharded_attention,
                     visible_pairs)

__all__ = [
    "attention", "attention_rows", "attention_backward", "attention_backward_block",
    "attention_gqa", "attention_backward_gqa", "kv_head_of",
    "backward_query_rows",
    "backward_key_columns", "merge_lse", "softmax_matrix", "chunk_len",
    "zigzag_order", "contiguous_order", "shard_order", "shard_positions",
    "permute_rows", "ring_visit_order", "double_ring_visit_order",
    "sharded_attention", "visible_pairs", "linear_attention", "linear_attention_backward",
    "lasp_forward", "lasp_backward", "shard_bounds", "linear_attention_rows", "linear_dq_rows",
    "linear_dkv_rows",
]
