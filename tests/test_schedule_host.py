"""Host-side argument checks of the sharded schedule (they run before any
device memory is touched, so no GPU is needed)."""
import pytest

import oracle
from sharded_causal_softmax_gb300.sharded import (ShardedCausalAttention, copy_runs, double_ring_block, hop_senders,
                                                  ring_block, shard_segs)


@pytest.mark.parametrize("kw,msg", [
    (dict(kv_heads=3), "kv_heads"),                          # 3 does not divide 8
    (dict(kv_heads=2, head_groups=4), "head_groups"),        # 4 groups cannot split 2 key/value heads
    (dict(schedule="spiral"), "schedule"),
    (dict(addressing="sideways"), "addressing"),
    (dict(addressing="position", S=768), "128"),             # zigzag chunks of 96 rows
    (dict(layout="diagonal"), "layout"),
    (dict(visit="double_ring"), "inner"),                    # no inner ring size
    (dict(visit="double_ring", inner=3), "inner"),           # 3 does not divide P = 4
    (dict(visit="spiral"), "visit"),
])
def test_schedule_rejects_bad_arguments(kw, msg):
    args = dict(B=1, H=8, S=1024, D=128, P=4)
    args.update({k: v for k, v in kw.items() if k in args})
    extra = {k: v for k, v in kw.items() if k not in args}
    with pytest.raises(ValueError, match=msg):
        ShardedCausalAttention(args["B"], args["H"], args["S"], args["D"], args["P"], **extra)


def test_ring_order_and_zigzag_segments():
    P = 4
    # every shard visits every block exactly once, starting with its own
    for r in range(P):
        assert sorted(ring_block(r, t, P) for t in range(P)) == list(range(P))
        assert ring_block(r, 0, P) == r
    s = shard_segs(1024, P, "zigzag", 1)
    assert (s.n, s.len, s.start[0], s.start[1]) == (2, 128, 128, 768)
    s = shard_segs(1024, P, "contiguous", 3)
    assert (s.n, s.len, s.start[0]) == (1, 256, 768)


def test_linear_attention_default_block():
    import torch
    from sharded_causal_softmax_gb300.lasp import default_block
    bf = torch.bfloat16
    assert default_block(1, 16, 32768, 128, 4, bf) == 4096      # 128 blocks of 4096 rows
    assert default_block(1, 4, 32768, 128, 4, bf) == 1024       # at least 128 blocks
    assert default_block(1, 2, 1024, 128, 4, bf) == 128         # too small for 128 blocks: the smallest
    assert default_block(1, 16, 32768, 128, 4, torch.float32) == 64   # fp32 inputs: CUDA cores
    assert default_block(1, 16, 32768, 64, 4, bf) == 64         # D = 64: CUDA cores
    for args in [(1, 16, 32768, 128, 4), (2, 3, 2304, 128, 3), (1, 1, 128, 128, 1)]:
        b = default_block(*args, bf)
        assert b % 128 == 0 and args[2] % (b * args[4]) == 0


def test_fp16_staging_flags():
    import torch
    from sharded_causal_softmax_gb300 import capi
    from sharded_causal_softmax_gb300.sharded import f16_input_flags
    auto, simt, tc = capi.SCA_ALGO_AUTO, capi.SCA_ALGO_SIMT, capi.SCA_ALGO_TC
    assert f16_input_flags(True, torch.bfloat16, auto, 16, 16) == capi.SCA_F16_Q
    assert f16_input_flags(True, torch.bfloat16, tc, 32, 8) == capi.SCA_F16_Q | capi.SCA_F16_DOUT
    assert f16_input_flags(True, torch.bfloat16, simt, 32, 8) == 0     # CUDA-core kernels read bf16
    assert f16_input_flags(True, torch.float32, auto, 16, 16) == 0     # fp32 inputs: no fp16 products
    assert f16_input_flags(False, torch.bfloat16, auto, 32, 8) == 0    # staging switched off


@pytest.mark.parametrize("n,per", [(0, 32), (1, 32), (16, 32), (32, 32), (33, 32), (64, 32), (100, 32), (7, 3)])
def test_launch_groups_cover_every_item_once(n, per):
    from sharded_causal_softmax_gb300.sharded import launch_groups
    groups = launch_groups(n, per)
    covered = [i for lo, hi in groups for i in range(lo, hi)]
    assert covered == list(range(n))
    assert all(0 < hi - lo <= per for lo, hi in groups)
    assert len(groups) == -(-n // per)


@pytest.mark.parametrize("P,inner", [(4, 2), (8, 4), (8, 2), (6, 3), (4, 4), (4, 1), (16, 4)])
def test_double_ring_schedule_follows_the_oracle_order(P, inner):
    for r in range(P):
        assert [double_ring_block(r, t, P, inner) for t in range(P)] == oracle.double_ring_visit_order(P, r, inner)


def test_ring_hand_off_is_two_copies():
    """Every ring hand-off is a rotation by one shard: two contiguous copies
    (shards 1..P-1 from 0..P-2, shard 0 from P-1)."""
    P = 8
    for t in range(1, P):
        runs = copy_runs(hop_senders(lambda r, s: ring_block(r, s, P), t, P))
        assert sorted(runs) == [(0, P - 1, 1), (1, 0, P - 1)]


@pytest.mark.parametrize("P,inner", [(8, 4), (8, 2), (6, 3)])
def test_double_ring_hand_offs(P, inner):
    """Inner hops rotate inside each group (two copies per group); outer hops
    take every block from a shard of the previous group.  Every run of a
    hand-off copies real staged slabs: each destination receives exactly the
    block it visits next."""
    blk = lambda r, t: double_ring_block(r, t, P, inner)
    for t in range(1, P):
        senders = hop_senders(blk, t, P)
        assert sorted(senders) == list(range(P))
        for r, s in enumerate(senders):
            assert blk(s, t - 1) == blk(r, t)
            if t % inner:   # inner hop
                assert s // inner == r // inner
            else:           # outer hop
                assert s // inner == (r // inner - 1) % (P // inner)
        covered = []
        for r0, s0, n in copy_runs(senders):
            covered += [(r0 + k, s0 + k) for k in range(n)]
        assert sorted(covered) == sorted(enumerate(senders))
        if t % inner:
            assert len(copy_runs(senders)) == 2 * (P // inner) - (P // inner if inner == 1 else 0)


def test_auto_schedule_fuses_short_shards_only():
    # "auto" fuses when a shard holds at most AUTO_FUSED_MAX_ROWS rows (ring
    # steps of at most 32 key tiles per CTA) and keeps the ring above, or
    # whenever the double ring is asked for; explicit schedules pass through
    from sharded_causal_softmax_gb300.sharded import AUTO_FUSED_MAX_ROWS, resolve_schedule
    assert AUTO_FUSED_MAX_ROWS == 4096
    assert resolve_schedule("auto", 8192, 4) == "fused"          # 2048 rows per shard
    assert resolve_schedule("auto", 16384, 4) == "fused"         # 4096
    assert resolve_schedule("auto", 32768, 4) == "ring"          # 8192
    assert resolve_schedule("auto", 131072, 8) == "ring"
    assert resolve_schedule("auto", 8192, 4, visit="double_ring") == "ring"
    assert resolve_schedule("auto", 1 << 20, 1) == "fused"       # one shard: nothing to pass around
    for s in ("ring", "direct", "fused"):
        assert resolve_schedule(s, 8192, 4) == s
