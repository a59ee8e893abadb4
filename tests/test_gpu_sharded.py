"""End-to-end sharded forward on the GPU (ring of per-block partials with
double-buffered staging and the lse merge, rows addressed by position or
through permuted copies; the fused one-launch schedule) against the fp64
oracle, on every forward workload at full size (sampled rows where the
oracle would take too long)."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs
from seeded_inputs import WORKLOADS
from tests.gpu_util import assert_close, scale_for, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


def _plan(sca, w, **kw):
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    args = dict(layout=w.layout, dtype=dtype, head_groups=w.head_groups, schedule=w.schedule)
    args.update(kw)
    return sca.ShardedCausalAttention(w.B, w.H, w.S, w.D, w.P, **args)


def _run(sca, w, q, k, v, **kw):
    plan = _plan(sca, w, **kw)
    o, lse = plan.forward(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    return plan, o, lse


@pytest.mark.parametrize("name,kw", [("tiny_f32", {}), ("fwd_s8k", {}), ("fwd_s8k", {"addressing": "permuted"}),
                                     ("fwd_s8k", {"schedule": "fused"}), ("tiny_f32", {"schedule": "fused"})])
def test_forward_full_oracle(sca, name, kw):
    w = WORKLOADS[name]
    q, k, v = seeded_inputs.workload_inputs(w)[:3]
    _, o, lse = _run(sca, w, q, k, v, **kw)
    ro, rl = oracle.attention(q, k, v, scale_for(w.D))
    assert_close("o", o, ro, tol_for(w.dtype))
    assert_close("lse", lse, rl, tol_for(w.dtype))


@pytest.mark.parametrize("name,kw", [("ring_s128k", {}), ("2d_s32k", {}), ("ring_s128k", {"schedule": "fused"}),
                                     ("ring_s128k", {"visit": "double_ring", "inner": 4})])
def test_forward_sampled_rows_full_size(sca, name, kw):
    w = WORKLOADS[name]
    q, k, v = seeded_inputs.workload_inputs(w)[:3]
    _, o, lse = _run(sca, w, q, k, v, **kw)
    rows = seeded_inputs.sample_rows(w.B, w.H, w.S, w.sample_rows, w.seed).numpy()
    ro, rl = oracle.attention_rows(q, k, v, scale_for(w.D), rows)
    idx = torch.as_tensor(rows, device=o.device)
    go = torch.gather(o, 2, idx[..., None].expand(-1, -1, -1, w.D))
    gl = torch.gather(lse, 2, idx)
    assert_close("o", go, ro, tol_for(w.dtype))
    assert_close("lse", gl, rl, tol_for(w.dtype))
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("layout,P,G,kw", [
    ("zigzag", 4, 1, {}), ("zigzag", 8, 1, {}), ("contiguous", 4, 1, {}), ("zigzag", 2, 4, {}),
    ("contiguous", 1, 1, {}), ("zigzag", 1, 2, {}), ("zigzag", 4, 1, {"addressing": "permuted"}),
    ("zigzag", 2, 4, {"addressing": "permuted", "schedule": "direct"}), ("zigzag", 4, 1, {"schedule": "fused"}),
    ("zigzag", 2, 4, {"schedule": "fused"}), ("contiguous", 4, 1, {"schedule": "direct"}),
    # 4 head groups x 4 shards x 4 blocks = 64 partials: two launches of 32
    ("zigzag", 4, 4, {"schedule": "direct"}),
    # double ring: 2 groups of 2 shards / 4 of 2; staged hand-offs inside and between groups
    ("zigzag", 4, 1, {"visit": "double_ring", "inner": 2}), ("zigzag", 8, 1, {"visit": "double_ring", "inner": 2}),
    ("zigzag", 4, 2, {"visit": "double_ring", "inner": 2, "addressing": "permuted"}),
    ("contiguous", 4, 1, {"visit": "double_ring", "inner": 2}),
    # the direct schedule, one launch per step (the ring's launches without its staging copies)
    ("zigzag", 4, 1, {"schedule": "direct", "group_steps": False})])
def test_forward_small_full_oracle(sca, layout, P, G, kw):
    B, H, S, D = 2, 4, 1024, 128
    q, k, v = seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=100 + P + G)
    plan = sca.ShardedCausalAttention(B, H, S, D, P, layout=layout, head_groups=G, **{"schedule": "ring", **kw})
    o, lse = plan.forward(q.cuda(), k.cuda(), v.cuda())
    ro, rl = oracle.attention(q, k, v, scale_for(D))
    assert_close("o", o, ro, tol_for("bf16"))
    assert_close("lse", lse, rl, tol_for("bf16"))
    # oracle-side sharded computation gives the same answer (merge invariance)
    so, sl = oracle.sharded_attention(q, k, v, scale_for(D), P, layout)
    np.testing.assert_allclose(so, ro, atol=1e-10)


def test_ring_staging_equals_direct_reads(sca):
    # staged or home blocks, positions or permuted copies: the same partials
    # and the same merge, so bit-identical results; the fused schedule sums
    # in another order, so equal up to rounding
    w = WORKLOADS["ring_s128k"]
    S, H = 16384, 4
    q, k, v = seeded_inputs.make_inputs(w.B, H, S, w.D, "bf16", seed=w.seed)
    outs = []
    for kw in ({"schedule": "ring"}, {"schedule": "direct"}, {"schedule": "ring", "addressing": "permuted"},
               {"schedule": "direct", "addressing": "permuted"}, {"schedule": "direct", "group_steps": False},
               {"schedule": "fused"}):
        plan = sca.ShardedCausalAttention(w.B, H, S, w.D, w.P, **kw)
        o, lse = plan.forward(q.cuda(), k.cuda(), v.cuda())
        outs.append((o.clone(), lse.clone()))
    for o, lse in outs[1:5]:
        assert torch.equal(outs[0][0], o) and torch.equal(outs[0][1], lse)
    assert torch.allclose(outs[0][0], outs[5][0], rtol=0, atol=2e-3)
    assert torch.allclose(outs[0][1], outs[5][1], rtol=0, atol=1e-4)


def test_double_ring_partials_are_the_ring_partials(sca):
    """The double ring visits the same (shard, block) pairs in another order:
    each pair's partial is computed by the same kernel from the same rows, so
    the partial stored for block j of shard r is bit for bit the ring's;
    only the merge order (step slots) differs, so O and lse agree up to fp32
    rounding.  Staged copies carry the blocks unchanged through inner and
    outer hops."""
    w = WORKLOADS["ring_s128k"]
    S, H, P, inner = 16384, 2, w.P, 4
    q, k, v = (x.cuda() for x in seeded_inputs.make_inputs(w.B, H, S, w.D, "bf16", seed=w.seed + 1))
    ring = sca.ShardedCausalAttention(w.B, H, S, w.D, P, schedule="ring")
    dbl = sca.ShardedCausalAttention(w.B, H, S, w.D, P, visit="double_ring", inner=inner)
    o1, l1 = ring.forward(q, k, v)
    o2, l2 = dbl.forward(q, k, v)
    assert ring.read_status() == 0 and dbl.read_status() == 0
    segs = [oracle.shard_positions(S, P, "zigzag")[r] for r in range(P)]
    for r in range(P):
        rows = torch.as_tensor(segs[r], device="cuda")
        for t in range(P):
            j = dbl.block(r, t)
            t_ring = (r - j) % P
            assert torch.equal(dbl.o_parts[t][:, :, rows], ring.o_parts[t_ring][:, :, rows])
            assert torch.equal(dbl.lse_parts[t][:, :, rows], ring.lse_parts[t_ring][:, :, rows])
    assert torch.allclose(o1, o2, rtol=0, atol=1e-5) and torch.allclose(l1, l2, rtol=0, atol=1e-5)


def test_repeated_calls_are_deterministic(sca):
    B, H, S, D, P = 1, 2, 2048, 128, 4
    q, k, v = seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=3)
    plan = sca.ShardedCausalAttention(B, H, S, D, P, head_groups=2, schedule="ring")
    a = [t.clone() for t in plan.forward(q.cuda(), k.cuda(), v.cuda())]
    b = plan.forward(q.cuda(), k.cuda(), v.cuda())
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("schedule", ["ring", "fused"])
def test_bf16_output_copy(sca, schedule):
    B, H, S, D, P = 1, 2, 512, 128, 2
    q, k, v = seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=4)
    plan = sca.ShardedCausalAttention(B, H, S, D, P, bf16_out=True, schedule=schedule)
    o, _ = plan.forward(q.cuda(), k.cuda(), v.cuda())
    assert torch.equal(plan.o_bf16, o.to(torch.bfloat16))
