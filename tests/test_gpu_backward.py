"""GPU parity of the sharded backward (delta, ring of attn_bwd_shard steps
recomputing P from the saved lse, dK/dV summed across shards; rows by
position or through permuted copies; the fused one-launch schedule) against
the fp64 oracle: small cases in full, the 32K training workload at full
size on sampled query and key rows."""
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


@pytest.mark.parametrize("dtype,layout,P,G,schedule,S,addressing", [
    ("bf16", "zigzag", 2, 1, "ring", 1024, "auto"), ("bf16", "zigzag", 4, 1, "ring", 1024, "auto"),
    ("bf16", "zigzag", 4, 2, "direct", 1024, "auto"), ("bf16", "contiguous", 2, 1, "ring", 768, "auto"),
    ("f32", "contiguous", 2, 1, "ring", 256, "auto"), ("f32", "zigzag", 4, 1, "ring", 200 * 8 // 8, "auto"),
    ("bf16", "zigzag", 4, 1, "ring", 1024, "permuted"), ("bf16", "zigzag", 2, 2, "direct", 1024, "permuted"),
    ("bf16", "zigzag", 4, 1, "fused", 1024, "auto"), ("bf16", "zigzag", 2, 2, "fused", 896, "auto"),
    ("f32", "contiguous", 2, 1, "fused", 256, "auto"), ("f32", "zigzag", 4, 1, "ring", 1024, "position"),
    ("bf16", "zigzag", 4, 1, "double_ring", 1024, "auto"), ("bf16", "zigzag", 8, 2, "double_ring", 2048, "auto"),
    ("bf16", "zigzag", 4, 1, "double_ring", 1024, "permuted")])
def test_backward_small_full_oracle(sca, dtype, layout, P, G, schedule, S, addressing):
    B, H, D = 1, 2, 128 if dtype == "bf16" else 64
    if layout == "zigzag" and S % (2 * P):
        S = 2 * P * (S // (2 * P))
    q, k, v, do = seeded_inputs.make_inputs(B, H, S, D, dtype, seed=200 + P, with_do=True)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    visit = {"visit": "double_ring", "inner": 2} if schedule == "double_ring" else {}
    plan = sca.ShardedCausalAttention(B, H, S, D, P, layout=layout, dtype=tdt, head_groups=G,
                                      schedule="ring" if visit else schedule, backward=True, addressing=addressing,
                                      **visit)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = plan.forward(qd, kd, vd)
    dq, dk, dv = plan.backward(dod, qd, kd, vd)
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    ro, rl = oracle.attention(q, k, v, scale_for(D))
    rq, rk, rv = oracle.attention_backward(q, k, v, do, scale_for(D), o=ro, lse=rl)
    tol = tol_for(dtype)
    for name, got, ref in (("o", o, ro), ("lse", lse, rl), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_close(name, got, ref, tol)


@pytest.mark.parametrize("schedule", ["ring", "fused"])
def test_backward_repeat_overwrites(sca, schedule):
    # step 0 overwrites the gradient buffers: a second call gives the same result
    B, H, S, D, P = 1, 2, 512, 128, 2
    q, k, v, do = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=9, with_do=True))
    plan = sca.ShardedCausalAttention(B, H, S, D, P, backward=True, schedule=schedule)
    plan.forward(q, k, v)
    a = [t.clone() for t in plan.backward(do)]
    plan.forward(q, k, v)
    b = plan.backward(do)
    # dK, dV: each key tile is owned by one CTA, summed over ring steps in a
    # fixed order -> bitwise equal.  dQ may gather key tiles through fp32
    # atomics, whose order varies -> equal up to rounding.
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    assert torch.allclose(a[0], b[0], rtol=0, atol=1e-5)


@pytest.mark.parametrize("schedule", ["ring", "fused", "double_ring"])
def test_training_step_full_size_sampled(sca, schedule):
    w = WORKLOADS["train_s32k"]
    q, k, v, do = seeded_inputs.workload_inputs(w)
    visit = {"visit": "double_ring", "inner": 2} if schedule == "double_ring" else {}
    plan = sca.ShardedCausalAttention(w.B, w.H, w.S, w.D, w.P, layout=w.layout,
                                      schedule="ring" if visit else schedule, backward=True, **visit)
    o, lse = plan.forward(q.cuda(), k.cuda(), v.cuda())
    dq, dk, dv = plan.backward(do.cuda())
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    scale = scale_for(w.D)
    rows = seeded_inputs.sample_rows(w.B, w.H, w.S, w.sample_rows, w.seed).numpy()
    ro, rl = oracle.attention_rows(q, k, v, scale, rows)
    tol = tol_for(w.dtype)
    o_c, lse_c, dq_c = o.cpu(), lse.cpu(), dq.cpu()
    got_o = torch.stack([o_c[0, h, rows[0, h]] for h in range(w.H)])[None]
    got_l = torch.stack([lse_c[0, h, rows[0, h]] for h in range(w.H)])[None]
    assert_close("o", got_o, ro, tol)
    assert_close("lse", got_l, rl, tol)
    # dQ of the sampled query rows, every head
    ref_dq = np.stack([oracle.backward_query_rows(q[0, h], k[0, h], v[0, h], do[0, h], ro[0, h], rl[0, h], scale,
                                                  rows[0, h]) for h in range(w.H)])
    got_dq = torch.stack([dq_c[0, h, rows[0, h]] for h in range(w.H)])
    assert_close("dq", got_dq, ref_dq, tol)
    # dK, dV of the sampled key rows on two heads (each needs that head's full forward)
    dk_c, dv_c = dk.cpu(), dv.cpu()
    for h in (0, w.H - 1):
        fo, fl = oracle.attention(q[0, h], k[0, h], v[0, h], scale)
        rk, rv = oracle.backward_key_columns(q[0, h], k[0, h], v[0, h], do[0, h], fo, fl, scale, rows[0, h])
        assert_close(f"dk head {h}", dk_c[0, h, rows[0, h]], rk, tol)
        assert_close(f"dv head {h}", dv_c[0, h, rows[0, h]], rv, tol)
