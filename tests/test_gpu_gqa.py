"""GPU parity of grouped-query attention (key/value heads shared by groups of
query heads; dK/dV summed over each group) through the sharded path, on the
tensor-core and the fp32-arithmetic kernels, every schedule and addressing,
against the fp64 oracle: small cases in full, the 32K grouped-query training
workload at full size on sampled rows."""
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


@pytest.mark.parametrize("dtype,algo,layout,P,G,H,Hkv,S,kw", [
    ("bf16", "auto", "zigzag", 4, 1, 4, 2, 1024, {}),
    ("bf16", "auto", "zigzag", 2, 1, 4, 1, 1024, {"addressing": "permuted"}),
    ("bf16", "auto", "zigzag", 2, 2, 8, 4, 1024, {"schedule": "direct"}),
    ("bf16", "auto", "zigzag", 2, 1, 6, 2, 768, {"schedule": "fused"}),
    ("bf16", "simt", "zigzag", 4, 1, 4, 2, 1024, {}),
    ("f32", "auto", "contiguous", 2, 1, 4, 2, 256, {}),
    ("f32", "auto", "zigzag", 2, 1, 4, 2, 256, {"schedule": "fused"}),
    ("bf16", "auto", "zigzag", 2, 1, 4, 1, 1024, {"D": 64}),                 # fp16 P/V/dO variant at D = 64
    ("bf16", "auto", "contiguous", 2, 1, 8, 2, 640, {"D": 64, "schedule": "fused"}),
])
def test_gqa_small_full_oracle(sca, dtype, algo, layout, P, G, H, Hkv, S, kw):
    kw = dict(kw)
    B, D = 1, kw.pop("D", 128 if dtype == "bf16" else 64)
    q, k, v, do = seeded_inputs.make_inputs(B, H, S, D, dtype, seed=300 + H + Hkv, with_do=True, kv_heads=Hkv)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    a = sca.capi.SCA_ALGO_SIMT if algo == "simt" else sca.capi.SCA_ALGO_AUTO
    plan = sca.ShardedCausalAttention(B, H, S, D, P, layout=layout, dtype=tdt, head_groups=G, backward=True,
                                      kv_heads=Hkv, algo=a, **{"schedule": "ring", **kw})
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = plan.forward(qd, kd, vd)
    dq, dk, dv = plan.backward(dod)
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    assert dk.shape == (B, Hkv, S, D) and dv.shape == (B, Hkv, S, D)
    ro, rl = oracle.attention_gqa(q, k, v, scale_for(D))
    rq, rk, rv = oracle.attention_backward_gqa(q, k, v, do, scale_for(D), o=ro, lse=rl)
    tol = tol_for(dtype)
    for name, got, ref in (("o", o, ro), ("lse", lse, rl), ("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_close(name, got, ref, tol)


@pytest.mark.parametrize("schedule", ["ring", "fused"])
def test_gqa_training_step_full_size_sampled(sca, schedule):
    w = WORKLOADS["gqa_s32k"]
    q, k, v, do = seeded_inputs.workload_inputs(w)
    Hkv, grp = w.kv_heads, w.H // w.kv_heads
    plan = sca.ShardedCausalAttention(w.B, w.H, w.S, w.D, w.P, layout=w.layout, schedule=schedule, backward=True,
                                      kv_heads=Hkv)
    o, lse = plan.forward(q.cuda(), k.cuda(), v.cuda())
    dq, dk, dv = plan.backward(do.cuda())
    torch.cuda.synchronize()
    assert plan.read_status() == 0
    scale = scale_for(w.D)
    rows = seeded_inputs.sample_rows(w.B, w.H, w.S, w.sample_rows, w.seed).numpy()
    tol = tol_for(w.dtype)
    o_c, lse_c, dq_c = o.cpu(), lse.cpu(), dq.cpu()
    # O, lse, dQ of the sampled query rows of every query head
    for h in range(w.H):
        hk = oracle.kv_head_of(h, w.H, Hkv)
        r = rows[0, h]
        ro, rl = oracle.attention_rows(q[:, h:h + 1], k[:, hk:hk + 1], v[:, hk:hk + 1], scale, rows[:, h:h + 1])
        assert_close(f"o h{h}", o_c[0, h, r], ro[0, 0], tol)
        assert_close(f"lse h{h}", lse_c[0, h, r], rl[0, 0], tol)
        rq = oracle.backward_query_rows(q[0, h], k[0, hk], v[0, hk], do[0, h], ro[0, 0], rl[0, 0], scale, r)
        assert_close(f"dq h{h}", dq_c[0, h, r], rq, tol)
    # dK, dV of the sampled key rows of key/value head 0: the sum over its
    # query heads, each needing its full forward
    cols = rows[0, 0]
    rk, rv = 0.0, 0.0
    for h in range(grp):
        fo, fl = oracle.attention(q[0, h], k[0, 0], v[0, 0], scale)
        gk, gv = oracle.backward_key_columns(q[0, h], k[0, 0], v[0, 0], do[0, h], fo, fl, scale, cols)
        rk, rv = rk + gk, rv + gv
    assert_close("dk kv-head 0", dk.cpu()[0, 0, cols], rk, tol)
    assert_close("dv kv-head 0", dv.cpu()[0, 0, cols], rv, tol)
