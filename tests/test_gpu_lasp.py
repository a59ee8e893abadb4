"""GPU parity of causal linear attention over P contiguous shards passing
states point to point (LASP) against the fp64 oracle, on the fp32 CUDA-core
kernels (blocks of 64 rows) and the tensor-core kernels (blocks of 128 rows,
fp32 operands split into two bf16 parts): small cases in full (outputs,
gradients and the states each shard receives), the 32K training workload at
full size on sampled rows.  Both keep about fp32 accuracy, and without
normalisation the outputs grow like sqrt(t): the fp32 bounds (2e-4 max-abs,
2e-5 mean-abs) apply row by row, relative to the largest reference
magnitude of that row (at least 1), so an early row of magnitude O(1) is held
to the absolute fp32 bounds however large the late rows grow."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs
from seeded_inputs import WORKLOADS
from tests.gpu_util import scale_for

pytestmark = pytest.mark.gpu
REL = (2e-4, 2e-5)


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


def assert_close_rel(name, got, ref, rel=REL):
    """Per row (the last axis is the row's D values): the row's max-abs
    error <= rel[0] * m_t and its mean-abs error <= rel[1] * m_t, with
    m_t = max(1, max |ref_t|)."""
    ref = np.asarray(ref, dtype=np.float64)
    g = got.double().cpu().numpy() if hasattr(got, "cpu") else np.asarray(got, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    err = np.abs(g - ref).reshape(-1, ref.shape[-1])
    mag = np.maximum(1.0, np.abs(ref).reshape(-1, ref.shape[-1]).max(axis=1))
    rmax, rmean = err.max(axis=1) / mag, err.mean(axis=1) / mag
    worst = int(np.argmax(np.maximum(rmax / rel[0], rmean / rel[1])))
    assert rmax[worst] <= rel[0] and rmean[worst] <= rel[1], \
        (f"{name}: row {worst}: max-abs {err[worst].max():.3e}, mean-abs {err[worst].mean():.3e} against its "
         f"magnitude {mag[worst]:.3e} (relative {rmax[worst]:.2e} / {rmean[worst]:.2e}, bounds {rel})")


@pytest.mark.parametrize("dtype,B,H,S,D,P,block", [
    ("bf16", 1, 2, 1024, 128, 4, 64), ("bf16", 2, 2, 512, 64, 2, 64), ("f32", 1, 2, 256, 64, 1, 64),
    ("f32", 1, 3, 768, 128, 3, 64), ("bf16", 1, 1, 2048, 128, 8, 64),
    ("bf16", 1, 2, 1024, 128, 4, 128), ("bf16", 2, 3, 768, 128, 3, 128), ("bf16", 1, 1, 128, 128, 1, 128),
    ("bf16", 1, 1, 2048, 128, 8, 128), ("bf16", 1, 2, 1024, 128, 4, 256), ("bf16", 2, 2, 2048, 128, 2, 512),
    ("bf16", 1, 3, 1536, 128, 1, 1536), ("bf16", 3, 1, 2304, 128, 3, 384)])
def test_lasp_small_full_oracle(sca, dtype, B, H, S, D, P, block):
    q, k, v, do = seeded_inputs.make_inputs(B, H, S, D, dtype, seed=500 + P + D, with_do=True)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    plan = sca.ShardedLinearAttention(B, H, S, D, P, dtype=tdt, backward=True, block=block)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o = plan.forward(qd, kd, vd)
    dq, dk, dv = plan.backward(dod)
    assert plan.read_status() == 0
    scale = scale_for(D)
    assert_close_rel("o", o, oracle.linear_attention(q, k, v, scale))
    rq, rk, rv = oracle.linear_attention_backward(q, k, v, do, scale)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        assert_close_rel(name, got, ref)
    # the states the shards received, both directions, against the oracle's passes
    in_f, in_b = plan.in_f.cpu().numpy(), plan.in_b.cpu().numpy()
    for b in range(B):
        for h in range(H):
            _, recv_f = oracle.lasp_forward(q[b, h], k[b, h], v[b, h], scale, P, 64)
            _, recv_b = oracle.lasp_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, P, 64)
            for r in range(P):
                assert_close_rel(f"fwd state b{b} h{h} r{r}", in_f[b * H + h, r], recv_f[r])
                assert_close_rel(f"bwd state b{b} h{h} r{r}", in_b[b * H + h, r], recv_b[r])


@pytest.mark.parametrize("block", [64, 128, 256])
def test_lasp_repeat_is_deterministic(sca, block):
    B, H, S, D, P = 1, 2, 1024, 128, 4
    q, k, v, do = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=7, with_do=True))
    plan = sca.ShardedLinearAttention(B, H, S, D, P, backward=True, block=block)
    a = [plan.forward(q, k, v).clone()] + [t.clone() for t in plan.backward(do)]
    b = [plan.forward(q, k, v)] + list(plan.backward(do))
    assert all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("block", [None, 512, 128, 64])   # None: the plan's default (4096 rows here)
def test_lasp_training_step_full_size_sampled(sca, block):
    w = WORKLOADS["lasp_s32k"]
    q, k, v, do = seeded_inputs.workload_inputs(w)
    plan = sca.ShardedLinearAttention(w.B, w.H, w.S, w.D, w.P, backward=True, block=block)
    assert block is not None or plan.block == 4096
    o = plan.forward(q.cuda(), k.cuda(), v.cuda())
    dq, dk, dv = plan.backward(do.cuda())
    assert plan.read_status() == 0
    scale = scale_for(w.D)
    rows = seeded_inputs.sample_rows(w.B, w.H, w.S, w.sample_rows, w.seed).numpy()
    o_c, dq_c, dk_c, dv_c = o.cpu(), dq.cpu(), dk.cpu(), dv.cpu()
    for h in range(w.H):
        r = rows[0, h]
        assert_close_rel(f"o h{h}", o_c[0, h, r], oracle.linear_attention_rows(q[0, h], k[0, h], v[0, h], scale, r))
        assert_close_rel(f"dq h{h}", dq_c[0, h, r],
                         oracle.linear_dq_rows(q[0, h], k[0, h], v[0, h], do[0, h], scale, r))
        rk, rv = oracle.linear_dkv_rows(q[0, h], k[0, h], v[0, h], do[0, h], scale, r)
        assert_close_rel(f"dk h{h}", dk_c[0, h, r], rk)
        assert_close_rel(f"dv h{h}", dv_c[0, h, r], rv)
