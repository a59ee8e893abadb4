"""cast_bf16_to_f16 against torch's own bf16 -> fp16 conversion (bit for
bit, special values included), and the backward with fp16 queries (and,
grouped, fp16 dO) staged once per call against the same backward converting
them tile by tile inside the kernel: the fp16 operands are the same values,
so dK and dV agree bit for bit; dQ, summed by reduce-adds in no fixed order,
agrees to rounding.  Parity of the staged path against the fp64 oracle is
covered by every plan-level backward test, where staging is the default."""
import pytest
import torch

import seeded_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


@pytest.mark.parametrize("n", [8, 8 * 37, 8 * 4096 + 8 * 3])
def test_cast_matches_torch_bit_for_bit(sca, n):
    g = torch.Generator().manual_seed(n)
    x = (torch.randn(n, generator=g) * torch.exp2(torch.randint(-30, 20, (n,), generator=g).float()))
    x = x.to(torch.bfloat16)
    special = torch.tensor([0.0, -0.0, 1e-8, -3e-7, 6.1e-5, 65504.0, 65520.0, 7e4, -1e6, float("inf"),
                            -float("inf"), 1.0], dtype=torch.bfloat16)
    x[: min(n, special.numel())] = special[: min(n, special.numel())]
    src = x.cuda()
    dst = torch.full((n,), float("nan"), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    sca.capi.cast_bf16_to_f16(src.data_ptr(), dst.data_ptr(), n, status.data_ptr(), stream)
    torch.cuda.synchronize()
    want = x.to(torch.float16)
    assert torch.equal(dst.cpu().view(torch.int16), want.view(torch.int16))
    # the specials include finite values beyond the fp16 range (65520 rounds
    # to bf16 65536; 7e4, -1e6): the conversion reports them
    beyond = (x.float().abs() >= 65536) & torch.isfinite(x.float())
    assert bool(beyond.any())
    assert sca.capi.sca_read_status(status.data_ptr(), stream) == sca.capi.SCA_ERR_RANGE


def test_cast_in_range_reports_nothing(sca):
    """The largest bf16 below 65536 (65280), infinities and NaN convert
    without a range report; the status word stays 0."""
    x = torch.tensor([65280.0, -65280.0, float("inf"), -float("inf"), float("nan"), 1e-9, 0.0, 3.5] * 4,
                     dtype=torch.bfloat16)
    src = x.cuda()
    dst = torch.empty(x.numel(), dtype=torch.float16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    sca.capi.cast_bf16_to_f16(src.data_ptr(), dst.data_ptr(), x.numel(), status.data_ptr(), stream)
    assert sca.capi.sca_read_status(status.data_ptr(), stream) == sca.capi.SCA_OK
    # a NaN stays NaN (its payload is the hardware's); everything else bit for bit
    got, want = dst.cpu(), x.to(torch.float16)
    nan = torch.isnan(want)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan].view(torch.int16), want[~nan].view(torch.int16))


@pytest.mark.parametrize("schedule,kv_heads,H", [("ring", None, 2), ("fused", None, 2), ("ring", 2, 4),
                                                 ("fused", 1, 4)])
def test_staged_backward_matches_in_kernel_conversion(sca, schedule, kv_heads, H):
    B, S, D, P = 1, 1024, 128, 4
    q, k, v, do = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=71, with_do=True,
                                                              kv_heads=kv_heads))
    grads = []
    for staging in (True, False):
        plan = sca.ShardedCausalAttention(B, H, S, D, P, schedule=schedule, backward=True, kv_heads=kv_heads,
                                          f16_staging=staging)
        assert bool(plan.f16_in) == staging
        plan.forward(q, k, v)
        grads.append([t.clone() for t in plan.backward(do)])
        assert plan.read_status() == 0
    (dq1, dk1, dv1), (dq0, dk0, dv0) = grads
    assert torch.equal(dk1, dk0) and torch.equal(dv1, dv0)
    torch.testing.assert_close(dq1, dq0, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("where,staging", [("q", True), ("q", False), ("k", True), ("v_grouped", True)])
def test_backward_reports_values_beyond_fp16(sca, where, staging):
    """A finite bf16 input that fp16 cannot hold (7e4 rounds to bf16 70144)
    would turn into +-inf inside the fp16 products of the backward: the call
    records SCA_ERR_RANGE in its status word instead of passing for a good
    one.  Q goes through the once-per-call cast (staging) or the kernel's own
    conversion; K always through the kernel's; V (grouped heads, where dP and
    dV are fp16 products) through the kernel's.  Nothing faults, and a clean
    call on the same plan afterwards reports nothing."""
    B, S, D, P = 1, 512, 128, 2
    kvh = 1 if where == "v_grouped" else None
    H = 2
    q, k, v, do = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=73, with_do=True,
                                                              kv_heads=kvh))
    bad = {"q": q, "k": k, "v_grouped": v}[where].clone()
    bad[0, 0, 300, 5] = 7e4
    ins = {"q": q, "k": k, "v": v}
    ins["v" if where == "v_grouped" else where] = bad
    plan = sca.ShardedCausalAttention(B, H, S, D, P, backward=True, kv_heads=kvh, f16_staging=staging,
                                      schedule="ring")
    plan.forward(ins["q"], ins["k"], ins["v"])
    plan.backward(do)
    assert plan.read_status() == sca.capi.SCA_ERR_RANGE
    plan.status.zero_()
    plan.forward(q, k, v)
    plan.backward(do)
    assert plan.read_status() == sca.capi.SCA_OK
