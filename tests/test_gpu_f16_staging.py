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
    sca.capi.cast_bf16_to_f16(src.data_ptr(), dst.data_ptr(), n, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = x.to(torch.float16)
    assert torch.equal(dst.cpu().view(torch.int16), want.view(torch.int16))


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
