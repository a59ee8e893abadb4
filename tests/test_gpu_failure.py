"""The failure path of the tensor-core kernels, on the GPU without a fault: a
bounded mbarrier wait that nothing completes gives up after the library's
wait limit and records SCA_ERR_TIMEOUT in the caller's status word; the
context stays usable and the next attention launch reports success."""
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


def test_bounded_wait_reports_timeout_and_context_survives(sca):
    capi = sca.capi
    st = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    capi.sca_selftest_wait_timeout(status.data_ptr(), st)
    assert capi.sca_read_status(status.data_ptr(), st) == capi.SCA_ERR_TIMEOUT
    # the context still runs kernels, and a fresh status word reads OK
    B, H, S, D, P = 1, 2, 512, 128, 2
    q, k, v = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, "bf16", seed=3))
    plan = sca.ShardedCausalAttention(B, H, S, D, P, schedule="ring")
    o, lse = plan.forward(q, k, v)
    assert plan.read_status() == 0
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
