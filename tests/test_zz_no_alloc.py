"""lasp_fwd_noalloc (the whole linear-attention forward with its states in the
library's fixed device array) against the four-call forward with caller
buffers, on two calls in a row with different inputs: the outputs must be
identical bit for bit (same kernels, same order).  The file sorts last so that
it also runs after every other test in one process."""
import pytest
import torch

import seeded_inputs

CASES = [
    # B, H, S, D, P, dtype
    (1, 4, 2048, 128, 4, "bf16"),
    (2, 2, 1024, 64, 2, "f32"),
]


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


def test_noalloc_rejects_oversize_before_any_device_work():
    from sharded_causal_softmax_gb300 import build, capi
    build.build()
    lib = capi.lib()
    A = 1 << 20   # never dereferenced: every check below fails before a launch
    # 16 heads of 32K rows at D = 128 need 134M floats of block states
    assert lib.lasp_fwd_noalloc(A, A, A, capi.SCA_BF16, A, 16, 32768, 128, 4, 0.1, None) == \
        capi.SCA_ERR_UNSUPPORTED
    assert "fixed workspace" in capi.last_error()
    assert lib.lasp_fwd_noalloc(None, A, A, capi.SCA_BF16, A, 1, 1024, 128, 4, 0.1, None) == capi.SCA_ERR_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,S,D,P,dtype", CASES)
def test_noalloc_matches_buffered_forward_twice(sca, B, H, S, D, P, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    plan = sca.ShardedLinearAttention(B, H, S, D, P, dtype=tdt, block=sca.capi.SCA_LASP_BLOCK_F32)
    st = torch.cuda.current_stream().cuda_stream
    for seed in (41, 42):
        q, k, v = (x.cuda() for x in seeded_inputs.make_inputs(B, H, S, D, dtype, seed=seed))
        ref = plan.forward(q, k, v).clone()
        o = torch.full((B, H, S, D), float("nan"), dtype=torch.float32, device="cuda")
        sca.capi.lasp_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), sca.lasp._DT[tdt], o.data_ptr(),
                                  B * H, S, D, P, plan.scale, st)
        torch.cuda.synchronize()
        assert torch.equal(o, ref), f"seed {seed}: max diff {(o - ref).abs().max().item()}"
