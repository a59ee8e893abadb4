"""GPU parity of the HBM-bound kernels: zigzag permute (bit exact), exact lse
merge and delta, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("dtype,D,P,S", [
    (torch.bfloat16, 128, 4, 8192), (torch.bfloat16, 128, 8, 1024), (torch.float32, 128, 4, 512),
    (torch.bfloat16, 64, 2, 12), (torch.float32, 1, 4, 8 * 33), (torch.bfloat16, 128, 1, 256),
    # chunks of 200 rows x 256 B = 51200 B: bulk pieces of 32 KB and a ragged 18 KB one
    (torch.bfloat16, 128, 3, 1200)])
def test_zigzag_permute_bit_exact(sca, dtype, D, P, S):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(2, 3, S, D, generator=g).to(dtype)
    xd = x.cuda()
    y = torch.empty_like(xd)
    row = D * x.element_size()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    sca.zigzag_permute(xd.data_ptr(), y.data_ptr(), 6, S, row, P, 0, status.data_ptr(), _stream())
    order = oracle.zigzag_order(S, P)
    ref = x[..., torch.as_tensor(order), :]
    assert torch.equal(y.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       ref.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    back = torch.empty_like(xd)
    sca.zigzag_permute(y.data_ptr(), back.data_ptr(), 6, S, row, P, 1, status.data_ptr(), _stream())
    assert torch.equal(back.cpu(), x)
    assert sca.sca_read_status(status.data_ptr(), _stream()) == 0


def test_zigzag_permute_full_size_bit_exact(sca):
    # the 32K training workload's tensors: [1, 16, 32768, 128] bf16, P = 4
    g = torch.Generator().manual_seed(9)
    x = torch.randn(1, 16, 32768, 128, generator=g).to(torch.bfloat16).cuda()
    y = torch.empty_like(x)
    sca.zigzag_permute(x.data_ptr(), y.data_ptr(), 16, 32768, 256, 4, 0, 0, _stream())
    order = torch.as_tensor(oracle.zigzag_order(32768, 4), device="cuda")
    assert torch.equal(y, x[..., order, :])


def _partials(n, rows, D, empty_frac=0.2, seed=0):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(n, rows, D, generator=g)
    lse = torch.randn(n, rows, generator=g) * 4
    drop = torch.rand(n, rows, generator=g) < empty_frac
    lse[drop] = -float("inf")
    o[drop] = 0
    lse[:, :3] = -float("inf")   # rows empty in every partial
    o[:, :3] = 0
    return o, lse


@pytest.mark.parametrize("n,D", [(1, 128), (2, 128), (3, 64), (8, 128), (5, 4), (16, 32)])
def test_merge_matches_oracle(sca, n, D):
    rows = 1000
    o, lse = _partials(n, rows, D, seed=n)
    od, ld = o.cuda(), lse.cuda()
    oo = torch.empty(rows, D, device="cuda")
    lo = torch.empty(rows, device="cuda")
    ob = torch.empty(rows, D, device="cuda", dtype=torch.bfloat16)
    sca.attn_merge_lse(od.data_ptr(), ld.data_ptr(), n, rows, D, rows * D, rows, oo.data_ptr(), lo.data_ptr(),
                       ob.data_ptr(), 0, 0, _stream())
    ro, rl = oracle.merge_lse(o.numpy(), lse.numpy())
    assert_close("o", oo, ro, (1e-5, 1e-6))
    assert_close("lse", lo, rl, (1e-5, 1e-6))
    assert torch.equal(ob.cpu(), oo.cpu().to(torch.bfloat16))


def test_merge_in_place_and_unpermuted(sca):
    B, H, S, D, P = 2, 3, 64, 128, 4
    rows = B * H * S
    o, lse = _partials(P, rows, D, seed=11)
    ro, rl = oracle.merge_lse(o.numpy(), lse.numpy())
    # in place into partial 0
    od, ld = o.clone().cuda(), lse.clone().cuda()
    sca.attn_merge_lse(od.data_ptr(), ld.data_ptr(), P, rows, D, rows * D, rows, od.data_ptr(), ld.data_ptr(), 0,
                       0, 0, _stream())
    assert_close("o in place", od[0], ro, (1e-5, 1e-6))
    # fused inverse zigzag permute: output row at its natural position
    od, ld = o.cuda(), lse.cuda()
    oo = torch.empty(rows, D, device="cuda")
    lo = torch.empty(rows, device="cuda")
    sca.attn_merge_lse(od.data_ptr(), ld.data_ptr(), P, rows, D, rows * D, rows, oo.data_ptr(), lo.data_ptr(), 0,
                       P, S, _stream())
    order = oracle.zigzag_order(S, P)
    nat_o = oracle.permute_rows(ro.reshape(B * H, S, D), order, inverse=True).reshape(rows, D)
    nat_l = oracle.permute_rows(rl.reshape(B * H, S, 1), order, inverse=True).reshape(rows)
    assert_close("o unpermuted", oo, nat_o, (1e-5, 1e-6))
    assert_close("lse unpermuted", lo, nat_l, (1e-5, 1e-6))


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_delta_matches_definition(sca, dtype, D):
    rows = 777
    g = torch.Generator().manual_seed(3)
    o = torch.randn(rows, D, generator=g)
    do = torch.randn(rows, D, generator=g).to(dtype)
    out = torch.empty(rows, device="cuda")
    od, dod = o.cuda(), do.cuda()     # keep both alive until the kernel has run
    sca.attn_bwd_delta(od.data_ptr(), dod.data_ptr(), 0 if dtype == torch.bfloat16 else 1,
                       out.data_ptr(), rows, D, _stream())
    torch.cuda.synchronize()
    ref = (o.double().numpy() * do.double().numpy()).sum(axis=1)
    assert_close("delta", out, ref, (1e-4, 1e-5))


def test_ring_stage_copies_bit_exact(sca):
    """One hand-off of mixed copies in one launch: strided gathers of a
    block's rows out of a [heads, S, D] tensor (narrow and wide rows), a
    flat copy larger than one unit of the kernel, and a one-row copy that is
    not a whole number of units; each lands exactly where torch puts it."""
    from sharded_causal_softmax_gb300 import capi
    g = torch.Generator().manual_seed(11)
    H, S, D = 3, 4096, 128
    x = torch.randn(H, S, D, generator=g).to(torch.bfloat16).cuda()
    row = D * 2
    a = torch.empty(H, 1000, D, dtype=torch.bfloat16, device="cuda")   # rows [700, 1700) of every head
    b = torch.empty(H, 32, D, dtype=torch.bfloat16, device="cuda")     # rows [8, 40): narrow
    flat = torch.empty(S * D, dtype=torch.bfloat16, device="cuda")     # head 1 whole (1 MB)
    odd = torch.empty(37 * D, dtype=torch.bfloat16, device="cuda")     # 37 rows of head 2 as one row
    cps = [capi.copy2d(x.data_ptr() + 700 * row, a.data_ptr(), H, 1000 * row, S * row, 1000 * row),
           capi.copy2d(x.data_ptr() + 8 * row, b.data_ptr(), H, 32 * row, S * row, 32 * row),
           capi.copy2d(x[1].data_ptr(), flat.data_ptr(), 1, S * row, S * row, S * row),
           capi.copy2d(x[2].data_ptr() + 100 * row, odd.data_ptr(), 1, 37 * row, 37 * row, 37 * row)]
    capi.ring_stage_copies(cps, _stream())
    torch.cuda.synchronize()
    assert torch.equal(a, x[:, 700:1700]) and torch.equal(b, x[:, 8:40])
    assert torch.equal(flat, x[1].reshape(-1)) and torch.equal(odd, x[2, 100:137].reshape(-1))
