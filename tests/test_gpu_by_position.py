"""GPU parity of position addressing (dims->q_by_pos / kv_by_pos /
dkv_by_pos): an item whose rows are zigzag chunks read and written at their
global positions in natural-order tensors must give, bit for bit, what the
same item gives on slabs gathered into shard-major order (the same
arithmetic on the same values), must match the oracle, and must leave every
row outside its segments untouched.  Also the staging gather
ring_stage_segments (bit exact)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import assert_close, scale_for, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sca():
    import sharded_causal_softmax_gb300 as m
    from sharded_causal_softmax_gb300 import build
    build.build()
    return m


def positions(seg):
    n, ln, st = seg
    return np.concatenate([np.arange(st[i], st[i] + ln) for i in range(n)])


def make(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def zig(S, P, r):
    """Segment map of zigzag shard r: chunks r and 2P-1-r of S/(2P) rows."""
    c = S // (2 * P)
    return (2, c, (r * c, (2 * P - 1 - r) * c))


def dims(capi, B, H, D, dtype, algo, q_rows, kv_rows, o_rows, dkv_rows=None, accumulate=0, by_pos=(0, 0, 0)):
    d = capi.sca_attn_dims()
    d.B, d.H, d.D = B, H, D
    d.dtype = capi.SCA_BF16 if dtype == torch.bfloat16 else capi.SCA_F32
    d.causal, d.algo, d.scale, d.accumulate = 1, algo, scale_for(D), accumulate
    d.q = capi.view(H * q_rows * D, q_rows * D, D)
    d.kv = capi.view(H * kv_rows * D, kv_rows * D, D)
    d.o = capi.view(H * o_rows * D, o_rows * D, D)
    r = dkv_rows if dkv_rows is not None else kv_rows
    d.dkv = capi.view(H * r * D, r * D, D)
    d.lse_b, d.lse_h = H * o_rows, o_rows
    d.q_by_pos, d.kv_by_pos, d.dkv_by_pos = by_pos
    return d


CASES = [  # (dtype, algo name, S, P, query shard r, key block j, D)
    ("bf16", "tc", 1024, 4, 1, 1, 128),
    ("bf16", "tc", 2048, 4, 3, 0, 128),
    ("bf16", "tc", 2048, 2, 0, 1, 64),
    ("bf16", "simt", 1024, 4, 2, 2, 128),
    ("f32", "simt", 1024, 2, 1, 0, 64),
]


def _algo(capi, name):
    return capi.SCA_ALGO_TC if name == "tc" else capi.SCA_ALGO_SIMT


@pytest.mark.parametrize("dtype,algo,S,P,r,j,D", CASES)
def test_forward_by_position_matches_slab_and_oracle(sca, dtype, algo, S, P, r, j, D):
    capi = sca.capi
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, H = 1, 2
    q, k, v = (make((B, H, S, D), tdt, 40 + i) for i in range(3))
    qs, ks = zig(S, P, r), zig(S, P, j)
    qp, kp = positions(qs), positions(ks)
    st = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # by position: natural tensors, outputs at the shard's global rows
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_nat = torch.full((B, H, S, D), float("nan"), device="cuda")
    l_nat = torch.full((B, H, S), float("nan"), device="cuda")
    it = capi.sca_fwd_item()
    it.q, it.k, it.v, it.o, it.lse = qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o_nat.data_ptr(), l_nat.data_ptr()
    it.q_pos, it.kv_pos = capi.segs(*qs), capi.segs(*ks)
    capi.attn_fwd_shard([it], dims(capi, B, H, D, tdt, _algo(capi, algo), S, S, S, by_pos=(1, 1, 0)),
                        status.data_ptr(), st)
    # the same item on gathered slabs
    qg, kg, vg = q[:, :, qp].contiguous().cuda(), k[:, :, kp].contiguous().cuda(), v[:, :, kp].contiguous().cuda()
    n = len(qp)
    o_sl = torch.empty((B, H, n, D), device="cuda")
    l_sl = torch.empty((B, H, n), device="cuda")
    it2 = capi.sca_fwd_item()
    it2.q, it2.k, it2.v, it2.o, it2.lse = (x.data_ptr() for x in (qg, kg, vg, o_sl, l_sl))
    it2.q_pos, it2.kv_pos = capi.segs(*qs), capi.segs(*ks)
    capi.attn_fwd_shard([it2], dims(capi, B, H, D, tdt, _algo(capi, algo), n, len(kp), n), status.data_ptr(), st)
    torch.cuda.synchronize()
    assert sca.sca_read_status(status.data_ptr(), st) == 0
    o_nat, l_nat, o_sl, l_sl = o_nat.cpu(), l_nat.cpu(), o_sl.cpu(), l_sl.cpu()
    assert torch.equal(o_nat[:, :, qp], o_sl) and torch.equal(l_nat[:, :, qp], l_sl)
    others = np.setdiff1d(np.arange(S), qp)
    assert torch.isnan(o_nat[:, :, others]).all() and torch.isnan(l_nat[:, :, others]).all()
    ro, rl = np.zeros((B, H, n, D)), np.zeros((B, H, n))
    for h in range(H):
        ro[0, h], rl[0, h] = oracle.attention(q[0, h, qp], k[0, h, kp], v[0, h, kp], scale_for(D),
                                              q_pos=qp, k_pos=kp)
    assert_close("o", o_sl, ro, tol_for(dtype))
    assert_close("lse", l_sl, rl, tol_for(dtype))


@pytest.mark.parametrize("accumulate", [0, 1])
@pytest.mark.parametrize("dtype,algo,S,P,r,j,D", CASES)
def test_backward_by_position_matches_slab_and_oracle(sca, dtype, algo, S, P, r, j, D, accumulate):
    capi = sca.capi
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    B, H = 1, 2
    q, k, v, do = (make((B, H, S, D), tdt, 60 + i) for i in range(4))
    qs, ks = zig(S, P, r), zig(S, P, j)
    qp, kp = positions(qs), positions(ks)
    n, m = len(qp), len(kp)
    # final lse of the full causal attention, delta arbitrary
    lse = torch.from_numpy(np.stack([oracle.attention(q[0, h], k[0, h], v[0, h], scale_for(D))[1]
                                     for h in range(H)])[None]).float()
    delta = make((B, H, S), torch.float32, 70) * 0.5
    prev = [make((B, H, S, D), torch.float32, 80 + i) for i in range(3)]   # dq, dk, dv before the call
    st = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(by_pos):
        if by_pos:
            ins = [x.cuda() for x in (q, k, v, do, lse, delta)]
            grads = [p.clone().cuda() for p in prev]
            d = dims(capi, B, H, D, tdt, _algo(capi, algo), S, S, S, S, accumulate, (1, 1, 1))
        else:
            ins = [q[:, :, qp], k[:, :, kp], v[:, :, kp], do[:, :, qp], lse[:, :, qp], delta[:, :, qp]]
            ins = [x.contiguous().cuda() for x in ins]
            grads = [prev[0][:, :, qp].contiguous().cuda(), prev[1][:, :, kp].contiguous().cuda(),
                     prev[2][:, :, kp].contiguous().cuda()]
            d = dims(capi, B, H, D, tdt, _algo(capi, algo), n, m, n, m, accumulate)
        it = capi.sca_bwd_item()
        it.q, it.k, it.v, it.dout, it.lse, it.delta = (x.data_ptr() for x in ins)
        it.dq, it.dk, it.dv = (g.data_ptr() for g in grads)
        it.q_pos, it.kv_pos = capi.segs(*qs), capi.segs(*ks)
        capi.attn_bwd_shard([it], d, status.data_ptr(), st)
        torch.cuda.synchronize()
        assert sca.sca_read_status(status.data_ptr(), st) == 0
        return [g.cpu() for g in grads]

    nat = run(True)
    sl = run(False)
    # dK, dV: one CTA per key tile, same arithmetic -> bitwise; dQ is summed
    # over key tiles in no fixed order on the tensor cores
    assert torch.equal(nat[1][:, :, kp], sl[1]) and torch.equal(nat[2][:, :, kp], sl[2])
    assert torch.allclose(nat[0][:, :, qp], sl[0], rtol=0, atol=1e-5)
    # rows outside the item keep their previous contents
    oq, ok_ = np.setdiff1d(np.arange(S), qp), np.setdiff1d(np.arange(S), kp)
    assert torch.equal(nat[0][:, :, oq], prev[0][:, :, oq])
    assert torch.equal(nat[1][:, :, ok_], prev[1][:, :, ok_]) and torch.equal(nat[2][:, :, ok_], prev[2][:, :, ok_])
    # against the oracle's block contributions
    tol = tol_for(dtype)
    for h in range(H):
        rq, rk, rv = oracle.attention_backward_block(q[0, h, qp], k[0, h, kp], v[0, h, kp], do[0, h, qp],
                                                     lse[0, h, qp], delta[0, h, qp], scale_for(D),
                                                     q_pos=qp, k_pos=kp)
        base = [p[0, h].double().numpy() for p in prev] if accumulate else [np.zeros((S, D))] * 3
        assert_close(f"dq h{h}", nat[0][0, h, qp], base[0][qp] + rq, tol)
        assert_close(f"dk h{h}", nat[1][0, h, kp], base[1][kp] + rk, tol)
        assert_close(f"dv h{h}", nat[2][0, h, kp], base[2][kp] + rv, tol)


@pytest.mark.parametrize("S,P,r", [(1024, 4, 0), (1024, 4, 3), (2048, 2, 1)])
def test_ring_stage_segments_gathers_shard(sca, S, P, r):
    capi = sca.capi
    B, H, D = 2, 3, 128
    x = make((B, H, S, D), torch.bfloat16, 90).cuda()
    seg = zig(S, P, r)
    n = 2 * seg[1]
    out = torch.zeros((B, H, n, D), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    for b in range(B):
        capi.ring_stage_segments(x[b].data_ptr(), out[b].data_ptr(), H, S, capi.segs(*seg), D * 2, st)
    torch.cuda.synchronize()
    assert torch.equal(out, x[:, :, positions(seg)])
