"""GPU parity of attn_bwd_shard on single (query shard, key block) items
against the oracle's per-block gradient contributions, on the tensor-core
kernel (bf16) and the fp32-arithmetic kernels (bf16, fp32): zigzag
segments, ragged tails, tiles straddling segments, blocks nobody sees,
non-causal rows, D = 64, several items per launch, accumulate vs
overwrite."""
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
    return np.concatenate([np.arange(st[i], st[i] + ln) for i in range(n)]) if ln else np.zeros(0, np.int64)


def make(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


class Spec:
    def __init__(self, B, H, D, Sq, Skv, qs, ks, dtype, seed, causal=True):
        self.q, self.do = make((B, H, Sq, D), dtype, seed), make((B, H, Sq, D), dtype, seed + 1)
        self.k, self.v = make((B, H, Skv, D), dtype, seed + 2), make((B, H, Skv, D), dtype, seed + 3)
        self.qs, self.ks = qs, ks
        # lse of the item itself (rows that see nothing keep -inf), delta arbitrary
        _, lse = oracle.attention(self.q, self.k, self.v, scale_for(D), causal=causal,
                                  q_pos=positions(qs), k_pos=positions(ks))
        self.lse = torch.from_numpy(lse).float()
        self.delta = make((B, H, Sq), torch.float32, seed + 4) * 0.5
        self.prev = [make((B, H, n, D), torch.float32, seed + 5 + i) for i, n in enumerate((Sq, Skv, Skv))]


def run(sca, specs, dtype, algo, D, B, H, causal=True, accumulate=0):
    capi = sca.capi
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    items, keep, outs = [], [], []
    for s in specs:
        dev = {n: getattr(s, n).cuda() for n in ("q", "k", "v", "do", "lse", "delta")}
        grads = [p.clone().cuda() for p in s.prev]
        it = capi.sca_bwd_item()
        it.q, it.k, it.v, it.dout = (dev[n].data_ptr() for n in ("q", "k", "v", "do"))
        it.lse, it.delta = dev["lse"].data_ptr(), dev["delta"].data_ptr()
        it.dq, it.dk, it.dv = (g.data_ptr() for g in grads)
        it.q_pos = capi.segs(s.qs[0], s.qs[1], s.qs[2])
        it.kv_pos = capi.segs(s.ks[0], s.ks[1], s.ks[2])
        items.append(it)
        keep.append(dev)
        outs.append(grads)
    d = capi.sca_attn_dims()
    d.B, d.H, d.D = B, H, D
    d.dtype = capi.SCA_BF16 if dtype == torch.bfloat16 else capi.SCA_F32
    d.causal, d.algo, d.scale, d.accumulate = 1 if causal else 0, algo, scale_for(D), accumulate
    q0, k0, g0, gk = keep[0]["q"], keep[0]["k"], outs[0][0], outs[0][1]
    d.q = capi.view(*q0.stride()[:3])
    d.kv = capi.view(*k0.stride()[:3])
    d.o = capi.view(*g0.stride()[:3])
    d.dkv = capi.view(*gk.stride()[:3])
    d.lse_b, d.lse_h = keep[0]["lse"].stride(0), keep[0]["lse"].stride(1)
    capi.attn_bwd_shard(items, d, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sca.sca_read_status(status.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    return [[g.cpu() for g in grads] for grads in outs]


def check(spec, got, dtype, D, causal=True, accumulate=0):
    B, H = spec.q.shape[:2]
    refs = [np.zeros(p.shape) for p in spec.prev]
    for b in range(B):
        for h in range(H):
            c = oracle.attention_backward_block(spec.q[b, h], spec.k[b, h], spec.v[b, h], spec.do[b, h],
                                                spec.lse[b, h], spec.delta[b, h], scale_for(D), causal=causal,
                                                q_pos=positions(spec.qs), k_pos=positions(spec.ks))
            for r, x in zip(refs, c):
                r[b, h] = x
    for name, g, r, p in zip(("dq", "dk", "dv"), got, refs, spec.prev):
        assert_close(name, g, r + (p.double().numpy() if accumulate else 0), tol_for(dtype))


ALGOS = [("tc", torch.bfloat16), ("simt", torch.bfloat16), ("simt", torch.float32)]


def _algo(sca, name):
    return sca.capi.SCA_ALGO_TC if name == "tc" else sca.capi.SCA_ALGO_SIMT


@pytest.mark.parametrize("algo,dtype", ALGOS)
@pytest.mark.parametrize("r,j", [(1, 1), (2, 0), (0, 3), (3, 3)])
@pytest.mark.parametrize("accumulate", [0, 1])
def test_zigzag_item(sca, algo, dtype, r, j, accumulate):
    P, c, D = 4, 256, 128
    qs, ks = (2, c, (r * c, (2 * P - 1 - r) * c)), (2, c, (j * c, (2 * P - 1 - j) * c))
    s = Spec(1, 2, D, 2 * c, 2 * c, qs, ks, dtype, seed=10 * r + j)
    got = run(sca, [s], dtype, _algo(sca, algo), D, 1, 2, accumulate=accumulate)[0]
    check(s, got, dtype, D, accumulate=accumulate)


@pytest.mark.parametrize("algo,dtype", ALGOS)
@pytest.mark.parametrize("Sq,Skv,q0,k0", [(200, 333, 133, 0), (130, 260, 300, 0), (64, 300, 0, 5),
                                           (257, 100, 1000, 0)])
def test_ragged_item(sca, algo, dtype, Sq, Skv, q0, k0):
    D = 128
    s = Spec(1, 2, D, Sq, Skv, (1, Sq, (q0, 0)), (1, Skv, (k0, 0)), dtype, seed=Sq + Skv)
    got = run(sca, [s], dtype, _algo(sca, algo), D, 1, 2)[0]
    check(s, got, dtype, D)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_tiles_straddle_segments(sca, algo, dtype):
    P, c, D, r, j = 4, 100, 128, 2, 1
    qs, ks = (2, c, (r * c, (2 * P - 1 - r) * c)), (2, c, (j * c, (2 * P - 1 - j) * c))
    s = Spec(1, 2, D, 2 * c, 2 * c, qs, ks, dtype, seed=77)
    got = run(sca, [s], dtype, _algo(sca, algo), D, 1, 2, accumulate=1)[0]
    check(s, got, dtype, D, accumulate=1)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_block_nobody_sees(sca, algo, dtype):
    D = 128
    s = Spec(1, 2, D, 256, 256, (1, 256, (0, 0)), (1, 256, (256, 0)), dtype, seed=5)
    for acc in (0, 1):
        got = run(sca, [s], dtype, _algo(sca, algo), D, 1, 2, accumulate=acc)[0]
        check(s, got, dtype, D, accumulate=acc)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_non_causal_and_head_dim_64(sca, algo, dtype):
    s = Spec(2, 3, 64, 192, 320, (1, 192, (0, 0)), (1, 320, (0, 0)), dtype, seed=8, causal=False)
    got = run(sca, [s], dtype, _algo(sca, algo), 64, 2, 3, causal=False)[0]
    check(s, got, dtype, 64, causal=False)
    s = Spec(2, 3, 64, 384, 384, (2, 192, (192, 384)), (2, 192, (0, 576)), dtype, seed=9)
    got = run(sca, [s], dtype, _algo(sca, algo), 64, 2, 3)[0]
    check(s, got, dtype, 64)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_several_items_one_launch(sca, algo, dtype):
    P, c, D = 4, 128, 128
    specs = []
    for n, (r, j) in enumerate([(0, 0), (1, 0), (2, 3), (3, 1)]):
        qs, ks = (2, c, (r * c, (2 * P - 1 - r) * c)), (2, c, (j * c, (2 * P - 1 - j) * c))
        specs.append(Spec(1, 2, D, 2 * c, 2 * c, qs, ks, dtype, seed=100 + n))
    outs = run(sca, specs, dtype, _algo(sca, algo), D, 1, 2, accumulate=1)
    for s, got in zip(specs, outs):
        check(s, got, dtype, D, accumulate=1)


def test_long_block_tensor_cores_vs_fp32_kernel(sca):
    D, dtype = 128, torch.bfloat16
    s = Spec(1, 4, D, 1024, 2048, (1, 1024, (1024, 0)), (1, 2048, (0, 0)), dtype, seed=31)
    a = run(sca, [s], dtype, sca.capi.SCA_ALGO_TC, D, 1, 4)[0]
    b = run(sca, [s], dtype, sca.capi.SCA_ALGO_SIMT, D, 1, 4)[0]
    for name, x, y in zip(("dq", "dk", "dv"), a, b):
        assert_close(name + " tc vs simt", x, y.double().numpy(), (1e-2, 1e-3))
    check(s, a, dtype, D)


@pytest.mark.parametrize("accumulate", [0, 1])
def test_most_items_one_call(sca, accumulate):
    # SCA_MAX_ITEMS items in one call (the tensor-core launcher splits them
    # into launches of 28): every (query shard, key block) pair of P = 4
    # zigzag shards twice over, each with its own inputs and gradients
    D, P, c = 128, 4, 64
    specs = []
    for n in range(sca.capi.SCA_MAX_ITEMS):
        r, j = (n // P) % P, n % P
        qs = (2, c, (r * c, (2 * P - 1 - r) * c))
        ks = (2, c, (j * c, (2 * P - 1 - j) * c))
        specs.append(Spec(1, 1, D, 2 * c, 2 * c, qs, ks, torch.bfloat16, 1000 + 10 * n))
    got = run(sca, specs, torch.bfloat16, sca.capi.SCA_ALGO_TC, D, 1, 1, accumulate=accumulate)
    for spec, g in zip(specs, got):
        check(spec, g, torch.bfloat16, D, accumulate=accumulate)
