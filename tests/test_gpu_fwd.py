"""GPU parity of attn_fwd_shard: (o, lse) partials of single (query shard,
key block) items against the fp64 oracle, on the tensor-core kernel (bf16)
and the fp32-arithmetic kernel (bf16 and fp32 inputs), including ragged
tails, two-segment zigzag shards, tiles straddling segments, empty blocks,
non-causal rows, D = 64, several items per launch and strided views."""
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


def make(shape, dtype, seed, mult=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * mult).to(dtype)


def run_items(sca, items_spec, dtype, algo, D, B=1, H=2, causal=True, scale=None):
    """items_spec: list of (q, k, v) CPU tensors + (q_seg, kv_seg); returns list of (o, lse) CPU."""
    capi = sca.capi
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    items, keep, outs = [], [], []
    for (q, k, v, qs, ks) in items_spec:
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        Sq = q.shape[2]
        o = torch.full((B, H, Sq, D), float("nan"), device="cuda")
        lse = torch.full((B, H, Sq), float("nan"), device="cuda")
        it = capi.sca_fwd_item()
        it.q, it.k, it.v, it.o, it.lse = qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), lse.data_ptr()
        it.q_pos = capi.segs(qs[0], qs[1], qs[2])
        it.kv_pos = capi.segs(ks[0], ks[1], ks[2])
        items.append(it)
        keep += [qd, kd, vd]
        outs.append((o, lse, qd.stride(), kd.stride()))
    # all items of one launch share the views: the specs use equal strides
    q0s, k0s = outs[0][2], outs[0][3]
    d = capi.sca_attn_dims()
    d.B, d.H, d.D = B, H, D
    d.dtype = capi.SCA_BF16 if dtype == torch.bfloat16 else capi.SCA_F32
    d.causal, d.algo = 1 if causal else 0, algo
    d.scale = scale_for(D) if scale is None else scale
    d.q = capi.view(q0s[0], q0s[1], q0s[2])
    d.kv = capi.view(k0s[0], k0s[1], k0s[2])
    o0 = outs[0][0]
    d.o = capi.view(o0.stride(0), o0.stride(1), o0.stride(2))
    d.lse_b, d.lse_h = outs[0][1].stride(0), outs[0][1].stride(1)
    capi.attn_fwd_shard(items, d, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert sca.sca_read_status(status.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    return [(o.cpu(), lse.cpu()) for (o, lse, _, _) in outs]


def check_item(q, k, v, qs, ks, got, dtype, D, causal=True):
    o, lse = got
    B, H = q.shape[:2]
    ro = np.zeros(o.shape)
    rl = np.zeros(lse.shape)
    for b in range(B):
        for h in range(H):
            ro[b, h], rl[b, h] = oracle.attention(q[b, h], k[b, h], v[b, h], scale_for(D), causal=causal,
                                                  q_pos=positions(qs), k_pos=positions(ks))
    assert_close("o", o, ro, tol_for(dtype))
    assert_close("lse", lse, rl, tol_for(dtype))


ALGOS = [("tc", torch.bfloat16), ("simt", torch.bfloat16), ("simt", torch.float32)]


def _algo(sca, name):
    return sca.capi.SCA_ALGO_TC if name == "tc" else sca.capi.SCA_ALGO_SIMT


ZZ = 256   # zigzag chunk for P = 4, S = 2048


@pytest.mark.parametrize("algo,dtype", ALGOS)
@pytest.mark.parametrize("r,j", [(1, 1), (1, 0), (1, 3), (0, 0), (3, 3), (2, 1)])
def test_zigzag_item(sca, algo, dtype, r, j):
    P, c, D = 4, ZZ, 128
    qs = (2, c, (r * c, (2 * P - 1 - r) * c))
    ks = (2, c, (j * c, (2 * P - 1 - j) * c))
    q, k, v = make((1, 2, 2 * c, D), dtype, 1), make((1, 2, 2 * c, D), dtype, 2), make((1, 2, 2 * c, D), dtype, 3)
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, _algo(sca, algo), D)[0]
    check_item(q, k, v, qs, ks, got, dtype, D)


@pytest.mark.parametrize("algo,dtype", ALGOS)
@pytest.mark.parametrize("Sq,Skv,q0,k0", [(200, 333, 133, 0), (1, 129, 128, 0), (130, 130, 0, 0),
                                           (257, 100, 1000, 0), (64, 300, 0, 5)])
def test_ragged_item(sca, algo, dtype, Sq, Skv, q0, k0):
    D = 128
    qs, ks = (1, Sq, (q0, 0)), (1, Skv, (k0, 0))
    q, k, v = make((1, 2, Sq, D), dtype, 4), make((1, 2, Skv, D), dtype, 5), make((1, 2, Skv, D), dtype, 6)
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, _algo(sca, algo), D)[0]
    check_item(q, k, v, qs, ks, got, dtype, D)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_tiles_straddle_segments(sca, algo, dtype):
    # zigzag chunk of 100 rows: 128-row tiles cross the segment boundary
    P, c, D, r, j = 4, 100, 128, 2, 1
    qs = (2, c, (r * c, (2 * P - 1 - r) * c))
    ks = (2, c, (j * c, (2 * P - 1 - j) * c))
    q, k, v = make((1, 2, 2 * c, D), dtype, 7), make((1, 2, 2 * c, D), dtype, 8), make((1, 2, 2 * c, D), dtype, 9)
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, _algo(sca, algo), D)[0]
    check_item(q, k, v, qs, ks, got, dtype, D)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_empty_block_gives_empty_partial(sca, algo, dtype):
    D = 128
    q = make((1, 2, 300, D), dtype, 10)
    k = make((1, 2, 8, D), dtype, 11)
    o, lse = run_items(sca, [(q, k, k, (1, 300, (0, 0)), (1, 0, (0, 0)))], dtype, _algo(sca, algo), D)[0]
    assert torch.all(o == 0) and torch.all(lse == -float("inf"))
    # a block entirely in the future of every query
    k = make((1, 2, 256, D), dtype, 12)
    o, lse = run_items(sca, [(q, k, k, (1, 300, (0, 0)), (1, 256, (300, 0)))], dtype, _algo(sca, algo), D)[0]
    assert torch.all(o == 0) and torch.all(lse == -float("inf"))


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_non_causal(sca, algo, dtype):
    D = 128
    q, k, v = make((1, 2, 200, D), dtype, 13), make((1, 2, 300, D), dtype, 14), make((1, 2, 300, D), dtype, 15)
    qs, ks = (1, 200, (0, 0)), (1, 300, (0, 0))
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, _algo(sca, algo), D, causal=False)[0]
    check_item(q, k, v, qs, ks, got, dtype, D, causal=False)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_head_dim_64(sca, algo, dtype):
    D, P, c, r, j = 64, 2, 192, 1, 1
    qs = (2, c, (r * c, (2 * P - 1 - r) * c))
    ks = (2, c, (j * c, (2 * P - 1 - j) * c))
    q, k, v = make((2, 3, 2 * c, D), dtype, 16), make((2, 3, 2 * c, D), dtype, 17), make((2, 3, 2 * c, D), dtype, 18)
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, _algo(sca, algo), D, B=2, H=3)[0]
    check_item(q, k, v, qs, ks, got, dtype, D)


@pytest.mark.parametrize("algo,dtype", ALGOS)
def test_several_items_one_launch(sca, algo, dtype):
    D, P, c = 128, 4, 128
    specs = []
    for n, (r, j) in enumerate([(0, 0), (1, 0), (2, 3), (3, 1), (3, 3)]):
        qs = (2, c, (r * c, (2 * P - 1 - r) * c))
        ks = (2, c, (j * c, (2 * P - 1 - j) * c))
        specs.append((make((1, 2, 2 * c, D), dtype, 20 + n), make((1, 2, 2 * c, D), dtype, 40 + n),
                      make((1, 2, 2 * c, D), dtype, 60 + n), qs, ks))
    outs = run_items(sca, specs, dtype, _algo(sca, algo), D)
    for (q, k, v, qs, ks), got in zip(specs, outs):
        check_item(q, k, v, qs, ks, got, dtype, D)


def test_tensor_cores_sharp_softmax_and_long_block(sca):
    # Q scaled by 2 (sharper softmax, more rescales) over 4096 keys
    D, dtype = 128, torch.bfloat16
    q = make((1, 2, 512, D), dtype, 70, mult=2.0)
    k, v = make((1, 2, 4096, D), dtype, 71), make((1, 2, 4096, D), dtype, 72)
    qs, ks = (1, 512, (3584, 0)), (1, 4096, (0, 0))
    got = run_items(sca, [(q, k, v, qs, ks)], dtype, sca.capi.SCA_ALGO_TC, D)[0]
    check_item(q, k, v, qs, ks, got, dtype, D)


def test_tensor_cores_agree_with_fp32_kernel(sca):
    D, dtype, P, c, r, j = 128, torch.bfloat16, 4, 512, 2, 2
    qs = (2, c, (r * c, (2 * P - 1 - r) * c))
    ks = (2, c, (j * c, (2 * P - 1 - j) * c))
    q, k, v = make((1, 4, 2 * c, D), dtype, 80), make((1, 4, 2 * c, D), dtype, 81), make((1, 4, 2 * c, D), dtype, 82)
    a = run_items(sca, [(q, k, v, qs, ks)], dtype, sca.capi.SCA_ALGO_TC, D, H=4)[0]
    b = run_items(sca, [(q, k, v, qs, ks)], dtype, sca.capi.SCA_ALGO_SIMT, D, H=4)[0]
    assert_close("o tc vs simt", a[0], b[0].double().numpy(), (1e-2, 1e-3))
    assert_close("lse tc vs simt", a[1], b[1].double().numpy(), (1e-2, 1e-3))


@pytest.mark.parametrize("algo,dtype", [("tc", torch.bfloat16), ("simt", torch.float32)])
def test_most_items_one_launch(sca, algo, dtype):
    # SCA_MAX_ITEMS items in one call: every (query shard, key block) pair of
    # P = 4 zigzag shards twice over, with different inputs
    D, P, c = 128 if dtype == torch.bfloat16 else 64, 4, 64
    specs = []
    for n in range(sca.capi.SCA_MAX_ITEMS):
        r, j = (n // P) % P, n % P
        qs = (2, c, (r * c, (2 * P - 1 - r) * c))
        ks = (2, c, (j * c, (2 * P - 1 - j) * c))
        specs.append((make((1, 1, 2 * c, D), dtype, 100 + n), make((1, 1, 2 * c, D), dtype, 200 + n),
                      make((1, 1, 2 * c, D), dtype, 300 + n), qs, ks))
    got = run_items(sca, specs, dtype, _algo(sca, algo), D, H=1)
    for (q, k, v, qs, ks), g in zip(specs, got):
        check_item(q, k, v, qs, ks, g, dtype, D)
