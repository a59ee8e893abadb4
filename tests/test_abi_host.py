"""The C ABI on the host, without a GPU: every symbol of include/sca.h is
exported, the ctypes mirrors match the C struct layouts, and invalid
arguments are rejected before anything is launched."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sca.h")

capi = pytest.importorskip("sharded_causal_softmax_gb300.capi")


@pytest.fixture(scope="module")
def lib():
    from sharded_causal_softmax_gb300 import build
    build.build()
    return capi.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:int|const char\s*\*)\s*(\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd_shard", "attn_merge_lse", "attn_bwd_shard", "zigzag_permute"):
        assert n in names
    assert set(names) == set(capi.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    if shutil.which("nm"):
        out = subprocess.run(["nm", "-D", "--defined-only", capi.LIB_PATH], capture_output=True, text=True).stdout
        for name in declared_functions():
            assert re.search(rf"\bT {name}$", out, flags=re.M), name


PROBE = r"""
#include <stddef.h>
#include <stdio.h>
#include "sca.h"
#define P(T) printf(#T " %zu\n", sizeof(T));
#define F(T, f) printf(#T "." #f " %zu\n", offsetof(T, f));
int main(void) {
  P(sca_segs) F(sca_segs, len) F(sca_segs, start)
  P(sca_view)
  P(sca_attn_dims) F(sca_attn_dims, scale) F(sca_attn_dims, accumulate) F(sca_attn_dims, q)
  F(sca_attn_dims, kv) F(sca_attn_dims, o) F(sca_attn_dims, dkv) F(sca_attn_dims, lse_b) F(sca_attn_dims, lse_h)
  F(sca_attn_dims, q_by_pos) F(sca_attn_dims, kv_by_pos) F(sca_attn_dims, dkv_by_pos) F(sca_attn_dims, kv_heads)
  P(sca_fwd_item) F(sca_fwd_item, o) F(sca_fwd_item, lse) F(sca_fwd_item, q_pos) F(sca_fwd_item, kv_pos)
  P(sca_bwd_item) F(sca_bwd_item, dout) F(sca_bwd_item, delta) F(sca_bwd_item, dv) F(sca_bwd_item, q_pos)
  F(sca_bwd_item, kv_pos)
  printf("SCA_MAX_ITEMS %d\n", SCA_MAX_ITEMS);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_ctypes_structs_match_c_layout(tmp_path):
    src = tmp_path / "probe.c"
    src.write_text(PROBE)
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                          check=True).stdout.splitlines())
    for key, val in got.items():
        if key == "SCA_MAX_ITEMS":
            assert int(val) == capi.SCA_MAX_ITEMS
            continue
        if "." in key:
            struct, field = key.split(".")
            assert getattr(getattr(capi, struct), field).offset == int(val), key
        else:
            assert ctypes.sizeof(getattr(capi, key)) == int(val), key


# --- argument validation (host only; pointers are never dereferenced) -----

A = 1 << 20   # an aligned fake device address


def _dims(**kw):
    d = capi.sca_attn_dims()
    d.B, d.H, d.D, d.dtype, d.causal, d.algo, d.scale = 1, 2, 128, capi.SCA_BF16, 1, 0, 0.088
    d.q = capi.view(2 * 256 * 128, 256 * 128, 128)
    d.kv = capi.view(2 * 256 * 128, 256 * 128, 128)
    d.o = capi.view(2 * 256 * 128, 256 * 128, 128)
    d.dkv = capi.view(2 * 256 * 128, 256 * 128, 128)
    d.lse_b, d.lse_h = 512, 256
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def _item(**kw):
    it = capi.sca_fwd_item()
    it.q = it.k = it.v = it.o = it.lse = A
    it.q_pos = capi.segs(1, 256, (0, 0))
    it.kv_pos = capi.segs(1, 256, (0, 0))
    for k, v in kw.items():
        setattr(it, k, v)
    return it


def _bwd_item(**kw):
    it = capi.sca_bwd_item()
    it.q = it.k = it.v = it.dout = it.lse = it.delta = it.dq = it.dk = it.dv = A
    it.q_pos = capi.segs(1, 256, (0, 0))
    it.kv_pos = capi.segs(1, 256, (0, 0))
    for k, v in kw.items():
        setattr(it, k, v)
    return it


def _fwd_rc(lib, items, dims, n=None):
    arr = (capi.sca_fwd_item * max(1, len(items)))(*items)
    return lib.attn_fwd_shard(arr, len(items) if n is None else n, ctypes.byref(dims), None, None)


@pytest.mark.parametrize("case,expect", [
    ("n_items_zero", capi.SCA_ERR_ARG),
    ("n_items_too_many", capi.SCA_ERR_ARG),
    ("head_dim_96", capi.SCA_ERR_UNSUPPORTED),
    ("f32_on_tensor_cores", capi.SCA_ERR_UNSUPPORTED),
    ("three_segments", capi.SCA_ERR_ARG),
    ("null_pointer", capi.SCA_ERR_ARG),
    ("misaligned_q", capi.SCA_ERR_ALIGN),
    ("odd_row_stride", capi.SCA_ERR_ALIGN),
    ("bad_dtype", capi.SCA_ERR_ARG),
    ("bad_algo", capi.SCA_ERR_ARG),
    ("nan_scale", capi.SCA_ERR_ARG),
    ("too_many_heads", capi.SCA_ERR_ARG),
    ("by_pos_flag_not_boolean", capi.SCA_ERR_ARG),
    ("by_pos_segment_not_x128", capi.SCA_ERR_UNSUPPORTED),
    ("by_pos_kv_segment_not_x128", capi.SCA_ERR_UNSUPPORTED),
    ("dkv_by_pos_in_forward", capi.SCA_ERR_ARG),
    ("kv_heads_not_dividing", capi.SCA_ERR_ARG),
    ("kv_heads_negative", capi.SCA_ERR_ARG),
])
def test_fwd_rejects_bad_arguments(lib, case, expect):
    items, dims, n = [_item()], _dims(), None
    if case == "n_items_zero":
        n = 0
    elif case == "n_items_too_many":
        n = capi.SCA_MAX_ITEMS + 1
    elif case == "head_dim_96":
        dims = _dims(D=96)
    elif case == "f32_on_tensor_cores":
        dims = _dims(dtype=capi.SCA_F32, algo=capi.SCA_ALGO_TC)
    elif case == "three_segments":
        items = [_item(q_pos=capi.segs(1, 256, (0, 0)))]
        items[0].q_pos.n = 3
    elif case == "null_pointer":
        items = [_item(v=None)]
    elif case == "misaligned_q":
        items = [_item(q=A + 2)]
    elif case == "odd_row_stride":
        dims = _dims(q=capi.view(2 * 256 * 130, 256 * 130, 130))
    elif case == "bad_dtype":
        dims = _dims(dtype=7)
    elif case == "bad_algo":
        dims = _dims(algo=9)
    elif case == "nan_scale":
        dims = _dims(scale=float("nan"))
    elif case == "too_many_heads":
        dims = _dims(B=300, H=300)
    elif case == "by_pos_flag_not_boolean":
        dims = _dims(q_by_pos=2)
    elif case == "by_pos_segment_not_x128":   # zigzag chunks of 96 rows: a tile would straddle two
        dims = _dims(q_by_pos=1)
        items = [_item(q_pos=capi.segs(2, 96, (0, 672)))]
    elif case == "by_pos_kv_segment_not_x128":
        dims = _dims(kv_by_pos=1)
        items = [_item(kv_pos=capi.segs(1, 200, (0, 0)))]
    elif case == "dkv_by_pos_in_forward":
        dims = _dims(dkv_by_pos=1)
    elif case == "kv_heads_not_dividing":   # H = 2
        dims = _dims(kv_heads=3)
    elif case == "kv_heads_negative":
        dims = _dims(kv_heads=-1)
    rc = _fwd_rc(lib, items, dims, n)
    assert rc == expect, (case, rc, capi.last_error())
    assert capi.last_error()


def test_bwd_rejects_bad_arguments(lib):
    arr = (capi.sca_bwd_item * 1)(_bwd_item(kv_pos=capi.segs(2, 64, (0, 192))))
    assert lib.attn_bwd_shard(arr, 1, ctypes.byref(_dims(dkv_by_pos=1)), None, None) == capi.SCA_ERR_UNSUPPORTED
    arr = (capi.sca_bwd_item * 1)(_bwd_item(delta=None))
    assert lib.attn_bwd_shard(arr, 1, ctypes.byref(_dims()), None, None) == capi.SCA_ERR_ARG


@pytest.mark.parametrize("case", ["unknown_bit", "forward", "f32_inputs", "simt_algo", "dout_without_groups"])
def test_f16_inputs_flag_rejected_outside_the_tensor_core_backward(lib, case):
    bwd = (capi.sca_bwd_item * 1)(_bwd_item())
    if case == "unknown_bit":
        rc = lib.attn_bwd_shard(bwd, 1, ctypes.byref(_dims(f16_inputs=4)), None, None)
    elif case == "forward":
        rc = _fwd_rc(lib, [_item()], _dims(f16_inputs=capi.SCA_F16_Q))
    elif case == "f32_inputs":
        rc = lib.attn_bwd_shard(bwd, 1, ctypes.byref(_dims(f16_inputs=capi.SCA_F16_Q, dtype=capi.SCA_F32)),
                                None, None)
    elif case == "simt_algo":
        rc = lib.attn_bwd_shard(bwd, 1, ctypes.byref(_dims(f16_inputs=capi.SCA_F16_Q, algo=capi.SCA_ALGO_SIMT)),
                                None, None)
    else:   # H = 2 query heads over 2 key/value heads: no groups, dO stays bf16
        rc = lib.attn_bwd_shard(bwd, 1, ctypes.byref(_dims(f16_inputs=capi.SCA_F16_DOUT, kv_heads=2)), None, None)
    assert rc == capi.SCA_ERR_ARG, (case, rc, capi.last_error())
    assert "f16_inputs" in capi.last_error()


def test_cast_rejects_bad_arguments(lib):
    f = lib.cast_bf16_to_f16
    assert f(None, A, 8, None, None) == capi.SCA_ERR_ARG
    assert f(A, 2 * A, 12, None, None) == capi.SCA_ERR_ARG          # not whole 16-byte vectors
    assert f(A, 2 * A, -8, None, None) == capi.SCA_ERR_ARG
    assert f(A + 8, 2 * A, 8, None, None) == capi.SCA_ERR_ALIGN
    assert f(A, A + 16, 64, None, None) == capi.SCA_ERR_ARG         # overlapping ranges
    assert f(A, 2 * A, 0, 3 * A, None) == capi.SCA_OK               # nothing to do, no launch
    arr = (capi.sca_bwd_item * 1)(_bwd_item(dk=A + 4))
    assert lib.attn_bwd_shard(arr, 1, ctypes.byref(_dims()), None, None) == capi.SCA_ERR_ALIGN
    assert lib.attn_bwd_shard(arr, 0, ctypes.byref(_dims()), None, None) == capi.SCA_ERR_ARG


def test_permute_rejects_bad_arguments(lib):
    f = lib.zigzag_permute
    assert f(A, 2 * A, 4, 100, 256, 4, 0, None, None) == capi.SCA_ERR_ARG           # 100 % 8 != 0
    assert f(A, 2 * A, 4, 64, 256, 0, 0, None, None) == capi.SCA_ERR_ARG             # P = 0
    assert f(A, 2 * A, 4, 64, 6, 4, 0, None, None) == capi.SCA_ERR_ARG               # row bytes not x4
    assert f(None, 2 * A, 4, 64, 256, 4, 0, None, None) == capi.SCA_ERR_ARG
    assert f(A, A + 256, 4, 64, 256, 4, 0, None, None) == capi.SCA_ERR_ARG           # overlap
    assert f(A + 2, 2 * A, 4, 64, 256, 4, 0, None, None) == capi.SCA_ERR_ALIGN
    assert f(A, 2 * A, 0, 64, 256, 4, 0, None, None) == capi.SCA_OK                  # empty: nothing to do


def test_merge_rejects_bad_arguments(lib):
    f = lib.attn_merge_lse
    assert f(A, 2 * A, 0, 10, 128, 1280, 10, 3 * A, 4 * A, None, 0, 0, None) == capi.SCA_ERR_ARG   # n = 0
    assert f(A, 2 * A, 2, 10, 96, 960, 10, 3 * A, 4 * A, None, 0, 0, None) == capi.SCA_ERR_ARG    # D = 96
    assert f(A, 2 * A, 2, 10, 128, 100, 10, 3 * A, 4 * A, None, 0, 0, None) == capi.SCA_ERR_ARG   # stride
    assert f(A + 4, 2 * A, 2, 10, 128, 1280, 10, 3 * A, 4 * A, None, 0, 0, None) == capi.SCA_ERR_ALIGN
    assert f(A, 2 * A, 2, 10, 128, 1280, 10, 3 * A, 4 * A, None, 4, 12, None) == capi.SCA_ERR_ARG  # S % 2P
    assert f(A, 2 * A, 2, 0, 128, 0, 0, 3 * A, 4 * A, None, 0, 0, None) == capi.SCA_OK


def test_merge_rejects_overlaps_other_than_one_partials_rows(lib):
    """An output may be exactly one partial's rows (each element is then read
    and written by the same lanes); any other overlap races and is refused
    before a launch.  (The exact alias itself runs on the GPU tests.)"""
    f = lib.attn_merge_lse
    rows, D, n = 10, 128, 2
    ob, lb = rows * D * 4, rows * 4
    op, lp = A, 2 * A          # partials: o at A (stride rows*D), lse at 2A (stride rows)
    def call(o_out, lse_out, bf=None, uP=0, S=0):
        return f(op, lp, n, rows, D, rows * D, rows, o_out, lse_out, bf, uP, S, None)
    assert call(op + 16, 4 * A) == capi.SCA_ERR_ARG               # o_out shifted by 4 columns into partial 0
    assert call(op + ob + 512, 4 * A) == capi.SCA_ERR_ARG         # o_out straddles partial 1 at a row offset
    assert call(3 * A, lp + 4) == capi.SCA_ERR_ARG                # lse_out one row into partial 0's lse
    assert call(3 * A, op + 64) == capi.SCA_ERR_ARG               # lse_out inside the o partials
    assert call(lp, 4 * A) == capi.SCA_ERR_ARG                    # o_out over the lse partials
    assert call(3 * A, 3 * A + 256) == capi.SCA_ERR_ARG           # lse_out inside o_out
    assert call(3 * A, 4 * A, bf=3 * A + 1024) == capi.SCA_ERR_ARG   # bf16 copy over o_out
    assert call(3 * A, 4 * A, bf=op) == capi.SCA_ERR_ARG             # bf16 copy over partial 0
    assert call(op, lp, uP=1, S=rows) == capi.SCA_ERR_ARG         # unpermuting: no alias at all
    assert call(op + ob, lp + lb, uP=1, S=rows) == capi.SCA_ERR_ARG


def test_stage_copies_reject_bad_arguments(lib):
    f = lib.ring_stage_copies
    ok = capi.copy2d(A, 2 * A, 4, 256, 512, 256)
    arr = lambda *cs: (capi.sca_copy * len(cs))(*cs)
    assert f(arr(ok), capi.SCA_MAX_COPIES + 1, None) == capi.SCA_ERR_ARG                       # too many copies
    assert f(None, 1, None) == capi.SCA_ERR_ARG
    assert f(arr(capi.copy2d(0, 2 * A, 4, 256, 512, 256)), 1, None) == capi.SCA_ERR_ARG        # NULL source
    assert f(arr(capi.copy2d(A, 2 * A, 4, 250, 512, 256)), 1, None) == capi.SCA_ERR_ARG        # width not x16
    assert f(arr(capi.copy2d(A, 2 * A, 4, 256, 128, 256)), 1, None) == capi.SCA_ERR_ARG        # pitch < width
    assert f(arr(capi.copy2d(A + 8, 2 * A, 4, 256, 512, 256)), 1, None) == capi.SCA_ERR_ALIGN
    assert f(arr(capi.copy2d(A, A + 512, 4, 256, 512, 256)), 1, None) == capi.SCA_ERR_ARG      # overlapping
    assert f(arr(ok), 0, None) == capi.SCA_OK                                                   # nothing to do
    assert f(arr(capi.copy2d(A, 2 * A, 0, 256, 512, 256)), 1, None) == capi.SCA_OK             # empty copy


def test_stage_and_delta_reject_bad_arguments(lib):
    assert lib.ring_stage_block(A, 2 * A, 4, 64, 60, 8, 256, None) == capi.SCA_ERR_ARG   # rows past S
    assert lib.attn_bwd_delta(A, 2 * A, capi.SCA_BF16, 3 * A, 10, 96, None) == capi.SCA_ERR_UNSUPPORTED
    assert lib.attn_bwd_delta(A + 4, 2 * A, capi.SCA_BF16, 3 * A, 10, 128, None) == capi.SCA_ERR_ALIGN
    assert lib.sca_read_status(None, None) == capi.SCA_ERR_ARG


def test_binding_raises_with_message(lib):
    with pytest.raises(capi.ScaError) as e:
        capi.zigzag_permute(A, 2 * A, 4, 100, 256, 4, 0, 0, 0)
    assert "SCA_ERR_ARG" in str(e.value) and "divisible" in str(e.value)


def test_lasp_rejects_bad_arguments(lib):
    bf, f32, F, T = capi.SCA_BF16, capi.SCA_F32, capi.SCA_LASP_BLOCK_F32, capi.SCA_LASP_BLOCK_TC
    assert lib.lasp_block_states(A, 2 * A, bf, 3 * A, 2, 1024, 96, F, None, None) == capi.SCA_ERR_UNSUPPORTED  # D
    assert lib.lasp_block_states(A, 2 * A, bf, 3 * A, 2, 1000, 128, F, None, None) == capi.SCA_ERR_ARG   # S % 64
    assert lib.lasp_block_states(A, 2 * A, bf, 3 * A, 2, 1088, 128, T, None, None) == capi.SCA_ERR_ARG   # S % 128
    assert lib.lasp_block_states(None, 2 * A, bf, 3 * A, 2, 1024, 128, F, None, None) == capi.SCA_ERR_ARG
    assert lib.lasp_block_states(A, 2 * A, bf, 3 * A, 2, 1024, 128, 96, None, None) == capi.SCA_ERR_ARG  # block
    assert lib.lasp_block_states(A, 2 * A, bf, 3 * A, 2, 8192, 128, 8192, None, None) == capi.SCA_ERR_ARG  # > 4096
    assert lib.lasp_scan(A, 2 * A, 2, 1024, 128, 4, 512, 0, None) == capi.SCA_ERR_ARG                  # 1024 % (512*4)
    # tensor-core blocks need bf16 and D = 128
    assert lib.lasp_block_states(A, 2 * A, f32, 3 * A, 2, 1024, 128, T, None, None) == capi.SCA_ERR_UNSUPPORTED
    assert lib.lasp_fwd(A, A, A, bf, A, A, A, 2, 1024, 64, 4, T, 0.1, None, None) == capi.SCA_ERR_UNSUPPORTED
    assert lib.lasp_scan(A, 2 * A, 2, 1024, 128, 3, F, 0, None) == capi.SCA_ERR_ARG                    # 1024 % (64*3)
    assert lib.lasp_scan(A, 2 * A, 2, 1024, 128, 16, T, 0, None) == capi.SCA_ERR_ARG                   # 1024 % (128*16)
    assert lib.lasp_exchange(A, 2 * A, 0, 128, 4, 0, None) == capi.SCA_ERR_ARG                         # BH = 0
    assert lib.lasp_fwd(A, A, A, 7, A, A, A, 2, 1024, 128, 4, F, 0.1, None, None) == capi.SCA_ERR_ARG  # dtype
    assert lib.lasp_bwd(A, A, A, A, bf, A, A, A, A, A, A, None, 2, 1024, 128, 4, T, 0.1, None, None) == \
        capi.SCA_ERR_ARG

def test_selftest_wait_rejects_null_status(lib):
    assert lib.sca_selftest_wait_timeout(None, None) == capi.SCA_ERR_ARG
