"""ctypes binding of libsca.so: the C ABI of ``include/sca.h``, one Python
function per entry point with the same name.  Argument marshalling only -
every step of the computation runs in the library's CUDA kernels.

Loading fails loudly (ImportError) when the library has not been built; there
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_void_p

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsca.so")

SCA_OK = 0
SCA_ERR_ARG = -1
SCA_ERR_UNSUPPORTED = -2
SCA_ERR_CUDA = -3
SCA_ERR_TIMEOUT = -4
SCA_ERR_ALIGN = -5
SCA_ERR_RANGE = -6
STATUS_NAMES = {0: "SCA_OK", -1: "SCA_ERR_ARG", -2: "SCA_ERR_UNSUPPORTED", -3: "SCA_ERR_CUDA",
                -4: "SCA_ERR_TIMEOUT", -5: "SCA_ERR_ALIGN", -6: "SCA_ERR_RANGE"}

SCA_BF16 = 0
SCA_F32 = 1
SCA_ALGO_AUTO = 0
SCA_ALGO_SIMT = 1
SCA_ALGO_TC = 2
SCA_MAX_ITEMS = 32
SCA_F16_Q = 1
SCA_F16_DOUT = 2
SCA_MAX_COPIES = 128

EXPORTED = ("attn_fwd_shard", "attn_merge_lse", "zigzag_permute", "ring_stage_block", "ring_stage_segments",
            "ring_stage_copies",
            "attn_bwd_shard", "attn_bwd_delta", "cast_bf16_to_f16", "lasp_block_states", "lasp_scan",
            "lasp_exchange", "lasp_fwd", "lasp_bwd", "lasp_fwd_noalloc", "sca_selftest_wait_timeout",
            "sca_last_error", "sca_read_status", "sca_version")
SCA_LASP_BLOCK_F32 = 64    # blocks of the fp32 CUDA-core kernels
SCA_LASP_BLOCK_TC = 128    # tensor-core kernels (bf16, D = 128): blocks of a multiple of this, up to 4096


class ScaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class sca_segs(ctypes.Structure):
    _fields_ = [("n", c_int32), ("reserved", c_int32), ("len", c_int64), ("start", c_int64 * 2)]


class sca_view(ctypes.Structure):
    _fields_ = [("b", c_int64), ("h", c_int64), ("s", c_int64)]


class sca_attn_dims(ctypes.Structure):
    _fields_ = [("B", c_int32), ("H", c_int32), ("D", c_int32), ("dtype", c_int32), ("causal", c_int32),
                ("algo", c_int32), ("scale", c_float), ("accumulate", c_int32), ("q", sca_view), ("kv", sca_view),
                ("o", sca_view), ("dkv", sca_view), ("lse_b", c_int64), ("lse_h", c_int64),
                ("q_by_pos", c_int32), ("kv_by_pos", c_int32), ("dkv_by_pos", c_int32), ("kv_heads", c_int32),
                ("f16_inputs", c_int32)]


class sca_copy(ctypes.Structure):
    _fields_ = [("src", c_void_p), ("dst", c_void_p), ("height", c_int64), ("width", c_int64),
                ("src_pitch", c_int64), ("dst_pitch", c_int64)]


class sca_fwd_item(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("o", c_void_p), ("lse", c_void_p),
                ("q_pos", sca_segs), ("kv_pos", sca_segs)]


class sca_bwd_item(ctypes.Structure):
    _fields_ = [("q", c_void_p), ("k", c_void_p), ("v", c_void_p), ("dout", c_void_p), ("lse", c_void_p),
                ("delta", c_void_p), ("dq", c_void_p), ("dk", c_void_p), ("dv", c_void_p),
                ("q_pos", sca_segs), ("kv_pos", sca_segs)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libsca.so not built ({LIB_PATH}); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` or "
                          "`python sharded_causal_softmax_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    sig = {
        "attn_fwd_shard": (c_int, [POINTER(sca_fwd_item), c_int, POINTER(sca_attn_dims), c_void_p, c_void_p]),
        "attn_merge_lse": (c_int, [c_void_p, c_void_p, c_int, c_int64, c_int, c_int64, c_int64, c_void_p,
                                   c_void_p, c_void_p, c_int, c_int64, c_void_p]),
        "zigzag_permute": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int, c_int, c_void_p, c_void_p]),
        "ring_stage_block": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int64, c_int64, c_int64, c_void_p]),
        "ring_stage_segments": (c_int, [c_void_p, c_void_p, c_int64, c_int64, POINTER(sca_segs), c_int64, c_void_p]),
        "ring_stage_copies": (c_int, [POINTER(sca_copy), c_int, c_void_p]),
        "attn_bwd_shard": (c_int, [POINTER(sca_bwd_item), c_int, POINTER(sca_attn_dims), c_void_p, c_void_p]),
        "attn_bwd_delta": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int64, c_int, c_void_p]),
        "cast_bf16_to_f16": (c_int, [c_void_p, c_void_p, c_int64, c_void_p, c_void_p]),
        "lasp_block_states": (c_int, [c_void_p, c_void_p, c_int, c_void_p, c_int64, c_int64, c_int, c_int, c_void_p,
                                      c_void_p]),
        "lasp_scan": (c_int, [c_void_p, c_void_p, c_int64, c_int64, c_int, c_int, c_int, c_int, c_void_p]),
        "lasp_exchange": (c_int, [c_void_p, c_void_p, c_int64, c_int, c_int, c_int, c_void_p]),
        "lasp_fwd": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_int64, c_int64,
                             c_int, c_int, c_int, c_float, c_void_p, c_void_p]),
        "lasp_bwd": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                             c_void_p, c_void_p, c_void_p, c_int64, c_int64, c_int, c_int, c_int, c_float, c_void_p,
                             c_void_p]),
        "lasp_fwd_noalloc": (c_int, [c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_int64, c_int64, c_int, c_int,
                                     c_float, c_void_p]),
        "sca_selftest_wait_timeout": (c_int, [c_void_p, c_void_p]),
        "sca_last_error": (c_char_p, []),
        "sca_read_status": (c_int, [c_void_p, c_void_p]),
        "sca_version": (c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def last_error() -> str:
    return lib().sca_last_error().decode(errors="replace")


def check(rc: int) -> int:
    if rc != SCA_OK:
        raise ScaError(rc, last_error())
    return rc


def _items_array(cls, items):
    arr = (cls * len(items))(*items)
    return arr


# ---- one function per C entry point (same names) -------------------------

def attn_fwd_shard(items, dims: sca_attn_dims, dev_status: int, stream: int) -> int:
    arr = _items_array(sca_fwd_item, items)
    return check(lib().attn_fwd_shard(arr, len(items), ctypes.byref(dims), dev_status, stream))


def attn_bwd_shard(items, dims: sca_attn_dims, dev_status: int, stream: int) -> int:
    arr = _items_array(sca_bwd_item, items)
    return check(lib().attn_bwd_shard(arr, len(items), ctypes.byref(dims), dev_status, stream))


def attn_merge_lse(o_parts: int, lse_parts: int, n: int, rows: int, D: int, o_part_stride: int,
                   lse_part_stride: int, o_out: int, lse_out: int, o_bf16_out: int, unpermute_P: int, S: int,
                   stream: int) -> int:
    return check(lib().attn_merge_lse(o_parts, lse_parts, n, rows, D, o_part_stride, lse_part_stride, o_out,
                                      lse_out, o_bf16_out, unpermute_P, S, stream))


def zigzag_permute(src: int, dst: int, outer: int, S: int, row_bytes: int, P: int, inverse: int,
                   dev_status: int, stream: int) -> int:
    return check(lib().zigzag_permute(src, dst, outer, S, row_bytes, P, inverse, dev_status, stream))


def ring_stage_block(src: int, dst: int, outer: int, S_src: int, row0: int, rows: int, row_bytes: int,
                     stream: int) -> int:
    return check(lib().ring_stage_block(src, dst, outer, S_src, row0, rows, row_bytes, stream))


def ring_stage_segments(src: int, dst: int, outer: int, S_src: int, seg: sca_segs, row_bytes: int,
                        stream: int) -> int:
    return check(lib().ring_stage_segments(src, dst, outer, S_src, ctypes.byref(seg), row_bytes, stream))


def ring_stage_copies(copies, stream: int) -> int:
    arr = (sca_copy * max(1, len(copies)))(*copies)
    return check(lib().ring_stage_copies(arr, len(copies), stream))


def copy2d(src: int, dst: int, height: int, width: int, src_pitch: int, dst_pitch: int) -> sca_copy:
    c = sca_copy()
    c.src, c.dst, c.height, c.width, c.src_pitch, c.dst_pitch = src, dst, height, width, src_pitch, dst_pitch
    return c


def lasp_block_states(a: int, b: int, dtype: int, st: int, BH: int, S: int, D: int, block: int, dev_status: int,
                      stream: int) -> int:
    return check(lib().lasp_block_states(a, b, dtype, st, BH, S, D, block, dev_status, stream))


def lasp_scan(st: int, shard_total: int, BH: int, S: int, D: int, P: int, block: int, reverse: int,
              stream: int) -> int:
    return check(lib().lasp_scan(st, shard_total, BH, S, D, P, block, reverse, stream))


def lasp_exchange(shard_total: int, shard_in: int, BH: int, D: int, P: int, reverse: int, stream: int) -> int:
    return check(lib().lasp_exchange(shard_total, shard_in, BH, D, P, reverse, stream))


def lasp_fwd(q: int, k: int, v: int, dtype: int, st: int, shard_in: int, o: int, BH: int, S: int, D: int, P: int,
             block: int, scale: float, dev_status: int, stream: int) -> int:
    return check(lib().lasp_fwd(q, k, v, dtype, st, shard_in, o, BH, S, D, P, block, scale, dev_status, stream))


def lasp_bwd(q: int, k: int, v: int, dout: int, dtype: int, st_fwd: int, in_fwd: int, st_bwd: int, in_bwd: int,
             dq: int, dk: int, dv: int, BH: int, S: int, D: int, P: int, block: int, scale: float, dev_status: int,
             stream: int) -> int:
    return check(lib().lasp_bwd(q, k, v, dout, dtype, st_fwd, in_fwd, st_bwd, in_bwd, dq, dk, dv, BH, S, D, P,
                                block, scale, dev_status, stream))


def sca_selftest_wait_timeout(dev_status: int, stream: int) -> int:
    return check(lib().sca_selftest_wait_timeout(dev_status, stream))


def lasp_fwd_noalloc(q: int, k: int, v: int, dtype: int, o: int, BH: int, S: int, D: int, P: int, scale: float,
                     stream: int) -> int:
    return check(lib().lasp_fwd_noalloc(q, k, v, dtype, o, BH, S, D, P, scale, stream))


def attn_bwd_delta(o: int, dout: int, dout_dtype: int, delta: int, rows: int, D: int, stream: int) -> int:
    return check(lib().attn_bwd_delta(o, dout, dout_dtype, delta, rows, D, stream))


def cast_bf16_to_f16(src: int, dst: int, n: int, dev_status: int, stream: int) -> int:
    return check(lib().cast_bf16_to_f16(src, dst, n, dev_status, stream))


def sca_read_status(dev_status: int, stream: int) -> int:
    return lib().sca_read_status(dev_status, stream)


def sca_version() -> int:
    return lib().sca_version()


def segs(n: int, length: int, starts) -> sca_segs:
    s = sca_segs()
    s.n = n
    s.len = length
    s.start[0] = starts[0]
    s.start[1] = starts[1] if n > 1 else 0
    return s


def view(b: int, h: int, s: int) -> sca_view:
    v = sca_view()
    v.b, v.h, v.s = b, h, s
    return v
