"""CPU oracle for per-token-group 8-bit quantization -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
leg of ``bench.py`` may import this package.  The product library never loads
it, and the oracle never loads the product: they share no code, header, table
or constant.  The arithmetic lives in ``ptgq_oracle.cpp`` (plain single-threaded
C++, binary32 steps in a fixed order); this module only builds it with g++ and
marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ptgq_oracle.cpp")
_LIB = os.path.join(_HERE, "libptgq_oracle.so")
_lock = threading.Lock()
_lib = None

IN_BF16, IN_FP16 = 0, 1
OUT_E4M3, OUT_INT8 = 0, 1
FMT_FP32, FMT_UE8M0_PACKED, FMT_UE8M0_FP32 = 0, 1, 2
LAYOUT_ROW, LAYOUT_COL = 0, 1
FLAG_UE8M0_SCALE_FLOOR = 1


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            f32, i32, i64, u16, vp = (ctypes.c_float, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_uint16, ctypes.c_void_p)
            L.oracle_bf16_to_float.argtypes = [u16]; L.oracle_bf16_to_float.restype = f32
            L.oracle_fp16_to_float.argtypes = [u16]; L.oracle_fp16_to_float.restype = f32
            L.oracle_exp_f32.argtypes = [f32]; L.oracle_exp_f32.restype = f32
            L.oracle_silu_mul.argtypes = [f32, f32]; L.oracle_silu_mul.restype = f32
            L.oracle_ue8m0_exponent.argtypes = [f32]; L.oracle_ue8m0_exponent.restype = i32
            L.oracle_pow2_from_biased.argtypes = [i32]; L.oracle_pow2_from_biased.restype = f32
            L.oracle_e4m3_encode.argtypes = [f32]; L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_int8_encode.argtypes = [f32]; L.oracle_int8_encode.restype = ctypes.c_int8
            L.oracle_scale_elems.argtypes = [i64, i64, i64, i32, i32, i32, i32]
            L.oracle_scale_elems.restype = i64
            L.oracle_quant.argtypes = [vp, i32, i64, i64, i64, i32, vp, i32, vp, i32, i32, i32, vp,
                                       f32, i32]
            L.oracle_quant.restype = i32
            L.oracle_quant_quotient_bound.argtypes = L.oracle_quant.argtypes + [i32]
            L.oracle_quant_quotient_bound.restype = i32
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = f32
            L.oracle_per_token_quant.argtypes = [vp, i32, i64, i64, vp, vp]
            L.oracle_per_token_quant.restype = i32
            L.oracle_requant_per_tensor.argtypes = [vp, vp, i64, i64, i64, vp, f32, vp, i64, i64,
                                                    i64, i32]
            L.oracle_requant_per_tensor.restype = i32
            _lib = L
    return _lib


def scale_elems(n, tokens_pad, hidden, group_size, scale_fmt, scale_layout, masked) -> int:
    return int(lib().oracle_scale_elems(n, tokens_pad, hidden, group_size, scale_fmt,
                                        scale_layout, int(bool(masked))))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def quant(x_bits: np.ndarray, in_dtype: int, n: int, tokens_pad: int, hidden: int,
          group_size: int, out_q: np.ndarray, out_dtype: int, out_s: np.ndarray,
          scale_fmt: int, scale_layout: int, fuse_silu: int, masked_m: np.ndarray | None,
          eps: float, flags: int = 0, quot_ulps: int = 0) -> None:
    """Run the oracle in place on numpy buffers (x as uint16 bit patterns).

    ``quot_ulps`` != 0 makes every code the encoding of a bound on the quotient, ``quot_ulps``
    binary32 ulps above (> 0) or below (< 0) the exact x / s, rounded outward; the scales are
    those of the operation itself.

    ``out_q`` (uint8) and ``out_s`` (float32, or uint32 for the packed format)
    keep whatever the caller put there wherever the method writes nothing.
    """
    assert x_bits.dtype == np.uint16 and x_bits.flags.c_contiguous
    assert out_q.dtype == np.uint8 and out_q.flags.c_contiguous
    assert out_s.dtype in (np.float32, np.uint32, np.int32) and out_s.flags.c_contiguous
    mm = None
    if masked_m is not None:
        mm = np.ascontiguousarray(masked_m, dtype=np.int32)
    args = (_ptr(x_bits), in_dtype, n, tokens_pad, hidden, group_size, _ptr(out_q), out_dtype,
            _ptr(out_s), scale_fmt, scale_layout, fuse_silu, _ptr(mm), float(eps), flags)
    if quot_ulps:
        rc = lib().oracle_quant_quotient_bound(*args, int(quot_ulps))
    else:
        rc = lib().oracle_quant(*args)
    if rc != 0:
        raise ValueError(f"oracle_quant rejected its arguments (rc={rc})")


def bf16_to_float(h: int) -> float:
    return lib().oracle_bf16_to_float(h)


def fp16_to_float(h: int) -> float:
    return lib().oracle_fp16_to_float(h)


def exp_f32(x: float) -> float:
    return lib().oracle_exp_f32(x)


def silu_mul(g: float, u: float) -> float:
    return lib().oracle_silu_mul(g, u)


def ue8m0_exponent(s: float) -> int:
    return lib().oracle_ue8m0_exponent(s)


def pow2_from_biased(e: int) -> float:
    return lib().oracle_pow2_from_biased(e)


def e4m3_encode(y: float) -> int:
    return lib().oracle_e4m3_encode(y)


def int8_encode(y: float) -> int:
    return lib().oracle_int8_encode(y)


def e4m3_decode(c: int) -> float:
    return lib().oracle_e4m3_decode(c)


IN_FP32 = 2


def per_token_quant(x: np.ndarray, in_dtype: int, out_q: np.ndarray, out_s: np.ndarray) -> None:
    """Per-token FP8 quantization of the rows of x ([T, hidden]: uint16 bit patterns for
    bf16/fp16, float32 for IN_FP32) into out_q (uint8, >= T rows) / out_s (float32)."""
    assert x.flags.c_contiguous and out_q.dtype == np.uint8 and out_s.dtype == np.float32
    T, hidden = x.shape
    rc = lib().oracle_per_token_quant(_ptr(x), in_dtype, T, hidden, _ptr(out_q), _ptr(out_s))
    if rc != 0:
        raise ValueError("oracle_per_token_quant rejected its arguments")


def requant_per_tensor(x: np.ndarray, x_scale: np.ndarray, strides, masked_m: np.ndarray,
                       output_scale: float, out: np.ndarray, group_size: int = 128) -> None:
    """Requantize e4m3 codes x [E, M, K] with per-token-group scales (element strides
    `strides` = (e, m, g) into x_scale) to one per-tensor scale, rows < masked_m only."""
    assert x.dtype == np.uint8 and out.dtype == np.uint8 and x_scale.dtype == np.float32
    E, M, K = x.shape
    mm = np.ascontiguousarray(masked_m, dtype=np.int32)
    rc = lib().oracle_requant_per_tensor(_ptr(x), _ptr(x_scale), strides[0], strides[1],
                                         strides[2], _ptr(mm), float(output_scale), _ptr(out),
                                         E, M, K, group_size)
    if rc != 0:
        raise ValueError("oracle_requant_per_tensor rejected its arguments")
