"""GB300 (sm_103a) per-token-group 8-bit activation quantization.

A thin ctypes binding over ``libptgq.so`` (the C ABI in ``include/ptgq.h``).  PyTorch is
only used to hold device memory and to name the current CUDA stream; every step of the
quantization runs in the library's CUDA kernels.  There is no CPU fallback: if the
library is missing or no GPU is present, calls raise.

Typical use::

    import torch, fp8_token_group_gb300 as ptgq
    x = torch.randn(4096, 7168, device="cuda", dtype=torch.bfloat16)
    q, s = ptgq.quantize(x, group_size=128, scale_fmt=ptgq.SCALE_UE8M0_PACKED,
                         scale_layout=ptgq.COL_MAJOR_TMA)
"""
from __future__ import annotations

import ctypes
import functools
import os
import re
import threading

__all__ = [
    "BF16", "FP16", "FP32", "E4M3", "INT8", "SCALE_FP32", "SCALE_UE8M0_PACKED", "SCALE_UE8M0_FP32",
    "ROW_MAJOR", "COL_MAJOR_TMA", "FLAG_NO_PDL", "FLAG_UE8M0_SCALE_FLOOR", "FLAG_FAST_DIVIDE",
    "EPS_MIN",
    "PtgqError", "lib", "lib_path", "header_functions", "quant", "quantize", "scale_elems",
    "alloc_outputs", "strerror", "per_token_quant", "requant_per_tensor",
]

BF16, FP16, FP32 = 0, 1, 2
E4M3, INT8 = 0, 1
SCALE_FP32, SCALE_UE8M0_PACKED, SCALE_UE8M0_FP32 = 0, 1, 2
ROW_MAJOR, COL_MAJOR_TMA = 0, 1
FLAG_NO_PDL, FLAG_UE8M0_SCALE_FLOOR, FLAG_FAST_DIVIDE = 1, 2, 4
EPS_MIN = 2.0 ** -140          # PTGQ_EPS_MIN

_HERE = os.path.dirname(os.path.abspath(__file__))
_HEADER = os.path.join(os.path.dirname(_HERE), "include", "ptgq.h")
_lock = threading.Lock()
_lib = None


class PtgqError(RuntimeError):
    def __init__(self, status: int, what: str = "ptgq_quant"):
        self.status = status
        super().__init__(f"{what} failed with status {status}: {strerror(status)}")


def lib_path() -> str:
    return os.path.join(_HERE, "libptgq.so")


def header_functions() -> list[str]:
    """Names of the functions ``include/ptgq.h`` declares."""
    text = open(_HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(ptgq_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    """Load libptgq.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
            import torch  # noqa: F401  (loads the CUDA runtime the library links against)
            L = ctypes.CDLL(path, mode=ctypes.RTLD_GLOBAL)
            i32, i64, vp, f32 = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float
            L.ptgq_quant.argtypes = [vp, i32, i64, i64, i64, i32, vp, i32, vp, i32, i32, i32, vp,
                                     f32, vp]
            L.ptgq_quant.restype = i32
            L.ptgq_quant_ex.argtypes = L.ptgq_quant.argtypes + [ctypes.c_uint, i64, vp]
            L.ptgq_quant_ex.restype = i32
            L.ptgq_scale_elems.argtypes = [i64, i64, i64, i32, i32, i32, i32,
                                           ctypes.POINTER(i64)]
            L.ptgq_scale_elems.restype = i32
            L.ptgq_per_token_quant.argtypes = [vp, i32, i64, i64, vp, vp, vp]
            L.ptgq_per_token_quant.restype = i32
            L.ptgq_requant_per_tensor.argtypes = [vp, vp, i64, i64, i64, vp, vp, vp, i64, i64,
                                                  i64, i32, vp]
            L.ptgq_requant_per_tensor.restype = i32
            L.ptgq_strerror.argtypes = [i32]
            L.ptgq_strerror.restype = ctypes.c_char_p
            _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().ptgq_strerror(status).decode()


@functools.lru_cache(maxsize=1024)
def scale_elems(n: int, tokens_pad: int, hidden: int, group_size: int, scale_fmt: int,
                scale_layout: int, masked: bool) -> int:
    """Scale elements (floats, or int32 words when packed) out_s must hold; see
    ``ptgq_scale_elems``."""
    out = ctypes.c_int64(0)
    rc = lib().ptgq_scale_elems(n, tokens_pad, hidden, group_size, scale_fmt, scale_layout,
                                int(bool(masked)), ctypes.byref(out))
    if rc != 0:
        raise PtgqError(rc, "ptgq_scale_elems")
    return out.value


def hidden_ok(hidden: int, group_size: int) -> bool:
    """Whether the size query is meaningful (otherwise the library rejects the call itself)."""
    return group_size in (16, 32, 64, 128) and hidden > 0 and hidden % group_size == 0


def _in_dtype(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    raise TypeError(f"input must be bfloat16 or float16, got {t.dtype}")


def alloc_outputs(x, group_size: int, *, out_dtype: int = E4M3, scale_fmt: int = SCALE_FP32,
                  scale_layout: int = ROW_MAJOR, fuse_silu: bool = False, masked: bool = False,
                  tokens_pad: int = 0):
    """Allocate (out_q, out_s) on x's device for the given configuration."""
    import torch
    if masked:
        E, tp, hin = x.shape
        n, rows = E, tp
        tokens_pad = tp
    else:
        n, hin = x.shape
        rows = tokens_pad or n
    if fuse_silu and hin % 2 != 0:
        raise ValueError(f"fuse_silu needs gate and up halves of equal width; the last "
                         f"dimension of x is {hin}")
    H = hin // 2 if fuse_silu else hin
    qshape = (n, rows, H) if masked else (rows, H)
    qdt = torch.float8_e4m3fn if out_dtype == E4M3 else torch.int8
    q = torch.empty(qshape, dtype=qdt, device=x.device)
    ns = scale_elems(n, tokens_pad, H, group_size, scale_fmt, scale_layout, masked)
    sdt = torch.int32 if scale_fmt == SCALE_UE8M0_PACKED else torch.float32
    s = torch.empty(ns, dtype=sdt, device=x.device)
    return q, s


def quant(x, out_q, out_s, group_size: int, *, out_dtype: int | None = None,
          scale_fmt: int = SCALE_FP32, scale_layout: int = ROW_MAJOR, fuse_silu: bool = False,
          masked_m=None, eps: float = 1e-10, tokens_pad: int = 0, flags: int = 0,
          expected_m: int = 0, masked_m_errors=None, stream=None) -> None:
    """Quantize ``x`` into the caller's ``out_q`` / ``out_s`` on ``stream`` (default: torch's
    current stream).  Tensors must be device-accessible: CUDA tensors, or pinned host tensors,
    which the GPU reads and writes in place over the host link (unified addressing).
    Arguments follow ``ptgq_quant_ex`` in include/ptgq.h; ``masked_m_errors`` is an optional
    device int32 tensor that counts masked_m entries outside [0, tokens_pad]."""
    import torch
    all_cuda = x.is_cuda and out_q.is_cuda and out_s.is_cuda
    if not all_cuda:
        for name, t in (("x", x), ("out_q", out_q), ("out_s", out_s)):
            if not (t.is_cuda or t.is_pinned()):
                raise ValueError(f"{name} must be a CUDA tensor or pinned host memory "
                                 "(use quantize() for pageable host tensors)")
    if not (x.is_contiguous() and out_q.is_contiguous() and out_s.is_contiguous()):
        raise ValueError("x, out_q and out_s must be contiguous")
    if out_dtype is None:
        out_dtype = INT8 if out_q.dtype == torch.int8 else E4M3
    if masked_m is not None:
        if masked_m.dtype != torch.int32 or not (masked_m.is_cuda or masked_m.is_pinned()):
            raise ValueError("masked_m must be a device-accessible int32 tensor")
        E, tp, hin = x.shape
        n, tokens_pad = E, tp
        if E == 0:
            return      # no experts: nothing to read or write (an empty masked_m has no address)
    else:
        n, hin = x.shape
    if fuse_silu and hin % 2 != 0:
        raise ValueError(f"fuse_silu needs gate and up halves of equal width; the last "
                         f"dimension of x is {hin}")
    H = hin // 2 if fuse_silu else hin
    # The library sees raw pointers; check here that the outputs hold what the call writes,
    # so a short buffer is an exception rather than a write past its end.
    rows = tokens_pad if masked_m is not None else (tokens_pad or n)
    need_q = (n if masked_m is not None else 1) * rows * H
    if out_q.numel() * out_q.element_size() < need_q:
        raise ValueError(f"out_q holds {out_q.numel() * out_q.element_size()} bytes; "
                         f"the call writes up to {need_q}")
    if hidden_ok(H, group_size):
        need_s = 4 * scale_elems(n, tokens_pad, H, group_size, scale_fmt, scale_layout,
                                 masked_m is not None)
        if out_s.numel() * out_s.element_size() < need_s:
            raise ValueError(f"out_s holds {out_s.numel() * out_s.element_size()} bytes; "
                             f"the call writes up to {need_s}")
    if masked_m is not None and masked_m.numel() < n:
        raise ValueError(f"masked_m has {masked_m.numel()} entries for {n} experts")
    err_ptr = None
    if masked_m_errors is not None:
        if masked_m_errors.dtype != torch.int32 or not masked_m_errors.is_cuda:
            raise ValueError("masked_m_errors must be an int32 CUDA tensor")
        err_ptr = masked_m_errors.data_ptr()
    handle = _stream_handle(stream, x.get_device() if x.is_cuda else None)
    rc = (_lib or lib()).ptgq_quant_ex(
        x.data_ptr(), _in_dtype(x), n, tokens_pad, H, group_size, out_q.data_ptr(), out_dtype,
        out_s.data_ptr(), scale_fmt, scale_layout, int(bool(fuse_silu)),
        None if masked_m is None else masked_m.data_ptr(), float(eps), handle, flags,
        int(expected_m), err_ptr)
    if rc != 0:
        raise PtgqError(rc)


def quantize(x, group_size: int = 128, *, out_dtype: int = E4M3, scale_fmt: int = SCALE_FP32,
             scale_layout: int = ROW_MAJOR, fuse_silu: bool = False, masked_m=None,
             eps: float = 1e-10, tokens_pad: int = 0, flags: int = 0, expected_m: int = 0):
    """Allocate outputs and quantize.  A host (CPU) ``x`` is copied to the current CUDA
    device, quantized there, and the outputs are copied back to the host."""
    import torch
    host = not x.is_cuda
    xd = x.to("cuda", non_blocking=True) if host else x
    mm = masked_m
    if mm is not None and not mm.is_cuda:
        mm = mm.to("cuda", non_blocking=True)
    q, s = alloc_outputs(xd, group_size, out_dtype=out_dtype, scale_fmt=scale_fmt,
                         scale_layout=scale_layout, fuse_silu=fuse_silu,
                         masked=mm is not None, tokens_pad=tokens_pad)
    quant(xd, q, s, group_size, out_dtype=out_dtype, scale_fmt=scale_fmt,
          scale_layout=scale_layout, fuse_silu=fuse_silu, masked_m=mm, eps=eps,
          tokens_pad=tokens_pad, flags=flags, expected_m=expected_m)
    if host:
        q, s = q.cpu(), s.cpu()
    return q, s


def _stream_handle(stream, device):
    """The raw cudaStream_t of ``stream`` (a torch stream or an integer handle), or of torch's
    current stream on ``device`` (an index, a torch device, or None for the current one)."""
    import torch
    if stream is None:
        idx = device.index if isinstance(device, torch.device) else device
        if idx is None:
            idx = torch.cuda.current_device()
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(idx)                # the handle without building a Stream object
        stream = torch.cuda.current_stream(idx)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def per_token_quant(x, out_q, out_s, *, num_tokens: int | None = None, stream=None) -> None:
    """Per-token FP8 quantization of the first ``num_tokens`` rows of x [T, hidden]
    (bf16/fp16/fp32) into out_q (e4m3, may have more rows) and out_s (float32, one per row).
    Rows past num_tokens are not touched.  Follows ``ptgq_per_token_quant``."""
    import torch
    if not (x.is_cuda and x.is_contiguous() and out_q.is_contiguous() and out_s.is_contiguous()):
        raise ValueError("x, out_q, out_s must be contiguous CUDA tensors")
    dt = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}.get(x.dtype)
    if dt is None:
        raise TypeError(f"unsupported dtype {x.dtype}")
    T, hidden = x.shape
    n = T if num_tokens is None else num_tokens
    if not 0 <= n <= T:
        raise ValueError(f"num_tokens {n} outside [0, {T}]")
    if out_q.numel() * out_q.element_size() < n * hidden or out_s.numel() < n:
        raise ValueError("out_q must hold num_tokens * hidden codes and out_s num_tokens scales")
    rc = lib().ptgq_per_token_quant(x.data_ptr(), dt, n, hidden, out_q.data_ptr(),
                                    out_s.data_ptr(), _stream_handle(stream, x.device))
    if rc != 0:
        raise PtgqError(rc, "ptgq_per_token_quant")


def requant_per_tensor(x, x_scale, masked_m, output_scale, out, *, group_size: int = 128,
                       stream=None) -> None:
    """Per-token-group FP8 -> per-tensor FP8 requant of x [E, M, K] (e4m3 codes) with
    x_scale indexed [e, m, k // group_size] through its strides; rows below masked_m[e]
    only (all rows when masked_m is None); output_scale is a 1-element float32 device
    tensor.  Follows ``ptgq_requant_per_tensor``."""
    if not (x.is_cuda and x.is_contiguous() and out.is_contiguous()):
        raise ValueError("x and out must be contiguous CUDA tensors")
    E, M, K = x.shape
    se, sm, sg = x_scale.stride()
    if out.numel() * out.element_size() < E * M * K:
        raise ValueError("out must hold E * M * K codes")
    if E * M > 0 and group_size in (16, 32, 64, 128) and K % group_size == 0:
        reach = (E - 1) * se + (M - 1) * sm + (K // group_size - 1) * sg + 1
        avail = x_scale.untyped_storage().nbytes() // 4 - x_scale.storage_offset()
        if min(se, sm, sg) < 0 or reach > avail:
            raise ValueError("x_scale's strides reach past its storage")
    if masked_m is not None and masked_m.numel() < E:
        raise ValueError(f"masked_m has {masked_m.numel()} entries for {E} experts")
    if output_scale.numel() < 1:
        raise ValueError("output_scale must hold one float")
    rc = lib().ptgq_requant_per_tensor(
        x.data_ptr(), x_scale.data_ptr(), se, sm, sg,
        None if masked_m is None or E == 0 else masked_m.data_ptr(), output_scale.data_ptr(),
        out.data_ptr(), E, M, K, group_size, _stream_handle(stream, x.device))
    if rc != 0:
        raise PtgqError(rc, "ptgq_requant_per_tensor")
