"""Python binding of libgq: weight-only FP8 / NVFP4 linear layers on GB300.

    out = alpha * x @ dequant(W)^T      (bf16 activations, fp32 accumulation)

This module only marshals arguments: it checks torch tensors (device, dtype,
contiguity), takes their device pointers and the current CUDA stream, and
calls the C ABI declared in ``include/gq.h``.  Every step of the computation
runs in the library's CUDA kernels; there is no other code path.  If
``libgq.so`` has not been built, or the current device is not an sm_103 GPU,
the calls raise.

Entry points (same names as the C ABI without the ``gq_`` prefix):
``fp8_gemv``, ``nvfp4_gemv``, ``fp8_matmul``, ``nvfp4_matmul``,
``fp8_grouped_matmul``, ``nvfp4_grouped_matmul``, ``int8_quantize_rows``,
``int8_matmul``, ``fp8_materialize``, ``nvfp4_materialize``.  The
product calls take ``bias=`` and ``activation=`` for the fused epilogue
(``out = act(alpha * acc + bias)``); with either given they call the ``_ex``
form of the C entry point.  Outputs may be float32, bfloat16 or float16.
"""

from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgq.so")

GQ_F32, GQ_BF16, GQ_F16 = 0, 1, 2

ACTIVATIONS = {"none": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


class Epilogue(ctypes.Structure):
    """struct gq_epilogue."""
    _fields_ = [("bias", ctypes.c_void_p), ("bias_dtype", ctypes.c_int),
                ("activation", ctypes.c_int)]

# Names and argument types of every exported symbol (mirrors include/gq.h).
_P, _I, _I64, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
_E = ctypes.POINTER(Epilogue)
SIGNATURES = {
    "gq_status_str": (ctypes.c_char_p, [_I]),
    "gq_version": (ctypes.c_char_p, []),
    "gq_fp8_gemv": (_I, [_P, _I, _P, _P, _I64, _I64, _F, _P]),
    "gq_nvfp4_gemv": (_I, [_P, _I, _P, _P, _P, _I64, _I64, _F, _P]),
    "gq_fp8_matmul": (_I, [_P, _I, _P, _P, _I64, _I64, _I64, _F, _P]),
    "gq_nvfp4_matmul": (_I, [_P, _I, _P, _P, _P, _I64, _I64, _I64, _F, _P]),
    "gq_fp8_grouped_matmul": (_I, [_P, _I, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                   _I64, _I64, _P]),
    "gq_fp8_gemv_ex": (_I, [_P, _I, _P, _P, _I64, _I64, _F, _E, _P]),
    "gq_nvfp4_gemv_ex": (_I, [_P, _I, _P, _P, _P, _I64, _I64, _F, _E, _P]),
    "gq_fp8_matmul_ex": (_I, [_P, _I, _P, _P, _I64, _I64, _I64, _F, _E, _P]),
    "gq_nvfp4_matmul_ex": (_I, [_P, _I, _P, _P, _P, _I64, _I64, _I64, _F, _E, _P]),
    "gq_fp8_grouped_matmul_ex": (_I, [_P, _I, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                      _I64, _I64, _E, _P]),
    "gq_nvfp4_grouped_matmul": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                     _I64, _I64, _P]),
    "gq_nvfp4_grouped_matmul_ex": (_I, [_P, _I, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                        _I64, _I64, _I64, _E, _P]),
    "gq_int8_quantize_rows": (_I, [_P, _P, _P, _I64, _I64, _P]),
    "gq_int8_matmul": (_I, [_P, _I, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "gq_int8_matmul_ex": (_I, [_P, _I, _P, _P, _P, _P, _I64, _I64, _I64, _E, _P]),
    "gq_fp8_materialize": (_I, [_P, _I, _P, _I64, _I64, _P]),
    "gq_nvfp4_materialize": (_I, [_P, _I, _P, _P, _I64, _I64, _P]),
    "gq_device_status": (_I, [ctypes.POINTER(ctypes.c_uint32), _I]),
    "gq_set_launch_flags": (_I, [ctypes.c_uint32]),
    "gq_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "gq_probe_gemv_read_floor": (_I, [_I, _P, _P, _P, _I64, _I64, _P]),
    "gq_get_launch_flags": (ctypes.c_uint32, []),
}

GQ_LAUNCH_OVERLAP_WEIGHT_READS = 1
GQ_LAUNCH_TEST_STALL_PRODUCER = 2     # tests of the failure path only (include/gq.h)


class GQError(RuntimeError):
    """A libgq call returned a non-zero gq_status."""

    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_str(status)} (status {status})")
        self.status = status


_lib = None


def load_library(path: str | None = None):
    """Load libgq.so (once) and declare its signatures."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libgq.so not found at {p}: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_str(status: int) -> str:
    return load_library().gq_status_str(int(status)).decode()


def version() -> str:
    return load_library().gq_version().decode()


def _check(status: int, where: str):
    if status != 0:
        raise GQError(status, where)


def _current_device_index() -> int:
    return torch.cuda.current_device()


def _same_device(device: torch.device, name: str) -> None:
    """The library launches on the current CUDA device and dereferences every
    pointer there: a tensor or stream of another GPU is refused here, before
    any launch, instead of reaching the kernels as a foreign address."""
    cur = _current_device_index()
    if device.type != "cuda" or device.index != cur:
        raise ValueError(f"{name} is on {device} but the current device is cuda:{cur}; "
                         "call torch.cuda.set_device() first")


def _stream_handle(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    _same_device(torch.device(s.device), "stream")
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    _same_device(t.device, name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _out_code(dtype) -> int:
    if dtype == torch.float32:
        return GQ_F32
    if dtype == torch.bfloat16:
        return GQ_BF16
    if dtype == torch.float16:
        return GQ_F16
    raise TypeError("dtype must be torch.float32, torch.bfloat16 or torch.float16")


def _epilogue(bias, activation, shape):
    """A gq_epilogue for bias / activation, or None when neither is given."""
    if bias is None and activation in (None, "none"):
        return None
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    ep = Epilogue(None, GQ_F32, ACTIVATIONS[activation])
    if bias is not None:
        if tuple(bias.shape) != tuple(shape):
            raise ValueError(f"bias must have shape {tuple(shape)}")
        ep.bias = _dev(bias, "bias")
        ep.bias_dtype = _out_code(bias.dtype)
    return ep


def _ref(ep):
    return ctypes.byref(ep)


def _out(out, shape, dtype, device):
    if out is None:
        return torch.empty(shape, dtype=dtype, device=device)
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must have shape {tuple(shape)}")
    return out


def _u8(t, name, ndim):
    if t.dtype == torch.float8_e4m3fn:
        t = t.view(torch.uint8)
    return t, _dev(t, name, torch.uint8, ndim)


def fp8_gemv(x, w, alpha=1.0, out=None, out_dtype=torch.bfloat16, stream=None, bias=None,
             activation="none"):
    """y[N] = act(alpha * x[K] @ e4m3(w[N, K])^T + bias)."""
    w, wp = _u8(w, "w", 2)
    n, k = w.shape
    xp = _dev(x.reshape(-1), "x", torch.bfloat16, 1)
    if x.numel() != k:
        raise ValueError("x must have K elements")
    dtype = out.dtype if out is not None else out_dtype
    y = _out(out, (n,), dtype, w.device)
    ep = _epilogue(bias, activation, (n,))
    lib = load_library()
    if ep is None:
        st = lib.gq_fp8_gemv(_dev(y, "out"), _out_code(dtype), xp, wp, n, k, float(alpha),
                             _stream_handle(stream))
    else:
        st = lib.gq_fp8_gemv_ex(_dev(y, "out"), _out_code(dtype), xp, wp, n, k, float(alpha),
                                _ref(ep), _stream_handle(stream))
    _check(st, "fp8_gemv")
    return y


def nvfp4_gemv(x, q, bs, alpha=1.0, out=None, out_dtype=torch.bfloat16, stream=None, bias=None,
               activation="none"):
    """y[N] = act(alpha * x[K] @ (e2m1(q) * e4m3(bs))^T + bias);  q [N, K/2], bs [N, K/16]."""
    q, qp = _u8(q, "q", 2)
    bs, bp = _u8(bs, "bs", 2)
    n, half = q.shape
    k = 2 * half
    xp = _dev(x.reshape(-1), "x", torch.bfloat16, 1)
    if x.numel() != k or tuple(bs.shape) != (n, k // 16):
        raise ValueError("shapes must be x [K], q [N, K/2], bs [N, K/16]")
    dtype = out.dtype if out is not None else out_dtype
    y = _out(out, (n,), dtype, q.device)
    ep = _epilogue(bias, activation, (n,))
    lib = load_library()
    if ep is None:
        st = lib.gq_nvfp4_gemv(_dev(y, "out"), _out_code(dtype), xp, qp, bp, n, k, float(alpha),
                               _stream_handle(stream))
    else:
        st = lib.gq_nvfp4_gemv_ex(_dev(y, "out"), _out_code(dtype), xp, qp, bp, n, k,
                                  float(alpha), _ref(ep), _stream_handle(stream))
    _check(st, "nvfp4_gemv")
    return y


def fp8_matmul(a, w, alpha=1.0, out=None, out_dtype=torch.bfloat16, stream=None, bias=None,
               activation="none"):
    """c[M, N] = act(alpha * a[M, K] @ e4m3(w[N, K])^T + bias[N])."""
    w, wp = _u8(w, "w", 2)
    ap = _dev(a, "a", torch.bfloat16, 2)
    m, k = a.shape
    n = w.shape[0]
    if w.shape[1] != k:
        raise ValueError("a and w disagree on K")
    dtype = out.dtype if out is not None else out_dtype
    c = _out(out, (m, n), dtype, a.device)
    ep = _epilogue(bias, activation, (n,))
    lib = load_library()
    if ep is None:
        st = lib.gq_fp8_matmul(_dev(c, "out"), _out_code(dtype), ap, wp, m, n, k, float(alpha),
                               _stream_handle(stream))
    else:
        st = lib.gq_fp8_matmul_ex(_dev(c, "out"), _out_code(dtype), ap, wp, m, n, k, float(alpha),
                                  _ref(ep), _stream_handle(stream))
    _check(st, "fp8_matmul")
    return c


def nvfp4_matmul(a, q, bs, alpha=1.0, out=None, out_dtype=torch.bfloat16, stream=None, bias=None,
                 activation="none"):
    """c[M, N] = act(alpha * a[M, K] @ (e2m1(q) * e4m3(bs))^T + bias[N])."""
    q, qp = _u8(q, "q", 2)
    bs, bp = _u8(bs, "bs", 2)
    ap = _dev(a, "a", torch.bfloat16, 2)
    m, k = a.shape
    n = q.shape[0]
    if q.shape[1] * 2 != k or tuple(bs.shape) != (n, k // 16):
        raise ValueError("shapes must be a [M, K], q [N, K/2], bs [N, K/16]")
    dtype = out.dtype if out is not None else out_dtype
    c = _out(out, (m, n), dtype, a.device)
    ep = _epilogue(bias, activation, (n,))
    lib = load_library()
    if ep is None:
        st = lib.gq_nvfp4_matmul(_dev(c, "out"), _out_code(dtype), ap, qp, bp, m, n, k,
                                 float(alpha), _stream_handle(stream))
    else:
        st = lib.gq_nvfp4_matmul_ex(_dev(c, "out"), _out_code(dtype), ap, qp, bp, m, n, k,
                                    float(alpha), _ref(ep), _stream_handle(stream))
    _check(st, "nvfp4_matmul")
    return c


def fp8_grouped_matmul(a, w, a_offsets, expert_ids, expert_scales=None, max_rows_per_group=None,
                       out=None, out_dtype=torch.bfloat16, stream=None, bias=None,
                       activation="none"):
    """Grouped MoE product.  a [total_M, K] bf16, w [E, N, K] e4m3,
    a_offsets [G+1] uint32/int32 (device), expert_ids [G] int32 (device),
    expert_scales [E] float32 or None, bias [E, N] or None (fused epilogue
    per expert).  Rows no group covers are left as they are in `out`
    (allocate it yourself to control them)."""
    w, wp = _u8(w, "w", 3)
    ap = _dev(a, "a", torch.bfloat16, 2)
    total_m, k = a.shape
    e, n, kw = w.shape
    if kw != k:
        raise ValueError("a and w disagree on K")
    if a_offsets.dtype not in (torch.int32, torch.uint32):
        raise TypeError("a_offsets must be int32 or uint32")
    op = _dev(a_offsets, "a_offsets", None, 1)
    ip = _dev(expert_ids, "expert_ids", torch.int32, 1)
    g = expert_ids.numel()
    if a_offsets.numel() != g + 1:
        raise ValueError("a_offsets must have G + 1 entries")
    sp = None if expert_scales is None else _dev(expert_scales, "expert_scales", torch.float32, 1)
    if max_rows_per_group is None:
        max_rows_per_group = total_m
    dtype = out.dtype if out is not None else out_dtype
    c = _out(out, (total_m, n), dtype, a.device)
    ep = _epilogue(bias, activation, (e, n))
    lib = load_library()
    if ep is None:
        st = lib.gq_fp8_grouped_matmul(_dev(c, "out"), _out_code(dtype), ap, wp, op, ip, sp, g, e,
                                       int(max_rows_per_group), total_m, n, k,
                                       _stream_handle(stream))
    else:
        st = lib.gq_fp8_grouped_matmul_ex(_dev(c, "out"), _out_code(dtype), ap, wp, op, ip, sp, g,
                                          e, int(max_rows_per_group), total_m, n, k, _ref(ep),
                                          _stream_handle(stream))
    _check(st, "fp8_grouped_matmul")
    return c


def nvfp4_grouped_matmul(a, q, bs, a_offsets, expert_ids, expert_scales=None,
                         max_rows_per_group=None, out=None, out_dtype=torch.bfloat16, stream=None,
                         bias=None, activation="none"):
    """Grouped MoE product with NVFP4 experts.  a [total_M, K] bf16,
    q [E, N, K/2] uint8, bs [E, N, K/16] uint8 (e4m3 codes), a_offsets [G+1]
    uint32/int32 (device), expert_ids [G] int32 (device), expert_scales [E]
    float32 (the experts' second scales) or None, bias [E, N] or None."""
    q, qp = _u8(q, "q", 3)
    bs, bp = _u8(bs, "bs", 3)
    ap = _dev(a, "a", torch.bfloat16, 2)
    total_m, k = a.shape
    e, n, half = q.shape
    if half * 2 != k or tuple(bs.shape) != (e, n, k // 16):
        raise ValueError("shapes must be a [M, K], q [E, N, K/2], bs [E, N, K/16]")
    if a_offsets.dtype not in (torch.int32, torch.uint32):
        raise TypeError("a_offsets must be int32 or uint32")
    op = _dev(a_offsets, "a_offsets", None, 1)
    ip = _dev(expert_ids, "expert_ids", torch.int32, 1)
    g = expert_ids.numel()
    if a_offsets.numel() != g + 1:
        raise ValueError("a_offsets must have G + 1 entries")
    sp = None if expert_scales is None else _dev(expert_scales, "expert_scales", torch.float32, 1)
    if max_rows_per_group is None:
        max_rows_per_group = total_m
    dtype = out.dtype if out is not None else out_dtype
    c = _out(out, (total_m, n), dtype, a.device)
    ep = _epilogue(bias, activation, (e, n))
    lib = load_library()
    if ep is None:
        st = lib.gq_nvfp4_grouped_matmul(_dev(c, "out"), _out_code(dtype), ap, qp, bp, op, ip, sp,
                                         g, e, int(max_rows_per_group), total_m, n, k,
                                         _stream_handle(stream))
    else:
        st = lib.gq_nvfp4_grouped_matmul_ex(_dev(c, "out"), _out_code(dtype), ap, qp, bp, op, ip,
                                            sp, g, e, int(max_rows_per_group), total_m, n, k,
                                            _ref(ep), _stream_handle(stream))
    _check(st, "nvfp4_grouped_matmul")
    return c


def int8_quantize_rows(x, q=None, scale=None, stream=None):
    """W8A8 activation side: x [M, K] bf16 -> (q [M, K] int8, scale [M] float32),
    scale = absmax / 127 per row, q = round-half-even(x / scale)."""
    xp = _dev(x, "x", torch.bfloat16, 2)
    m, k = x.shape
    q = _out(q, (m, k), torch.int8, x.device)
    scale = _out(scale, (m,), torch.float32, x.device)
    st = load_library().gq_int8_quantize_rows(_dev(q, "q"), _dev(scale, "scale"), xp, m, k,
                                              _stream_handle(stream))
    _check(st, "int8_quantize_rows")
    return q, scale


def int8_matmul(a, b, a_scale, b_scale, out=None, out_dtype=torch.bfloat16, stream=None,
                bias=None, activation="none"):
    """W8A8 GEMM: c[M, N] = act((sum_k a[m,k] b[n,k]) * a_scale[m] * b_scale[n] + bias[n]);
    a [M, K] int8, b [N, K] int8, a_scale [M], b_scale [N] float32."""
    ap = _dev(a, "a", torch.int8, 2)
    bp = _dev(b, "b", torch.int8, 2)
    m, k = a.shape
    n = b.shape[0]
    if b.shape[1] != k:
        raise ValueError("a and b disagree on K")
    sap = _dev(a_scale, "a_scale", torch.float32, 1)
    sbp = _dev(b_scale, "b_scale", torch.float32, 1)
    if a_scale.numel() != m or b_scale.numel() != n:
        raise ValueError("a_scale must have M entries and b_scale N")
    dtype = out.dtype if out is not None else out_dtype
    c = _out(out, (m, n), dtype, a.device)
    ep = _epilogue(bias, activation, (n,))
    lib = load_library()
    if ep is None:
        st = lib.gq_int8_matmul(_dev(c, "out"), _out_code(dtype), ap, bp, sap, sbp, m, n, k,
                                _stream_handle(stream))
    else:
        st = lib.gq_int8_matmul_ex(_dev(c, "out"), _out_code(dtype), ap, bp, sap, sbp, m, n, k,
                                   _ref(ep), _stream_handle(stream))
    _check(st, "int8_matmul")
    return c


def fp8_materialize(w, out=None, out_dtype=torch.bfloat16, stream=None):
    """Dense e4m3(w) [N, K] as float32, bf16 or float16 (exact, unscaled)."""
    w, wp = _u8(w, "w", 2)
    n, k = w.shape
    dtype = out.dtype if out is not None else out_dtype
    o = _out(out, (n, k), dtype, w.device)
    _check(load_library().gq_fp8_materialize(_dev(o, "out"), _out_code(dtype), wp, n, k,
                                             _stream_handle(stream)), "fp8_materialize")
    return o


def nvfp4_materialize(q, bs, out=None, out_dtype=torch.bfloat16, stream=None):
    """Dense e2m1(q) * e4m3(bs) [N, K] as float32, bf16 or float16 (exact, unscaled)."""
    q, qp = _u8(q, "q", 2)
    bs, bp = _u8(bs, "bs", 2)
    n, half = q.shape
    k = 2 * half
    dtype = out.dtype if out is not None else out_dtype
    o = _out(out, (n, k), dtype, q.device)
    _check(load_library().gq_nvfp4_materialize(_dev(o, "out"), _out_code(dtype), qp, bp, n, k,
                                               _stream_handle(stream)), "nvfp4_materialize")
    return o


def set_launch_flags(flags: int) -> None:
    """Process-wide launch options; GQ_LAUNCH_OVERLAP_WEIGHT_READS lets a GEMV's
    weight reads overlap the previous kernel in the stream (see include/gq.h:
    only when that kernel does not write the weights)."""
    _check(load_library().gq_set_launch_flags(int(flags)), "set_launch_flags")


def get_launch_flags() -> int:
    return int(load_library().gq_get_launch_flags())


def probe_gemv_read_floor(w, bs=None, out=None, stream=None):
    """The GEMV launch shape with loads only (gq_probe_gemv_read_floor): FP8
    when bs is None (w [N, K] e4m3/uint8), else NVFP4 (w = q [N, K/2] uint8,
    bs [N, K/16]).  Returns the checksum vector [N] bf16 (not a product)."""
    w, wp = _u8(w, "w", 2)
    n = w.shape[0]
    if bs is None:
        fmt, k, bp = 0, w.shape[1], None
    else:
        bs, bp = _u8(bs, "bs", 2)
        fmt, k = 1, 2 * w.shape[1]
    y = _out(out, (n,), torch.bfloat16, w.device)
    _check(load_library().gq_probe_gemv_read_floor(fmt, _dev(y, "out"), wp, bp, n, k,
                                                   _stream_handle(stream)),
           "probe_gemv_read_floor")
    return y


def set_wait_limit_ns(ns: int) -> None:
    """Limit of the kernels' bounded waits on the current device (0 = the
    default 2 s); for tests of the failure path (synchronizes)."""
    _check(load_library().gq_set_wait_limit_ns(int(ns)), "set_wait_limit_ns")


def device_status(reset: bool = False) -> int:
    """Status flags recorded by bounded in-kernel waits that ran out (synchronizes)."""
    v = ctypes.c_uint32(0)
    _check(load_library().gq_device_status(ctypes.byref(v), 1 if reset else 0), "device_status")
    return int(v.value)


__all__ = [
    "fp8_gemv", "nvfp4_gemv", "fp8_matmul", "nvfp4_matmul", "fp8_grouped_matmul",
    "nvfp4_grouped_matmul", "int8_quantize_rows", "int8_matmul",
    "fp8_materialize", "nvfp4_materialize", "device_status", "load_library", "GQError",
    "set_launch_flags", "get_launch_flags", "GQ_LAUNCH_OVERLAP_WEIGHT_READS",
    "GQ_LAUNCH_TEST_STALL_PRODUCER", "set_wait_limit_ns", "probe_gemv_read_floor",
    "SIGNATURES", "LIB_PATH", "version", "status_str", "ACTIVATIONS", "Epilogue",
]
