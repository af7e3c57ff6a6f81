"""Python binding of libq8gemv, the GB300 Q8_0 block-quantized GEMV library.

Argument marshalling only: every step of the product runs in the library's CUDA kernels (device entry points) or its
C++ host code (repack, quantize).  PyTorch supplies device memory and streams.  The names follow the C ABI in
``include/q8_gemv.h``:

* :func:`gemv` -- ``q8_gemv`` / ``q8_gemv_ex``: y[r, n] = sum_b s[b, n] sum_i x[r, 32b+i] q[32b+i, n]
  ("from_q8.rs", module doc), bf16 x [m, K], int8 q [K, Np], fp32 s [K/32, Np] -> fp32 y [m, Np];
* :func:`gemv_argmax` -- ``q8_gemv_argmax``: the product and the first-maximum arg-max that ends a decode step;
* :func:`quantize_act` -- ``q8_quantize_act``: the quantized form of an activation (int8 values and an fp32 scale per
  32, "plan.rs" ``QBLOCK``); every product function takes the :class:`QuantAct` it returns in place of bf16 x
  (``Q8_FLAG_Q8_ACT``, tiled weights);
* :func:`repack` -- ``q8_repack``: 36-byte checkpoint blocks -> (q, s) on the host;
* :func:`quantize` -- ``q8_quantize``: the Q8_0 rule of "from_q8.rs" ``quantize`` on the host.

The library must have been built (``python -m q8_block_quantized_gemv_gb300.build``); there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB as _LIB_PATH

Q8_BLOCK = 32
MAX_ROWS = 16
MAX_CHUNK = 512  # rows one call over tiled weights takes
VARIANTS = {"auto": 0, "simt": 1, "mma": 2, "tma": 3}

_STATUS = {0: "Q8_OK", 1: "Q8_ERR_ARG", 2: "Q8_ERR_SHAPE", 3: "Q8_ERR_ALIGN", 4: "Q8_ERR_NOT_Q8_0", 5: "Q8_ERR_CUDA"}

# Every symbol include/q8_gemv.h declares, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
SIGNATURES = {
    "q8_padded_n": (_I, [_I]),
    "q8_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _P]),
    "q8_gemv_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_gemv_argmax": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "q8_gemv_argmax_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_tiled_n": (_I, [_I]),
    "q8_tile": (_I, [_P, _P, _I, _I, _P, _P]),
    "q8_tile_device": (_I, [_P, _P, _I, _I, _P, _P, _P]),
    "q8_repack": (_I, [_P, _I, _I, _P, _P]),
    "q8_quantize": (_I, [_P, _I, _I, _P, _P]),
    "q8_status_string": (ctypes.c_char_p, [_I]),
    "q8_last_cuda_error": (_I, []),
    "q8_version": (_I, []),
    "q8_device_fault": (_I, [_P, _I]),
    "q8_gemv_parts": (_I, [_P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_gemv_glu": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_gemv_residual_norm": (_I, [_P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_act_bytes": (ctypes.c_int64, [_I, _I]),
    "q8_repack_f16": (_I, [_P, _I, _I, _P, _P]),
    "q8_gemv_glu_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_gemv_residual_norm_ex": (_I, [_P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P, _I, _I, _I, ctypes.c_uint, _P]),
    "q8_quantize_act": (_I, [_P, _P, _I, _I, _P]),
    "q8_gemv_residual_norm_noalloc": (_I, [_P, _P, _P, _P, _P, ctypes.c_float, _P, _P, _I, _I, _I, ctypes.c_uint,
                                          _P]),
    "q8_plan_launches": (_I, [_I, _I, _P, _I, ctypes.c_uint]),
    "q8_plan_glu_launches": (_I, [_I, _I, _I, ctypes.c_uint]),
    "q8_set_tuning": (_I, [_I, _I]),
    "q8_get_tuning": (_I, [_I]),
}


class _Part(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("y", ctypes.c_void_p), ("N", ctypes.c_int)]

_lib = None


class Q8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = lib().q8_status_string(status).decode()
        if status == 5:
            detail += f" (cudaError {lib().q8_last_cuda_error()})"
        super().__init__(f"{where}: {_STATUS.get(status, status)}: {detail}")


def library_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises when it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libq8gemv is not built ({_LIB_PATH} missing); run "
                               "`python -m q8_block_quantized_gemv_gb300.build`")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status: int, where: str):
    if status != 0:
        raise Q8Error(status, where)


def padded_n(N: int) -> int:
    return lib().q8_padded_n(N)


def status_string(status: int) -> str:
    return lib().q8_status_string(status).decode()


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def tiled_n(N: int) -> int:
    return lib().q8_tiled_n(N)


class QuantAct:
    """The quantized form of an activation (q8_quantize_act): one uint8 CUDA buffer of ``act_bytes(m, K)`` bytes
    holding int8 values [m, K] followed by fp32 scales [m, K/32].  Pass it as ``x`` to any product function (tiled
    weights only)."""

    def __init__(self, buf, m: int, K: int):
        self.buf, self.shape = buf, (m, K)

    @property
    def device(self):
        return self.buf.device

    @property
    def is_cuda(self):
        return self.buf.is_cuda

    def data_ptr(self) -> int:
        return self.buf.data_ptr()

    def values(self):
        """int8 [m, K] view of the codes."""
        import torch
        m, K = self.shape
        return self.buf[: m * K].view(torch.int8).view(m, K)

    def scales(self):
        """fp32 [m, K/32] view of the scales."""
        import torch
        m, K = self.shape
        return self.buf[m * K:].view(torch.float32).view(m, K // Q8_BLOCK)


def act_bytes(m: int, K: int) -> int:
    return int(lib().q8_act_bytes(m, K))


def quantize_act(x, out: QuantAct | None = None, stream=None) -> QuantAct:
    """bf16 x [m, K] (CUDA, contiguous) -> its quantized form (q8_quantize_act)."""
    import torch
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D bfloat16 CUDA tensor")
    m, K = x.shape
    nbytes = act_bytes(m, K)
    if nbytes < 0:
        raise ValueError("K must be a positive multiple of 32")
    if out is None:
        out = QuantAct(torch.empty((nbytes,), dtype=torch.uint8, device=x.device), m, K)
    elif out.shape != (m, K) or out.buf.numel() != nbytes:
        raise ValueError("out must be a QuantAct of the same shape")
    _check(lib().q8_quantize_act(x.data_ptr(), out.data_ptr(), m, K, _stream_handle(stream)), "q8_quantize_act")
    return out


def _check_operands(x, q, s, N, tiled=False):
    import torch
    if isinstance(x, QuantAct):
        if not tiled:
            raise ValueError("a quantized activation takes tiled weights")
        if not (q.is_cuda and s.is_cuda and x.is_cuda):
            raise ValueError("x, q and s must be CUDA tensors")
        if q.dtype != torch.int8 or s.dtype != torch.float32 or not (q.is_contiguous() and s.is_contiguous()):
            raise TypeError("q must be contiguous int8 and s contiguous float32")
        m, K = x.shape
    else:
        if not (x.is_cuda and q.is_cuda and s.is_cuda):
            raise ValueError("x, q and s must be CUDA tensors")
        if x.dtype != torch.bfloat16 or q.dtype != torch.int8 or s.dtype != torch.float32:
            raise TypeError("x must be bfloat16, q int8 and s float32")
        if not (x.is_contiguous() and q.is_contiguous() and s.is_contiguous()):
            raise ValueError("x, q and s must be contiguous")
        if x.dim() != 2:
            raise ValueError("x must be 2-D [m, K]")
        m, K = x.shape
    Np = padded_n(N) if N > 0 else -1
    if tiled:
        Nt = tiled_n(N) if N > 0 else -1
        if q.numel() != K * Nt or s.numel() != (K // Q8_BLOCK) * Nt:
            raise ValueError(f"tiled q must hold K * Nt = {K * Nt} values and s (K/32) * Nt scales")
    elif q.shape != (K, Np) or s.shape != (K // Q8_BLOCK, Np):
        raise ValueError(f"q must be [K, Np] = [{K}, {Np}] and s [K/32, Np]; got {tuple(q.shape)}, {tuple(s.shape)}")
    return m, K, Np


FLAG_CONSTANT_WEIGHTS = 1
FLAG_TILED = 2
FLAG_Q8_ACT = 4


def _flags(constant_weights, tiled, x=None):
    return ((FLAG_CONSTANT_WEIGHTS if constant_weights else 0) | (FLAG_TILED if tiled else 0)
            | (FLAG_Q8_ACT if isinstance(x, QuantAct) else 0))


def gemv(x, q, s, N: int, y=None, variant: str = "auto", constant_weights: bool = False, tiled: bool = False,
         stream=None):
    """y = x . W over the Q8_0 weight (q, s); returns y, fp32 [m, Np] (columns N .. Np-1 are 0).

    constant_weights: nothing enqueued earlier on the stream writes q or s (Q8_FLAG_CONSTANT_WEIGHTS), so the
    kernel may stream them before the previous kernel finishes.  tiled: q and s are in the tiled layout
    (:func:`tile_device`, Q8_FLAG_TILED)."""
    import torch
    m, K, Np = _check_operands(x, q, s, N, tiled)
    if y is None:
        y = torch.empty((m, Np), dtype=torch.float32, device=x.device)
    elif y.dtype != torch.float32 or y.shape != (m, Np) or not y.is_contiguous() or not y.is_cuda:
        raise ValueError("y must be a contiguous fp32 CUDA tensor [m, Np]")
    _check(lib().q8_gemv_ex(x.data_ptr(), q.data_ptr(), s.data_ptr(), y.data_ptr(), m, K, N, VARIANTS[variant],
                            _flags(constant_weights, tiled, x), _stream_handle(stream)), "q8_gemv")
    return y


def gemv_argmax(x, q, s, N: int, idx=None, logits=None, constant_weights: bool = False, tiled: bool = False,
                stream=None):
    """The product and its first-maximum arg-max per row: returns idx, int64 [m] (0-based).

    ``logits``: None (not stored) or a contiguous fp32 [m, Np] CUDA tensor that receives y.
    """
    import torch
    m, K, Np = _check_operands(x, q, s, N, tiled)
    if idx is None:
        idx = torch.empty((m,), dtype=torch.int64, device=x.device)
    elif idx.dtype != torch.int64 or idx.numel() < m or not idx.is_contiguous() or not idx.is_cuda:
        raise ValueError("idx must be a contiguous int64 CUDA tensor of m elements")
    lp = None
    if logits is not None:
        if logits.dtype != torch.float32 or logits.shape != (m, Np) or not logits.is_contiguous():
            raise ValueError("logits must be a contiguous fp32 CUDA tensor [m, Np]")
        lp = logits.data_ptr()
    _check(lib().q8_gemv_argmax_ex(x.data_ptr(), q.data_ptr(), s.data_ptr(), idx.data_ptr(), lp, m, K, N,
                                   _flags(constant_weights, tiled, x), _stream_handle(stream)), "q8_gemv_argmax")
    return idx


def tile(q, s, N: int):
    """Host: row-major (q [K, Np], s [K/32, Np]) numpy arrays -> the tiled layout (qt int8 [K * Nt], st fp32
    [K/32 * Nt]) (q8_tile)."""
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    K = q.shape[0]
    Nt = tiled_n(N) if N > 0 else 1
    qt = np.empty(max(K * Nt, 1), dtype=np.int8)
    st = np.empty(max((K // Q8_BLOCK) * Nt, 1), dtype=np.float32)
    _check(lib().q8_tile(q.ctypes.data, s.ctypes.data, K, N, qt.ctypes.data, st.ctypes.data), "q8_tile")
    return qt, st


def tile_device(q, s, N: int, stream=None):
    """Device: row-major CUDA tensors (q [K, Np] int8, s [K/32, Np] fp32) -> tiled CUDA tensors (q8_tile_device)."""
    import torch
    K = q.shape[0]
    Nt = tiled_n(N)
    qt = torch.empty((K * Nt,), dtype=torch.int8, device=q.device)
    st = torch.empty(((K // Q8_BLOCK) * Nt,), dtype=torch.float32, device=q.device)
    _check(lib().q8_tile_device(q.data_ptr(), s.data_ptr(), K, N, qt.data_ptr(), st.data_ptr(),
                                _stream_handle(stream)), "q8_tile_device")
    return qt, st


def gemv_parts(x, weights, ys=None, constant_weights: bool = False, tiled: bool = False, stream=None):
    """Several products of one activation in one call (q8_gemv_parts): weights is a list of (q, s, N); returns the
    list of outputs y_p, fp32 [m, Np_p]."""
    import torch
    if not weights or len(weights) > 8:
        raise ValueError("1 to 8 parts")
    m, K = x.shape
    arr = (_Part * len(weights))()
    outs = []
    for i, (q, s, N) in enumerate(weights):
        _check_operands(x, q, s, N, tiled)
        Np = padded_n(N)
        y = ys[i] if ys is not None else torch.empty((m, Np), dtype=torch.float32, device=x.device)
        if y.dtype != torch.float32 or y.shape != (m, Np) or not y.is_contiguous() or not y.is_cuda:
            raise ValueError("each y must be a contiguous fp32 CUDA tensor [m, Np]")
        arr[i] = _Part(q.data_ptr(), s.data_ptr(), y.data_ptr(), N)
        outs.append(y)
    _check(lib().q8_gemv_parts(x.data_ptr(), ctypes.cast(arr, ctypes.c_void_p), len(weights), m, K,
                               _flags(constant_weights, tiled, x), _stream_handle(stream)), "q8_gemv_parts")
    return outs


def plan_launches(m: int, K: int, Ns, tiled: bool = True, q8_act: bool = False) -> int:
    """How many product kernels a gemv / gemv_argmax / gemv_parts call of these sizes launches on the current device
    (q8_plan_launches): 1, or 2 when the planner splits it in two."""
    arr = (ctypes.c_int * len(Ns))(*[int(n) for n in Ns])
    flags = (FLAG_TILED if tiled else 0) | (FLAG_Q8_ACT if q8_act else 0)
    n = int(lib().q8_plan_launches(int(m), int(K), ctypes.cast(arr, ctypes.c_void_p), len(Ns), flags))
    if n < 0:
        raise Q8Error(-n, "q8_plan_launches")
    return n


def plan_glu_launches(m: int, K: int, N: int, q8_act: bool = False) -> int:
    """How many kernels a gemv_glu call of these sizes launches on the current device (q8_plan_glu_launches)."""
    n = int(lib().q8_plan_glu_launches(int(m), int(K), int(N), FLAG_TILED | (FLAG_Q8_ACT if q8_act else 0)))
    if n < 0:
        raise Q8Error(-n, "q8_plan_glu_launches")
    return n


def _q8_out(out_q8, m, Np, device):
    import torch
    if out_q8 is None:
        return QuantAct(torch.empty((act_bytes(m, Np),), dtype=torch.uint8, device=device), m, Np)
    if out_q8.shape != (m, Np) or out_q8.buf.numel() != act_bytes(m, Np):
        raise ValueError("out_q8 must be a QuantAct of [m, Np]")
    return out_q8


def gemv_glu(x, gate, up, N: int, out=None, out_bf16=None, want=("f32",), constant_weights: bool = False,
             stream=None, out_q8=None):
    """The gated pair (q8_gemv_glu_ex, SwiGLU): silu(x.Wg) * (x.Wu) with both weights tiled; gate and up are (q, s).

    ``want``: which outputs to allocate when not given -- "f32" (fp32 [m, Np]), "bf16" (bf16 [m, Np]) and/or "q8"
    (the quantized form of the bf16 output, a QuantAct of [m, Np]).  Returns (out, out_bf16), either None when not
    requested, or (out, out_bf16, out_q8) when "q8" is wanted or out_q8 given."""
    import torch
    m, K, Np = _check_operands(x, gate[0], gate[1], N, True)
    _check_operands(x, up[0], up[1], N, True)
    if out is None and "f32" in want:
        out = torch.empty((m, Np), dtype=torch.float32, device=x.device)
    if out_bf16 is None and "bf16" in want:
        out_bf16 = torch.empty((m, Np), dtype=torch.bfloat16, device=x.device)
    q8out = out_q8 is not None or "q8" in want
    if q8out:
        out_q8 = _q8_out(out_q8, m, Np, x.device)
    if out is not None and (out.dtype != torch.float32 or out.shape != (m, Np) or not out.is_contiguous()):
        raise ValueError("out must be a contiguous fp32 CUDA tensor [m, Np]")
    if out_bf16 is not None and (out_bf16.dtype != torch.bfloat16 or out_bf16.shape != (m, Np)
                                 or not out_bf16.is_contiguous()):
        raise ValueError("out_bf16 must be a contiguous bf16 CUDA tensor [m, Np]")
    _check(lib().q8_gemv_glu_ex(x.data_ptr(), gate[0].data_ptr(), gate[1].data_ptr(), up[0].data_ptr(),
                                up[1].data_ptr(), out.data_ptr() if out is not None else None,
                                out_bf16.data_ptr() if out_bf16 is not None else None,
                                out_q8.data_ptr() if q8out else None, m, K, N,
                                _flags(constant_weights, True, x), _stream_handle(stream)), "q8_gemv_glu")
    return (out, out_bf16, out_q8) if q8out else (out, out_bf16)


def gemv_residual_norm(x, q, s, N: int, residual, gamma, eps: float, h=None, out_bf16=None,
                       constant_weights: bool = False, stream=None, want=("bf16",), out_q8=None):
    """A projection followed by the residual add and the following RMS norm (q8_gemv_residual_norm_ex), tiled weight:
    h = residual + x.W, out = h / sqrt(mean(h^2) + eps) * gamma.  Returns (h fp32 [m, Np], out bf16 [m, Np]), or
    (h, out_bf16 or None, out_q8) when ``want`` holds "q8" or out_q8 is given (the quantized form of the bf16 rows);
    ``h`` may be ``residual`` (in place)."""
    import torch
    m, K, Np = _check_operands(x, q, s, N, True)
    if residual.dtype != torch.float32 or residual.shape != (m, Np) or not residual.is_contiguous():
        raise ValueError("residual must be a contiguous fp32 CUDA tensor [m, Np]")
    if gamma.dtype != torch.float32 or gamma.numel() < N or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous fp32 CUDA tensor of at least N values")
    if h is None:
        h = torch.empty((m, Np), dtype=torch.float32, device=x.device)
    if out_bf16 is None and "bf16" in want:
        out_bf16 = torch.empty((m, Np), dtype=torch.bfloat16, device=x.device)
    q8out = out_q8 is not None or "q8" in want
    if q8out:
        out_q8 = _q8_out(out_q8, m, Np, x.device)
    _check(lib().q8_gemv_residual_norm_ex(x.data_ptr(), q.data_ptr(), s.data_ptr(), residual.data_ptr(),
                                          gamma.data_ptr(), float(eps), h.data_ptr(),
                                          out_bf16.data_ptr() if out_bf16 is not None else None,
                                          out_q8.data_ptr() if q8out else None, m, K, N,
                                          _flags(constant_weights, True, x), _stream_handle(stream)),
           "q8_gemv_residual_norm")
    return (h, out_bf16, out_q8) if q8out else (h, out_bf16)


# Planner overrides (q8_set_tuning): the K split (0 = the planner's, 1..8 forced), the prefill GEMM (-1 = the
# planner's, 0 = row groups, 1 = GEMM), the residual norm's route (0 = own launch, 1 = the one-launch fold) and the
# two-launch split of plain products (1 = where the planner finds one, 0 = never).
TUNING = {"ksplit": 0, "gemm": 1, "norm_fold": 2, "split": 3}


def set_tuning(option: str, value: int) -> None:
    """Set a process-wide planner override (q8_set_tuning) for tests and benchmarks."""
    _check(lib().q8_set_tuning(TUNING[option], int(value)), "q8_set_tuning")


def get_tuning(option: str) -> int:
    """The current value of a planner override (q8_get_tuning)."""
    return int(lib().q8_get_tuning(TUNING[option]))


class tuning:
    """Context manager: ``with tuning(ksplit=4): ...`` sets overrides and restores the previous values on exit."""

    def __init__(self, **overrides):
        self.overrides, self.saved = overrides, {}

    def __enter__(self):
        for k, v in self.overrides.items():
            self.saved.setdefault(k, get_tuning(k))
            set_tuning(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            set_tuning(k, v)


def gemv_residual_norm_noalloc(x, q, s, N: int, residual, gamma, eps: float, h, out_bf16,
                               constant_weights: bool = False, stream=None):
    """q8_gemv_residual_norm_noalloc: the residual add and RMS norm as one launch whose scratch is the library's own
    static counters (no device allocation by anyone).  h and out_bf16 must be given (h may be ``residual``); calls
    that overlap on the GPU race on the shared counters.  Returns (h, out_bf16)."""
    import torch
    m, K, Np = _check_operands(x, q, s, N, True)
    if residual.dtype != torch.float32 or residual.shape != (m, Np) or not residual.is_contiguous():
        raise ValueError("residual must be a contiguous fp32 CUDA tensor [m, Np]")
    if gamma.dtype != torch.float32 or gamma.numel() < N or not gamma.is_contiguous():
        raise ValueError("gamma must be a contiguous fp32 CUDA tensor of at least N values")
    if h.dtype != torch.float32 or h.shape != (m, Np) or not h.is_contiguous():
        raise ValueError("h must be a contiguous fp32 CUDA tensor [m, Np]")
    if out_bf16.dtype != torch.bfloat16 or out_bf16.shape != (m, Np) or not out_bf16.is_contiguous():
        raise ValueError("out_bf16 must be a contiguous bf16 CUDA tensor [m, Np]")
    _check(lib().q8_gemv_residual_norm_noalloc(x.data_ptr(), q.data_ptr(), s.data_ptr(), residual.data_ptr(),
                                               gamma.data_ptr(), float(eps), h.data_ptr(), out_bf16.data_ptr(), m, K,
                                               N, _flags(constant_weights, True, x), _stream_handle(stream)),
           "q8_gemv_residual_norm_noalloc")
    return h, out_bf16


def residual_norm_launches() -> int:
    """Kernel launches one gemv_residual_norm call makes, by the library's current rule: the product, then the norm as
    a launch of its own (2); 1 when the one-launch fold is selected (tuning ``norm_fold`` = 1)."""
    return 1 if get_tuning("norm_fold") == 1 else 2


def device_fault(clear: bool = False) -> int:
    """The device fault word (nonzero when a kernel's bounded pipeline wait ran out); see q8_device_fault."""
    word = ctypes.c_uint(0)
    _check(lib().q8_device_fault(ctypes.byref(word), int(clear)), "q8_device_fault")
    return word.value


def repack(blocks, K: int, N: int, scale: str = "f32"):
    """(q int8 [K, Np], s fp32 [K/32, Np]) from N * K/32 checkpoint blocks (host): 36-byte blocks with an fp32 scale
    (q8_repack), or with scale="f16" GGML-style 34-byte blocks with a binary16 scale (q8_repack_f16)."""
    size = {"f32": 36, "f16": 34}[scale]
    raw = np.frombuffer(bytes(blocks), dtype=np.uint8) if not isinstance(blocks, np.ndarray) else \
        np.ascontiguousarray(blocks).view(np.uint8).reshape(-1)
    Np = padded_n(N) if N > 0 else 1
    nb = max(K // Q8_BLOCK, 1)
    if K > 0 and N > 0 and raw.size != N * nb * size:
        raise ValueError("block buffer size does not match K and N")
    q = np.empty((max(K, 1), Np), dtype=np.int8)
    s = np.empty((nb, Np), dtype=np.float32)
    fn = lib().q8_repack if scale == "f32" else lib().q8_repack_f16
    name = "q8_repack" if scale == "f32" else "q8_repack_f16"
    _check(fn(raw.ctypes.data, K, N, q.ctypes.data, s.ctypes.data), name)
    return q, s


def quantize(w):
    """(q int8 [K, Np], s fp32 [K/32, Np]) for a declared fp64 weight [K, N] (host); raises Q8Error if not Q8_0."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    K, N = w.shape
    Np = padded_n(N) if N > 0 else 1
    q = np.empty((max(K, 1), Np), dtype=np.int8)
    s = np.empty((max(K // Q8_BLOCK, 1), Np), dtype=np.float32)
    _check(lib().q8_quantize(w.ctypes.data, K, N, q.ctypes.data, s.ctypes.data), "q8_quantize")
    return q, s
