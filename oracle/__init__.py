"""Q8_0 product oracle -- TEST INFRASTRUCTURE ONLY.

Plain, slow CPU statements of what the Q8_0 path computes, used to check the CUDA library and nothing else. Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg import this package; the library never
does, and this package imports nothing from the library (they share only the seeded input generator in
``synth_inputs.py``, which holds none of the method's arithmetic).

Contents, each citing the passage it follows (page titles as printed on the pages):

* :func:`gemv` -- ``from_q8.rs`` module doc and ``q8_fold``: y[r,n] = sum_b s[b,n] * sum_i x[r,32b+i] q[32b+i,n],
  done in fp64 by the C file ``q8_oracle.c`` (plain loops, the formula's order), with the error scale
  A[r,n] = sum_b |s[b,n]| sum_i |x q|.
* :func:`argmax` -- ``int8_model.rs`` ``decode_step_lg`` (the lowest index among the largest logits) and the tie
  rule of its CUDA warp arg-max in ``reference_cuda`` (equal values go to the lower index); 0-based here.
* :func:`quantize` -- ``from_q8.rs`` ``quantize``: the Q8_0 rule and its rejections.
* :func:`repack` -- ``from_q8.rs`` ``Q8Part`` (on the host, the checkpoint's blocks become the int8 values and the fp32
  scales); the block layout is the reading stated in the design notes (36-byte blocks, fp32 scale first).
* :func:`repack_f16` -- the same repack from GGML-style blocks (``plan.rs`` names the checkpoint format
  ``GgmlType::Q8_0``): 34-byte blocks, an IEEE binary16 scale then 32 int8 values.
* :func:`dequantize` -- ``from_q8.rs`` module doc, w = q * d.
* :func:`residual_norm` -- ``plan.rs`` ``Launch::Fold`` of a projection with ``Launch::Norm`` (``gemv_norm_epilogue``:
  a projection whose epilogue adds the residual and applies the following norm; the norm launch is the lane's
  "rmsnorm"):
  h = residual + x.W, out = h / sqrt(mean_n h^2 + eps) * gamma, in fp64.
* :func:`quantize_act` -- ``plan.rs`` ``QBLOCK`` / ``Buffer::quantized`` and the quantized numerics of
  ``Launch::projected_input`` (an activation a projection reads quantized: int8 values and one scale per 32 values),
  with the weight rule's shape (``from_q8.rs`` ``quantize``: d = amax / 127, q = round(x / d)) taken in fp32.
* :func:`gemv_q8act` -- the product under those numerics: y[r,n] = sum_b s[b,n] d[r,b] sum_i xq[r,32b+i] q[32b+i,n],
  the inner sums exact integers, the rest in fp64, with its error scale.
* :func:`glu` -- ``plan.rs`` ``Launch::GemvGlu``: two projections of one activation through a gate,
  out = act(x.wg + bg) * (x.wu + bu), silu gating (SwiGLU) by default; here without biases, so
  out = silu(g) * u with g = x.Wg, u = x.Wu (each as :func:`gemv`) and silu(g) = g / (1 + exp(-g)), in fp64.

Every function here is pinned by ``tests/test_oracle_pins.py`` to facts the pages and the mathematics fix (brute
force in exact rational arithmetic, closed forms, a dense fp64 matmul of the dequantized weight, the quantize
round trip and hand-derived fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import numpy as np

Q8_BLOCK = 32  # rows of a Q8_0 block (from_q8.rs, ``Q8_BLOCK``)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_q8.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``q8_oracle.c`` with gcc (fp64, no fast-math, OpenMP over output columns)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_q8_gemv.restype = ctypes.c_int
        lib.oracle_q8_gemv.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_void_p]
        lib.oracle_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    """Threads the oracle's OpenMP loop uses."""
    return int(_load().oracle_threads())


def padded_n(n: int) -> int:
    """Columns padded to whole 32-column tiles (from_q8.rs ``q8_gemv_applies``: the last tile is zero-padded)."""
    return -(-n // Q8_BLOCK) * Q8_BLOCK


def gemv(x_bits: np.ndarray, q: np.ndarray, s: np.ndarray, cols=None):
    """fp64 Q8_0 product and its error scale.

    x_bits: uint16 bf16 patterns [m, K]; q: int8 [K, Np]; s: float32 [K/32, Np]; cols: optional column indices.
    Returns (y, A), fp64 [m, len(cols) or Np].
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    m, K = x_bits.shape
    K2, Np = q.shape
    if K2 != K or s.shape != (K // Q8_BLOCK, Np):
        raise ValueError("shape mismatch")
    if cols is None:
        ncols, cols_arr, cols_ptr = Np, None, None
    else:
        cols_arr = np.ascontiguousarray(cols, dtype=np.int64)
        if cols_arr.size and (cols_arr.min() < 0 or cols_arr.max() >= Np):
            raise ValueError("column out of range")
        ncols, cols_ptr = cols_arr.size, cols_arr.ctypes.data
    y = np.empty((m, ncols), dtype=np.float64)
    a = np.empty((m, ncols), dtype=np.float64)
    rc = _load().oracle_q8_gemv(x_bits.ctypes.data, q.ctypes.data, s.ctypes.data, m, K, Np, cols_ptr, ncols,
                                y.ctypes.data, a.ctypes.data)
    if rc != 0:
        raise ValueError("shape the Q8_0 product does not take")
    return y, a


def argmax(y: np.ndarray, n: int) -> np.ndarray:
    """Per row, the smallest index j < n with y[r, j] equal to the row's maximum over j < n (0-based).

    Pad columns (j >= n) never take part.  +0.0 and -0.0 compare equal.  A NaN logit (of either sign) ranks above
    every number, +inf included, so a row holding NaN gives its first NaN: the pages' logits are never NaN, and this
    is the reading that extends their first-maximum rule to a total order.
    """
    y = np.asarray(y, dtype=np.float64)
    out = np.empty(y.shape[0], dtype=np.int64)
    for r in range(y.shape[0]):
        row = y[r, :n]
        nan = np.flatnonzero(np.isnan(row))
        if nan.size:
            out[r] = int(nan[0])
            continue
        best = row.max()
        out[r] = int(np.flatnonzero(row == best)[0])
    return out


def _round_half_away(v: np.ndarray) -> np.ndarray:
    return np.where(v >= 0, np.floor(v + 0.5), -np.floor(-v + 0.5))


def quantize(w: np.ndarray):
    """Q8_0 values and scales of a declared weight, or None when the weight is not Q8_0 (from_q8.rs ``quantize``).

    For every 32-row block b and column: amax = max |w|; a zero block keeps q = 0 and d = 0; otherwise
    d = amax / 127 must survive a round trip through fp32, and every value w / d must lie within 1e-9 of an integer
    r with |r| <= 127 and r * d == w exactly.  w: float64 [K, N].  Returns (q int8 [K, N], s float32 [K/32, N]).
    """
    w = np.asarray(w, dtype=np.float64)
    K, N = w.shape
    if K % Q8_BLOCK != 0:
        return None
    q = np.zeros((K, N), dtype=np.int8)
    s = np.zeros((K // Q8_BLOCK, N), dtype=np.float32)
    for b in range(K // Q8_BLOCK):
        blk = w[Q8_BLOCK * b:Q8_BLOCK * (b + 1), :]            # [32, N]
        amax = np.abs(blk).max(axis=0)                          # [N]
        live = amax != 0.0                                       # zero blocks are skipped
        d = amax / 127.0
        if np.any(live & (d.astype(np.float32).astype(np.float64) != d)):
            return None
        with np.errstate(divide="ignore", invalid="ignore"):
            v = blk / np.where(live, d, 1.0)[None, :]
        r = _round_half_away(v)
        bad = (np.abs(v - r) > 1e-9) | (np.abs(r) > 127.0) | (r * d[None, :] != blk)
        if np.any(bad & live[None, :]):
            return None
        q[Q8_BLOCK * b:Q8_BLOCK * (b + 1), :] = np.where(live[None, :], r, 0).astype(np.int8)
        s[b, :] = np.where(live, d, 0.0).astype(np.float32)
    return q, s


def dequantize(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """w[k, n] = q[k, n] * s[k // 32, n] in fp64 (exact: 8-bit by 24-bit significands)."""
    q = np.asarray(q)
    s = np.asarray(s, dtype=np.float64)
    return q.astype(np.float64) * np.repeat(s, Q8_BLOCK, axis=0)


def repack(blocks: bytes | np.ndarray, K: int, N: int):
    """The int8 values [K, Np] and fp32 scales [K/32, Np] from checkpoint blocks (from_q8.rs ``Q8Part``).

    The blocks are column-major by block: column n's K/32 blocks one after another, each 36 bytes, a little-endian
    fp32 scale d followed by 32 int8 values.  Pad columns come out zero.  Returns None when a value is -128 (outside
    the Q8_0 range |q| <= 127) or a scale is not finite.
    """
    if K <= 0 or K % Q8_BLOCK or N <= 0:
        return None
    nb = K // Q8_BLOCK
    raw = np.frombuffer(bytes(blocks), dtype=np.uint8)
    if raw.size != N * nb * 36:
        raise ValueError("block buffer size does not match K and N")
    rec = raw.reshape(N, nb, 36)
    d = rec[:, :, 0:4].copy().view("<f4").reshape(N, nb)
    vals = rec[:, :, 4:36].copy().view(np.int8).reshape(N, nb, Q8_BLOCK)
    if np.any(vals == -128) or not np.all(np.isfinite(d)):
        return None
    Np = padded_n(N)
    q = np.zeros((K, Np), dtype=np.int8)
    s = np.zeros((nb, Np), dtype=np.float32)
    q[:, :N] = vals.reshape(N, K).T      # column n's blocks b = 0, 1, ... are its rows 32b .. 32b + 31
    s[:, :N] = d.T
    return q, s


def repack_f16(blocks: bytes | np.ndarray, K: int, N: int):
    """The int8 values [K, Np] and fp32 scales [K/32, Np] from GGML-style checkpoint blocks (``plan.rs``
    ``GgmlType::Q8_0``; ``from_q8.rs`` ``Q8Part``).

    The blocks are column-major by block as :func:`repack` reads them, each 34 bytes: a little-endian IEEE binary16
    scale d (widened to fp32 exactly: every binary16 value is a binary32 value) followed by 32 int8 values.  Pad
    columns come out zero.  Returns None when a value is -128 or a scale is not finite."""
    if K <= 0 or K % Q8_BLOCK or N <= 0:
        return None
    nb = K // Q8_BLOCK
    raw = np.frombuffer(bytes(blocks), dtype=np.uint8)
    if raw.size != N * nb * 34:
        raise ValueError("block buffer size does not match K and N")
    rec = raw.reshape(N, nb, 34)
    d = rec[:, :, 0:2].copy().view("<f2").reshape(N, nb).astype(np.float32)
    vals = rec[:, :, 2:34].copy().view(np.int8).reshape(N, nb, Q8_BLOCK)
    if np.any(vals == -128) or not np.all(np.isfinite(d)):
        return None
    Np = padded_n(N)
    q = np.zeros((K, Np), dtype=np.int8)
    s = np.zeros((nb, Np), dtype=np.float32)
    q[:, :N] = vals.reshape(N, K).T
    s[:, :N] = d.T
    return q, s


def silu(g: np.ndarray) -> np.ndarray:
    """The SiLU of SwiGLU (``plan.rs`` ``Launch::GemvGlu``): g * sigmoid(g) = g / (1 + exp(-g)), in fp64; exp(-g)
    overflows to inf for g below about -709, giving -0 or +0 as the limit does."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        return g / (1.0 + np.exp(-g))


def _product(x_bits, q, s, cols=None, act=None):
    """:func:`gemv` of bf16 x, or :func:`gemv_q8act` of the quantized activation ``act`` = (xq, xd) when given."""
    return gemv(x_bits, q, s, cols) if act is None else gemv_q8act(act[0], act[1], q, s, cols)


def glu(x_bits: np.ndarray, qg: np.ndarray, sg: np.ndarray, qu: np.ndarray, su: np.ndarray, cols=None, act=None):
    """The gated pair of ``plan.rs`` ``Launch::GemvGlu`` (SwiGLU, no biases): out = silu(x.Wg) * (x.Wu), fp64.

    Returns (out, g, u, a_g, a_u): the two products and their error scales as :func:`gemv` returns them, for the
    bound a GPU result is judged by.  ``act`` = (xq, xd): the products of the quantized activation instead
    (:func:`gemv_q8act`; x_bits is then unused)."""
    g, a_g = _product(x_bits, qg, sg, cols, act)
    u, a_u = _product(x_bits, qu, su, cols, act)
    return silu(g) * u, g, u, a_g, a_u


def rmsnorm(h: np.ndarray, gamma: np.ndarray, eps: float, N: int) -> np.ndarray:
    """RMS norm of each row's first N values (the lane's "rmsnorm", ``plan.rs`` ``Launch::Norm``):
    h / sqrt(mean(h^2) + eps) * gamma, fp64; columns >= N are 0."""
    h = np.asarray(h, dtype=np.float64)
    ms = np.mean(h[:, :N] ** 2, axis=1, keepdims=True)
    out = np.zeros_like(h)
    out[:, :N] = h[:, :N] / np.sqrt(ms + float(eps)) * np.asarray(gamma, dtype=np.float64)[:N]
    return out


def rmsnorm_bound(h: np.ndarray, out: np.ndarray, tol_h: np.ndarray, gamma: np.ndarray, eps: float,
                  N: int) -> np.ndarray:
    """How far a bf16 RMS-normed row computed in fp32 may lie from :func:`rmsnorm` of the exact h, per output.

    h, out: the exact (fp64) h and normed row; tol_h: the bound on each computed h.  Terms:
    * half a bf16 unit: rounding to 8 significant bits moves a value by at most 2^-8 of itself;
    * the h error carried through the norm: out_n = g_n h_n r with r = (mean h^2 + eps)^-1/2, so
      |d out_n| <= |g_n| r (|d h_n| + |h_n| sum_k |h_k| |d h_k| / (N (mean h^2 + eps)));
    * the fp32 arithmetic, in units u = 2^-24: the sum of squares of N values by a tree whose deepest path has
      D = 4 ceil(Np / 512) + 12 additions (four products a 16-byte chunk, the chunks of one of at least 128 threads
      in order, five shuffle levels, at most eight warps in order) is within D u of itself; the mean, + eps, the
      square root and the reciprocal add u, u, u/2 + half the sum's error, and u; the two multiplies 2u; with the
      bf16 rounding taken on the computed value, D/2 + 7 units in all."""
    h = np.asarray(h, dtype=np.float64)
    tol_h = np.asarray(tol_h, dtype=np.float64)
    g = np.abs(np.asarray(gamma, dtype=np.float64)[:N])
    Np = h.shape[1]
    ms = np.mean(h[:, :N] ** 2, axis=1, keepdims=True) + float(eps)
    r = 1.0 / np.sqrt(ms)
    carried = np.zeros_like(h)
    carried[:, :N] = g[None, :] * r * (tol_h[:, :N] + np.abs(h[:, :N]) *
                                       np.sum(np.abs(h[:, :N]) * tol_h[:, :N], axis=1, keepdims=True) / (N * ms))
    depth = 4 * -(-Np // 512) + 12
    return 2.0 ** -8 * np.abs(out) + (1.0 + 2.0 ** -8) * carried + (depth / 2 + 7) * 2.0 ** -24 * np.abs(out)


def residual_norm(x_bits: np.ndarray, q: np.ndarray, s: np.ndarray, residual: np.ndarray, gamma: np.ndarray,
                  eps: float, N: int, act=None):
    """A projection followed by the residual add and the following norm (``plan.rs`` ``Launch::Fold`` /
    ``gemv_norm_epilogue``): h = residual + x.W (each output as :func:`gemv`), out = rmsnorm(h) * gamma.

    Returns (h, out, y, a): the new residual stream, the normed activation, the product and its error scale.
    ``act`` = (xq, xd): the product of the quantized activation instead (:func:`gemv_q8act`)."""
    y, a = _product(x_bits, q, s, None, act)
    h = np.asarray(residual, dtype=np.float64)[:, : y.shape[1]] + y
    h[:, N:] = 0.0
    return h, rmsnorm(h, gamma, eps, N), y, a


def _f32_div(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """The IEEE fp32 quotient of fp32 values, correctly rounded (to nearest, ties to even): the fp64 quotient rounded
    to fp32.  Rounding twice is harmless for a quotient when the wider format has at least 2p + 2 significant bits
    (53 >= 2 * 24 + 2), subnormal results included."""
    with np.errstate(divide="ignore", invalid="ignore", over="ignore", under="ignore"):
        return (np.asarray(a, dtype=np.float64) / np.asarray(b, dtype=np.float64)).astype(np.float32)


def quantize_act(x_bits: np.ndarray):
    """The quantized form of an activation (``plan.rs`` ``QBLOCK``: 32 values share one scale; ``Buffer::quantized``:
    int8 values and a scale per 32).

    The pages name the form but not its rounding; the reading here is the weight rule of ``from_q8.rs``
    ``quantize`` in the precision the values have (fp32): for each row and block of 32 values,
    amax = max |x|, d = fp32(amax / 127), q = round-half-away-from-zero(fp32(x / d)), clamped to [-127, 127] (the
    clamp never binds for bf16 inputs: d's relative error is at most 2^-10 even at the smallest bf16 subnormal).
    A block of zeros has d = 0 and q = 0; a block holding inf or NaN has d = NaN and q = 0.

    x_bits: uint16 bf16 patterns [m, K] (K a multiple of 32).  Returns (xq int8 [m, K], xd float32 [m, K/32]).
    """
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    m, K = x_bits.shape
    if K % Q8_BLOCK:
        raise ValueError("K must be a multiple of 32")
    nb = K // Q8_BLOCK
    x = (x_bits.astype(np.uint32) << 16).view(np.float32).reshape(m, nb, Q8_BLOCK)
    amax = np.abs(x).max(axis=2)                                   # NaN when the block holds NaN
    bad = ~np.isfinite(amax)
    zero = amax == 0.0
    d = _f32_div(amax, np.float32(127.0))
    safe = np.where(bad | zero, np.float32(1.0), d)
    v = _f32_div(x, safe[:, :, None]).astype(np.float64)
    r = np.clip(_round_half_away(v), -127.0, 127.0)
    r[bad | zero] = 0.0
    xq = r.astype(np.int8).reshape(m, K)
    xd = np.where(bad, np.float32(np.nan), np.where(zero, np.float32(0.0), d)).astype(np.float32)
    return xq, xd


def gemv_q8act(xq: np.ndarray, xd: np.ndarray, q: np.ndarray, s: np.ndarray, cols=None):
    """The Q8_0 product of a quantized activation (the quantized numerics of ``plan.rs``): per row r and column n,
    y = sum_b s[b, n] * d[r, b] * sum_i xq[r, 32b + i] * q[32b + i, n].

    The inner sums are exact integers (int64); each is multiplied by s * d (exact in fp64: 24 by 24 bits) and added
    to the fp64 carry, block b ascending.  A[r, n] = sum_b |s d| sum_i |xq q| is the error scale.
    xq int8 [m, K]; xd float32 [m, K/32]; q int8 [K, Np]; s float32 [K/32, Np]; cols: optional column indices.
    Returns (y, A), fp64 [m, len(cols) or Np]."""
    xq = np.asarray(xq, dtype=np.int8)
    xd = np.asarray(xd, dtype=np.float32)
    m, K = xq.shape
    nb = K // Q8_BLOCK
    if K % Q8_BLOCK or xd.shape != (m, nb) or q.shape[0] != K or s.shape != (nb, q.shape[1]):
        raise ValueError("shape mismatch")
    cols = np.arange(q.shape[1]) if cols is None else np.asarray(cols, dtype=np.int64)
    qc = np.asarray(q, dtype=np.int8)[:, cols].astype(np.int64).reshape(nb, Q8_BLOCK, cols.size)
    sc = np.asarray(s, dtype=np.float32)[:, cols].astype(np.float64)          # [nb, ncols]
    xb = xq.astype(np.int64).reshape(m, nb, Q8_BLOCK).transpose(1, 0, 2)     # [nb, m, 32]
    inner = np.matmul(xb, qc)                                                # [nb, m, ncols], exact
    inner_abs = np.matmul(np.abs(xb), np.abs(qc))
    y = np.zeros((m, cols.size), dtype=np.float64)
    a = np.zeros((m, cols.size), dtype=np.float64)
    dd = xd.astype(np.float64)
    with np.errstate(invalid="ignore"):
        for b in range(nb):
            f = sc[b][None, :] * dd[:, b][:, None]                               # s[b, n] * d[r, b]
            y += f * inner[b].astype(np.float64)
            a += np.abs(f) * inner_abs[b].astype(np.float64)
    return y, a
