"""Pins of the fp64 oracle to what the pages and the mathematics fix (CPU only).

Each pin is chosen so that a plausible slip in the oracle (a dropped block or lane, a wrong sign, a transposed index
of q or s, a wrong bf16 decode, a wrong abs in the error scale) fails at least one test:

* brute force in exact rational arithmetic (Python ``fractions``) on one- and two-block products and on the pages'
  ragged shapes;
* a dense fp64 matmul of the dequantized weight (a special case that reduces to a library routine);
* closed forms from ``tests/golden/closed_forms.txt`` and one-hot activations;
* the exactness of every int8 x bf16 product in fp32 (from_q8.rs module doc);
* the Q8_0 quantize rule and its round trip (from_q8.rs ``quantize``);
* the arg-max's first-maximum rule (int8_model.rs ``decode_step_lg`` and the tie rule of ``reference_cuda``);
* the gated pair (plan.rs ``Launch::GemvGlu``, SwiGLU): the identities silu(g) - silu(-g) = g and
  silu(g) + silu(-g) = g tanh(g/2), which together fix silu(g) = g sigmoid(g), and exact g, u against SiLU evaluated
  in 40-digit decimal arithmetic;
* the residual add and RMS norm (plan.rs ``Launch::Fold`` with ``Launch::Norm``): constant rows normalise to their sign,
  the norm is invariant to scaling the row (eps = 0), the normed row's mean square is 1, a hand-derived 3-4 row in
  decimal arithmetic, and h - residual is the product;
* the quantized activation (plan.rs ``QBLOCK``, ``Buffer::quantized``) and the product that reads it: exact codes
  where d is a power of two, ties away from zero, zero and non-finite blocks, every d and code against the rule in
  exact rational arithmetic with binary32 rounding written out (normal, tiny and subnormal d), the code bounds and
  the d/2 error over every bf16 magnitude, brute force of the product, its integer and one-hot special cases, a
  dense fp64 matmul of the dequantized operands, and the distance to the bf16 product.
"""
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _bf16(v: float) -> int:
    """bf16 bit pattern of a value that bf16 represents exactly."""
    bits = si.f32_to_bf16_bits(np.array([v], dtype=np.float32))[0]
    assert float(si.bf16_bits_to_f32(np.array([bits]))[0]) == v
    return int(bits)


def _exact(x_bits, q, s, r, n):
    """(y, A) of one output in exact rational arithmetic."""
    xf = si.bf16_bits_to_f32(x_bits[r]).astype(np.float64)
    K = x_bits.shape[1]
    y, a = Fraction(0), Fraction(0)
    for b in range(K // 32):
        inner, inner_abs = Fraction(0), Fraction(0)
        for i in range(32):
            k = 32 * b + i
            p = Fraction(float(xf[k])) * int(q[k, n])
            inner += p
            inner_abs += abs(p)
        sv = Fraction(float(s[b, n]))
        y += sv * inner
        a += abs(sv) * inner_abs
    return y, a


# --------------------------------------------------------------------------------------------------------------------
# brute force
# --------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("m", [1, 3])
def test_one_block_is_exact(seed, m):
    """K = 32, N = 1: y = s * sum_i x q has no rounding in fp64, so the oracle equals the rational value exactly."""
    x, q, s = si.case(m, 32, 1, seed)
    y, a = oracle.gemv(x, q, s)
    for r in range(m):
        ey, ea = _exact(x, q, s, r, 0)
        assert y[r, 0] == float(ey)
        assert a[r, 0] == float(ea)
        assert np.all(y[r, 1:] == 0.0) and np.all(a[r, 1:] == 0.0)    # the 31 pad columns


@pytest.mark.parametrize("seed", [4, 5])
def test_two_blocks_two_columns(seed):
    """K = 64, N = 2: at most one rounding (the final add), so |y - exact| <= 2^-52 A; distinguishes q[k,n] from
    q[n,k] and s[b,n] from s[n,b] (both would read other columns' data)."""
    x, q, s = si.case(2, 64, 2, seed)
    y, a = oracle.gemv(x, q, s)
    for r in range(2):
        for n in range(2):
            ey, ea = _exact(x, q, s, r, n)
            assert abs(Fraction(y[r, n]) - ey) <= Fraction(2) ** -52 * ea
            assert abs(Fraction(a[r, n]) - ea) <= Fraction(2) ** -52 * ea


@pytest.mark.parametrize("row", _golden_rows("ragged_shapes.txt"))
def test_pages_ragged_shapes(row):
    """The pages' row-split tails (768, 2,176 rows) and width of 40: brute force on sampled outputs, pads zero."""
    K, N, Np, nblocks, tail = (int(v) for v in row)
    assert oracle.padded_n(N) == Np and K // 32 == nblocks and (K % 1024) // 32 == tail
    x, q, s = si.case(2, K, N, 100 + K)
    y, a = oracle.gemv(x, q, s)
    assert y.shape == (2, Np)
    assert np.all(y[:, N:] == 0.0) and np.all(a[:, N:] == 0.0)
    bound = Fraction(nblocks + 32) * Fraction(2) ** -52
    for r in range(2):
        for n in (0, 17, N - 1):
            ey, ea = _exact(x, q, s, r, n)
            assert abs(Fraction(y[r, n]) - ey) <= bound * ea
            assert abs(Fraction(a[r, n]) - ea) <= bound * ea


def test_column_subset_matches_full():
    x, q, s = si.case(3, 256, 100, 9)
    y, a = oracle.gemv(x, q, s)
    cols = np.array([99, 0, 57, 57, 127])
    ys, as_ = oracle.gemv(x, q, s, cols)
    assert np.array_equal(ys, y[:, cols]) and np.array_equal(as_, a[:, cols])


def test_batch_rows_equal_single_rows():
    """Every row of a batch reads the same weight (from_q8.rs module doc): row r of an m-row product is the
    one-row product of row r, exactly."""
    x, q, s = si.case(5, 512, 70, 11)
    y, _ = oracle.gemv(x, q, s)
    for r in range(5):
        y1, _ = oracle.gemv(x[r:r + 1], q, s)
        assert np.array_equal(y1[0], y[r])


# --------------------------------------------------------------------------------------------------------------------
# dense fp64 matmul and closed forms
# --------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("m,K,N", [(4, 1024, 96), (1, 4096, 40), (16, 256, 33)])
def test_dense_fp64_matmul(m, K, N):
    """y equals x @ W with W = q * s dequantized in fp64 (numpy's matmul), within 1e-12 A."""
    x, q, s = si.case(m, K, N, 20 + m)
    y, a = oracle.gemv(x, q, s)
    dense = si.bf16_bits_to_f32(x).astype(np.float64) @ oracle.dequantize(q, s)
    assert np.all(np.abs(y - dense) <= 1e-12 * a)
    # A is the same matmul over absolute values
    dense_abs = np.abs(si.bf16_bits_to_f32(x).astype(np.float64)) @ np.abs(oracle.dequantize(q, s))
    assert np.all(np.abs(a - dense_abs) <= 1e-12 * a)


@pytest.mark.parametrize("row", _golden_rows("closed_forms.txt"))
def test_closed_forms(row):
    name, K, N, m, expect = row[0], int(row[1]), int(row[2]), int(row[3]), float(row[4])
    Np, nb = oracle.padded_n(N), K // 32
    q = np.zeros((K, Np), np.int8)
    s = np.zeros((nb, Np), np.float32)
    x = np.zeros((m, K), np.uint16)
    if name == "ones":
        x[:] = _bf16(1.0); q[:, :N] = 1; s[:, :N] = 1.0
    elif name == "ramp":
        for r in range(m):
            x[r] = _bf16(float(r + 1))
        q[:, :N] = 1
        s[:, :N] = (2.0 ** -np.arange(nb, dtype=np.float64))[:, None]
    elif name == "alt":
        x[:, 0::2] = _bf16(1.0); x[:, 1::2] = _bf16(-1.0); q[:, :N] = 127; s[:, :N] = 1.0 / 128
    elif name == "signflip":
        x[:] = _bf16(1.0); q[0::2, :N] = 127; q[1::2, :N] = -127; s[:, :N] = 1.0
    y, a = oracle.gemv(x, q, s)
    assert np.all(y[0, :N] == expect)
    assert np.all(y[:, N:] == 0.0) and np.all(a[:, N:] == 0.0)
    if name == "ramp" and m > 1:
        assert np.all(y[1, :N] == 2 * expect)


def test_one_hot_activation():
    """x = e_k: y[n] = s[k/32, n] * q[k, n] exactly, for every k of a block boundary and interior."""
    K, N = 128, 64
    _, q, s = si.case(1, K, N, 31)
    for k in (0, 31, 32, 77, 127):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = _bf16(1.0)
        y, a = oracle.gemv(x, q, s)
        want = s[k // 32].astype(np.float64) * q[k].astype(np.float64)
        assert np.array_equal(y[0], want)
        assert np.array_equal(a[0], np.abs(want))


def test_zero_activation_and_zero_weight():
    x, q, s = si.case(2, 256, 50, 3)
    y, a = oracle.gemv(np.zeros_like(x), q, s)
    assert np.all(y == 0.0) and np.all(a == 0.0)
    y, a = oracle.gemv(x, np.zeros_like(q), np.zeros_like(s))
    assert np.all(y == 0.0) and np.all(a == 0.0)


def test_sign_symmetry_and_linearity():
    """y(-x) = -y(x) exactly (rounding is symmetric in sign); y(x1 + x2) = y(x1) + y(x2) within 1e-12 (A1 + A2)
    for activations whose sum bf16 represents exactly (small integers)."""
    x, q, s = si.case(3, 512, 64, 41)
    y, _ = oracle.gemv(x, q, s)
    yn, _ = oracle.gemv(x ^ np.uint16(0x8000), q, s)
    assert np.array_equal(yn, -y)
    rng = np.random.default_rng(5)
    x1 = rng.integers(-8, 9, size=(3, 512)).astype(np.float32)
    x2 = rng.integers(-8, 9, size=(3, 512)).astype(np.float32)
    b = si.f32_to_bf16_bits
    y1, a1 = oracle.gemv(b(x1), q, s)
    y2, a2 = oracle.gemv(b(x2), q, s)
    y12, _ = oracle.gemv(b(x1 + x2), q, s)
    assert np.all(np.abs(y12 - (y1 + y2)) <= 1e-12 * (a1 + a2))


def test_int8_times_bf16_is_exact_in_fp32():
    """from_q8.rs module doc: an int8 times a bf16 activation is exact in fp32 -- every finite bf16 pattern against
    every int8 in [-127, 127]; the fp32 product equals the fp64 product."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    xf = si.bf16_bits_to_f32(bits)
    finite = np.isfinite(xf)
    xf = xf[finite]
    # the largest finite bf16 times 127 overflows fp32; exactness is claimed for products fp32 can hold
    for qv in range(-127, 128):
        with np.errstate(over="ignore"):
            p32 = (xf * np.float32(qv)).astype(np.float64)
        p64 = xf.astype(np.float64) * qv
        ok = np.abs(p64) < np.float64(np.finfo(np.float32).max)
        assert np.array_equal(p32[ok], p64[ok]), qv


# --------------------------------------------------------------------------------------------------------------------
# quantize (from_q8.rs `quantize`)
# --------------------------------------------------------------------------------------------------------------------

def test_quantize_round_trip():
    """A weight drawn as (q, s) with one +-127 per block dequantizes to values whose Q8_0 quantization is (q, s)."""
    _, q, s = si.case(1, 256, 48, 17)
    w = oracle.dequantize(q[:, :48], s[:, :48])
    got = oracle.quantize(w)
    assert got is not None
    assert np.array_equal(got[0], q[:, :48]) and np.array_equal(got[1], s[:, :48])


def test_quantize_rejects_one_ulp():
    _, q, s = si.case(1, 64, 4, 18)
    w = oracle.dequantize(q[:, :4], s[:, :4])
    w[5, 2] = np.nextafter(w[5, 2], np.inf)
    assert oracle.quantize(w) is None


def test_quantize_rejects_scale_not_fp32():
    """amax = 1 gives d = 1/127, which fp32 does not hold: rejected even though every value is an int multiple."""
    w = np.zeros((32, 1))
    w[0, 0] = 1.0
    assert oracle.quantize(w) is None


def test_quantize_rejects_half_steps_and_keeps_zero_blocks():
    d = 2.0 ** -10
    w = np.zeros((64, 2))
    w[0, 0] = 127 * d
    w[1, 0] = 63.5 * d                 # not an int8 multiple of the block's scale
    assert oracle.quantize(w) is None
    w[1, 0] = -63 * d
    q, s = oracle.quantize(w)
    assert q[0, 0] == 127 and q[1, 0] == -63 and s[0, 0] == np.float32(d)
    assert np.all(q[32:] == 0) and np.all(s[1] == 0) and np.all(q[:, 1] == 0) and s[0, 1] == 0   # zero blocks


# --------------------------------------------------------------------------------------------------------------------
# arg-max
# --------------------------------------------------------------------------------------------------------------------

def test_argmax_first_maximum_and_pads():
    y = np.array([[1.0, 3.0, 3.0, -1.0, 0.0, 0.0],
                  [-5.0, -4.0, -4.5, -7.0, 0.0, 0.0],      # all real logits negative: the pads (0) must not win
                  [0.0, -0.0, -1.0, -0.0, 0.0, 0.0]])      # +0 and -0 are equal: the first one wins
    assert list(oracle.argmax(y, 4)) == [1, 1, 0]
    y2 = y.copy()
    y2[2, 0] = -0.0
    assert oracle.argmax(y2, 4)[2] == 0


def test_argmax_nan_ranks_above_every_number():
    """The reading for NaN logits: a NaN of either sign ranks above +inf, the first NaN of a row wins; without NaN,
    +inf is an ordinary largest value (first one wins) and -inf never beats a number."""
    import struct
    neg_nan = struct.unpack("<d", struct.pack("<Q", 0xFFF8000000000000))[0]
    pos_nan = struct.unpack("<d", struct.pack("<Q", 0x7FF8000000000000))[0]
    inf = float("inf")
    y = np.array([[1.0, inf, 2.0, neg_nan, pos_nan, 0.0],    # NaN above +inf: the first NaN (a negative one)
                  [-inf, 3.0, inf, -2.0, inf, 9.0],          # +inf is the maximum, first one
                  [-inf, -inf, -5.0, -inf, 0.0, 0.0],        # -inf loses to a finite number; pads never count
                  [pos_nan, 1.0, 2.0, 3.0, 0.0, 0.0],        # NaN in the first column
                  [1.0, 2.0, 3.0, 4.0, pos_nan, neg_nan]])   # NaN in the pads does not count
    assert list(oracle.argmax(y, 4)) == [3, 2, 2, 0, 3]
    assert np.signbit(neg_nan) and np.isnan(neg_nan)


def test_argmax_of_product_with_planted_winner():
    x, q, s = si.case(2, 512, 200, 23)
    y, _ = oracle.gemv(x, q, s)
    idx = oracle.argmax(y, 200)
    for r in range(2):
        assert y[r, idx[r]] == y[r, :200].max()
        assert np.all(y[r, :idx[r]] < y[r, idx[r]])


# --------------------------------------------------------------------------------------------------------------------
# repack (from_q8.rs `Q8Part`)
# --------------------------------------------------------------------------------------------------------------------

def _blocks_of(q, s, N):
    """Checkpoint blocks written field by field with struct (independent of the oracle's numpy views)."""
    K = q.shape[0]
    out = bytearray()
    for n in range(N):
        for b in range(K // 32):
            out += struct.pack("<f", float(s[b, n]))
            out += struct.pack("<32b", *[int(v) for v in q[32 * b:32 * b + 32, n]])
    return bytes(out)


def test_repack_round_trip_and_rejects_minus_128():
    _, q, s = si.case(1, 128, 40, 29)
    blk = _blocks_of(q, s, 40)
    got = oracle.repack(blk, 128, 40)
    assert np.array_equal(got[0], q) and np.array_equal(got[1], s)
    q2 = q.copy()
    q2[3, 7] = -128
    assert oracle.repack(_blocks_of(q2, s, 40), 128, 40) is None


def _f16_blocks_of(q, d_bits, N):
    """GGML-style blocks written field by field: the binary16 scale's bit pattern, then the 32 values."""
    K = q.shape[0]
    out = bytearray()
    for n in range(N):
        for b in range(K // 32):
            out += struct.pack("<H", int(d_bits[b, n]))
            out += struct.pack("<32b", *[int(v) for v in q[32 * b:32 * b + 32, n]])
    return bytes(out)


def _half_value(bits: int) -> Fraction:
    """A binary16 bit pattern's value from the IEEE 754 definition (finite patterns)."""
    sign = -1 if bits & 0x8000 else 1
    e, f = (bits >> 10) & 0x1F, bits & 0x3FF
    if e == 0:
        return sign * Fraction(f, 1 << 10) * Fraction(1, 1 << 14)
    return sign * (1 + Fraction(f, 1 << 10)) * Fraction(2) ** (e - 15)


def test_repack_f16_round_trip_and_scales_exact():
    """Every scale comes out as its binary16 value exactly (subnormals, the largest finite, signed zero included);
    values land at [32b + i, n]; -128 and non-finite scales are rejected."""
    rng = np.random.default_rng(31)
    K, N = 96, 40
    q = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    d_bits = rng.integers(0, 0x7C00, size=(K // 32, N)).astype(np.uint16)
    d_bits[0, 0], d_bits[0, 1], d_bits[1, 2], d_bits[2, 3] = 0x0001, 0x03FF, 0x7BFF, 0x8000
    d_bits[1, 5] |= 0x8000
    got = oracle.repack_f16(_f16_blocks_of(q, d_bits, N), K, N)
    assert got is not None and np.array_equal(got[0][:, :N], q) and np.all(got[0][:, N:] == 0)
    for b in range(K // 32):
        for n in range(N):
            assert Fraction(float(got[1][b, n])) == _half_value(int(d_bits[b, n]))
    assert np.all(got[1][:, N:] == 0)
    q2 = q.copy()
    q2[40, 9] = -128
    assert oracle.repack_f16(_f16_blocks_of(q2, d_bits, N), K, N) is None
    for bad in (0x7C00, 0xFC00, 0x7E00):
        d2 = d_bits.copy()
        d2[1, 7] = bad
        assert oracle.repack_f16(_f16_blocks_of(q, d2, N), K, N) is None


def test_bytes_per_weight_fixture():
    """The byte figures the pages print (used by the benchmark's algorithmic byte count)."""
    vals = {r[0]: float(r[1]) for r in _golden_rows("bytes_per_weight.txt")}
    assert vals["q8_bytes_per_weight"] == 1 + 4 / 32
    assert round(vals["q8_bytes_per_weight"], 2) == 1.13 or abs(vals["q8_bytes_per_weight"] - 1.13) < 0.01
    m, wb = 8, 2
    assert abs(vals["view_overhead_m8_wb2"] - (m * 2) / (1.125 * 32 * wb)) < 1e-15


# --------------------------------------------------------------------------------------------------------------------
# the pins catch planted slips: mutants of the oracle's C source, compiled on the CPU, must fail the brute force
# --------------------------------------------------------------------------------------------------------------------

MUTANTS = {
    "scale dropped": ("y += sv * inner;", "y += inner;"),
    "q transposed": ("q[(int64_t)k * Np + n]", "q[(int64_t)n * K + k]"),
    "s transposed": ("s[(int64_t)b * Np + n]", "s[(int64_t)n * (K / ORACLE_BLOCK) + b]"),
    "lane dropped": ("for (int i = 0; i < ORACLE_BLOCK; ++i)", "for (int i = 0; i < ORACLE_BLOCK - 1; ++i)"),
    "bf16 decode": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "abs dropped": ("inner_abs += absd(xv * qv);", "inner_abs += xv * qv;"),
    "block dropped": ("for (int b = 0; b < nblocks; ++b)", "for (int b = 1; b < nblocks; ++b)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "q8_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib_path = tmp_path / "mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(lib_path)])
    lib = ctypes.CDLL(str(lib_path))
    caught = False
    for seed in (4, 5):
        x, q, s = si.case(2, 64, 2, seed)
        Np = q.shape[1]
        y = np.empty((2, Np))
        a = np.empty((2, Np))
        lib.oracle_q8_gemv(ctypes.c_void_p(x.ctypes.data), ctypes.c_void_p(q.ctypes.data),
                           ctypes.c_void_p(s.ctypes.data), 2, 64, Np, None, ctypes.c_int64(Np),
                           ctypes.c_void_p(y.ctypes.data), ctypes.c_void_p(a.ctypes.data))
        for r in range(2):
            for n in range(2):
                ey, ea = _exact(x, q, s, r, n)
                if abs(Fraction(y[r, n]) - ey) > Fraction(2) ** -52 * ea or \
                        abs(Fraction(a[r, n]) - ea) > Fraction(2) ** -52 * ea:
                    caught = True
    assert caught, f"the brute-force pin did not catch: {name}"
# --------------------------------------------------------------------------------------------------------------------
# residual add and RMS norm
# --------------------------------------------------------------------------------------------------------------------

def test_norm_constant_row_is_its_sign():
    """x = 0 (so h = residual): a row of equal values c normalises to sign(c) * gamma exactly when eps = 0."""
    K, N = 64, 40
    x = np.zeros((2, K), dtype=np.uint16)
    _, q, s = si.case(1, K, N, 77)
    res = np.zeros((2, oracle.padded_n(N)), dtype=np.float32)
    res[0, :N], res[1, :N] = 0.75, -3.0
    gamma = np.linspace(0.5, 2.0, oracle.padded_n(N)).astype(np.float32)
    h, out, y, _ = oracle.residual_norm(x, q, s, res, gamma, 0.0, N)
    assert np.all(y == 0.0) and np.array_equal(h[:, :N], res[:, :N].astype(np.float64))
    assert np.array_equal(out[0, :N], gamma[:N].astype(np.float64))
    assert np.array_equal(out[1, :N], -gamma[:N].astype(np.float64))
    assert np.all(out[:, N:] == 0.0)


def test_norm_scale_invariance_and_unit_mean_square():
    """With gamma = 1 and eps = 0: rmsnorm(alpha h) = rmsnorm(h) (alpha a power of two: exact) and the normed row's
    mean square is 1 -- a missing square root or a sum where a mean belongs fails one of them."""
    x, q, s = si.case(3, 256, 300, 78)
    res = np.random.default_rng(3).standard_normal((3, oracle.padded_n(300))).astype(np.float32)
    ones = np.ones(oracle.padded_n(300), dtype=np.float32)
    h, out, _, _ = oracle.residual_norm(x, q, s, res, ones, 0.0, 300)
    out2 = oracle.rmsnorm(8.0 * h, ones, 0.0, 300)
    assert np.allclose(out2, out, rtol=1e-15, atol=0)
    assert np.allclose(np.mean(out[:, :300] ** 2, axis=1), 1.0, rtol=1e-14)


@pytest.mark.parametrize("eps", ["0", "0.000001", "0.5"])
def test_norm_three_four_row_against_decimal(eps):
    """h = (3, 4) (N = 2, x = 0): out = h / sqrt(12.5 + eps) * gamma, in 40-digit decimal arithmetic."""
    from decimal import Decimal, getcontext
    getcontext().prec = 40
    x = np.zeros((1, 32), dtype=np.uint16)
    q = np.zeros((32, 32), dtype=np.int8)
    s = np.zeros((1, 32), dtype=np.float32)
    res = np.zeros((1, 32), dtype=np.float32)
    res[0, 0], res[0, 1] = 3.0, 4.0
    gamma = np.zeros(32, dtype=np.float32)
    gamma[0], gamma[1] = 1.5, -0.25
    _, out, _, _ = oracle.residual_norm(x, q, s, res, gamma, float(eps), 2)
    e = Decimal(float(eps))
    r = (Decimal("12.5") + e).sqrt()
    for n, (hv, gv) in enumerate([(3, Decimal("1.5")), (4, Decimal("-0.25"))]):
        ref = Decimal(hv) / r * gv
        assert abs(Decimal(float(out[0, n])) - ref) <= Decimal(2) ** -50 * abs(ref)


@pytest.mark.parametrize("wrong", ["sum_not_mean", "no_sqrt", "eps_outside"])
def test_norm_pins_catch_planted_mistakes(wrong, monkeypatch):
    """A wrong RMS norm planted in the oracle fails the pins."""
    def bad(h, gamma, eps, N):
        h = np.asarray(h, dtype=np.float64)
        sq = np.sum(h[:, :N] ** 2, axis=1, keepdims=True)
        ms = sq if wrong == "sum_not_mean" else sq / N
        d = {"sum_not_mean": np.sqrt(ms + eps), "no_sqrt": ms + eps, "eps_outside": np.sqrt(ms) + eps}[wrong]
        out = np.zeros_like(h)
        out[:, :N] = h[:, :N] / d * np.asarray(gamma, dtype=np.float64)[:N]
        return out
    monkeypatch.setattr(oracle, "rmsnorm", bad)
    failed = 0
    for pin in (test_norm_constant_row_is_its_sign, test_norm_scale_invariance_and_unit_mean_square,
                lambda: test_norm_three_four_row_against_decimal("0.5")):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


def _norm_like_the_kernels(h32, gamma32, eps, N, threads):
    """The RMS norm the way the library's kernels compute it: float32 sums of squares (thread t takes the 16-byte
    chunks t, t + threads, ... in order, four fused products a chunk), a five-level shuffle tree, the warps in order;
    the mean, + eps, a correctly rounded square root and reciprocal, two products; then rounding to bf16."""
    m, Np = h32.shape
    chunks = Np // 4
    out = np.zeros((m, Np), dtype=np.float32)
    for r in range(m):
        part = np.zeros(threads, dtype=np.float32)
        for t in range(threads):
            acc = np.float32(0.0)
            for j in range(t, chunks, threads):
                for e in range(4):
                    v = np.float64(h32[r, 4 * j + e])
                    acc = np.float32(v * v + np.float64(acc))  # one rounding, as fmaf
            part[t] = acc
        warp = part.reshape(threads // 32, 32)
        for o in (16, 8, 4, 2, 1):
            warp = (warp + np.roll(warp, -o, axis=1)).astype(np.float32)
        ss = np.float32(0.0)
        for w in range(threads // 32):
            ss = np.float32(ss + warp[w, 0])
        rstd = np.float32(1.0) / np.sqrt(np.float32(np.float32(ss / np.float32(N)) + np.float32(eps)))
        out[r, :N] = (h32[r, :N] * rstd).astype(np.float32) * gamma32[:N]
    return si.bf16_bits_to_f32(si.f32_to_bf16_bits(out)).astype(np.float64)


@pytest.mark.parametrize("N,threads", [(300, 256), (4096, 160), (5000, 256)])
def test_rmsnorm_bound_covers_the_kernels_arithmetic(N, threads):
    """oracle.rmsnorm_bound holds for the norm computed in fp32 and rounded to bf16 (rows of very different scales,
    h exact, so only the arithmetic's roundings count), and it is not vacuous: below one bf16 unit of each output."""
    rng = np.random.default_rng(N)
    Np = oracle.padded_n(N)
    h = np.zeros((4, Np))
    h[:, :N] = rng.standard_normal((4, N)) * np.array([[1.0], [1e3], [1e-3], [7.0]])
    h32 = h.astype(np.float32)
    gamma = (0.5 + rng.random(Np)).astype(np.float32)
    eps = 1e-5
    got = _norm_like_the_kernels(h32, gamma, eps, N, threads)
    h64 = h32.astype(np.float64)
    out_o = oracle.rmsnorm(h64, gamma, eps, N)
    bound = oracle.rmsnorm_bound(h64, out_o, np.zeros_like(h64), gamma, eps, N)
    assert np.all(np.abs(got - out_o) <= bound)
    assert np.all(bound[:, :N] < 2.0 ** -7 * np.abs(out_o[:, :N]))
    assert np.all(got[:, N:] == 0.0)


def test_norm_residual_is_added_to_the_product():
    """h - residual equals the product of gemv, column by column (fp64: the add of an fp32 and an fp64 value is
    exact when their magnitudes are close; here checked to 1 ulp of h)."""
    x, q, s = si.case(2, 128, 70, 79)
    res = np.random.default_rng(4).standard_normal((2, oracle.padded_n(70))).astype(np.float32)
    h, _, y, _ = oracle.residual_norm(x, q, s, res, np.ones(96, np.float32), 1e-6, 70)
    assert np.all(np.abs(h[:, :70] - res[:, :70] - y[:, :70]) <= 2.0 ** -52 * np.abs(h[:, :70]) * 2)
    assert np.all(h[:, 70:] == 0.0)


# --------------------------------------------------------------------------------------------------------------------
# the gated pair (SwiGLU)
# --------------------------------------------------------------------------------------------------------------------

def test_glu_odd_and_even_parts_fix_silu():
    """With the gate's weight negated (g -> -g exactly, by the product's sign symmetry):
    glu(Wg) - glu(-Wg) = (silu(g) - silu(-g)) u = g u and glu(Wg) + glu(-Wg) = g tanh(g/2) u (math.tanh), the odd and
    even parts of g sigmoid(g) -- a swapped sign in the exponent or a missing factor fails one of them."""
    import math
    x, qg, sg = si.case(3, 256, 70, 611)
    _, qu, su = si.case(3, 256, 70, 612)
    out, g, u, _, _ = oracle.glu(x, qg, sg, qu, su)
    out_n, g_n, _, _, _ = oracle.glu(x, -qg, sg, qu, su)
    assert np.array_equal(g_n, -g)
    odd = out - out_n
    even = out + out_n
    tanh = np.vectorize(math.tanh)(g / 2.0)
    scale = np.abs(g * u) + 1e-300
    assert np.all(np.abs(odd - g * u) <= 1e-14 * scale)
    assert np.all(np.abs(even - g * tanh * u) <= 1e-14 * scale)


@pytest.mark.parametrize("wrong", ["exp_sign", "no_gate", "sigmoid_only"])
def test_glu_pins_catch_planted_mistakes(wrong, monkeypatch):
    """A wrong SiLU planted in the oracle fails the pins: exp(+g) for exp(-g), silu = g, silu = sigmoid(g)."""
    bad = {"exp_sign": lambda g: g / (1.0 + np.exp(np.asarray(g, dtype=np.float64))),
           "no_gate": lambda g: np.asarray(g, dtype=np.float64),
           "sigmoid_only": lambda g: 1.0 / (1.0 + np.exp(-np.asarray(g, dtype=np.float64)))}[wrong]
    monkeypatch.setattr(oracle, "silu", bad)
    failed = 0
    for pin in (test_glu_odd_and_even_parts_fix_silu, lambda: test_glu_exact_inputs_against_decimal_silu(100, 5)):
        try:
            with np.errstate(over="ignore"):
                pin()
        except AssertionError:
            failed += 1
    assert failed >= 1


@pytest.mark.parametrize("c,e", [(1, 0), (-1, 0), (100, 5), (-100, 5), (127, 2), (-127, 2), (3, 9), (0, 0)])
def test_glu_exact_inputs_against_decimal_silu(c, e):
    """One-hot activation: g = c 2^-e and u = 1/2 exactly (s = 2^-e with q = c; s = 2^-8 with q = 128 is not int8,
    so u = 64 * 2^-7); out = silu(g) / 2 against g / (1 + exp(-g)) in 40-digit decimal arithmetic."""
    from decimal import Decimal, getcontext
    getcontext().prec = 40
    K, N = 32, 1
    x = np.zeros((1, K), dtype=np.uint16)
    x[0, 5] = _bf16(1.0)
    qg = np.zeros((K, 32), dtype=np.int8)
    qu = np.zeros((K, 32), dtype=np.int8)
    qg[5, 0], qu[5, 0] = c, 64
    sg = np.zeros((1, 32), dtype=np.float32)
    su = np.zeros((1, 32), dtype=np.float32)
    sg[0, 0], su[0, 0] = 2.0 ** -e, 2.0 ** -7
    out, g, u, _, _ = oracle.glu(x, qg, sg, qu, su)
    gd = Decimal(c) / (Decimal(2) ** e)
    ref = gd / (1 + (-gd).exp()) / 2
    assert g[0, 0] == float(gd) and u[0, 0] == 0.5
    assert abs(Decimal(float(out[0, 0])) - ref) <= Decimal(2) ** -52 * (abs(ref) + Decimal(10) ** -300)
    assert np.all(out[0, 1:] == 0.0)




# --------------------------------------------------------------------------------------------------------------------
# quantized activations (int8 values and one scale per 32 values)
# --------------------------------------------------------------------------------------------------------------------

def _fp32_round(v: Fraction) -> Fraction:
    """The binary32 value nearest to v (ties to even), subnormals included, in exact rational arithmetic."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()  # 2^e <= a < 2^(e+2)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    return sign * round(a / quantum) * quantum  # round() of a Fraction: nearest, ties to even


def _half_away(v: Fraction) -> int:
    n = int((abs(v) + Fraction(1, 2)) // 1)
    return -n if v < 0 else n


def _act_block(values):
    """bf16 bit patterns [1, 32] of exactly representable values."""
    return np.array([[_bf16(float(v)) for v in values]], dtype=np.uint16)


@pytest.mark.parametrize("e", [-100, -20, -7, 0, 3, 60])
def test_act_quantize_exact_codes(e):
    """x = k 2^e with integers |k| <= 127 and 127 present: d = 127 2^e / 127 = 2^e exactly and every code is k."""
    rng = np.random.default_rng(e + 200)
    k = rng.integers(-127, 128, size=32)
    k[7] = 127 if e % 2 else -127
    x = _act_block([int(v) * 2.0 ** e for v in k])
    xq, xd = oracle.quantize_act(x)
    assert float(xd[0, 0]) == 2.0 ** e
    assert np.array_equal(xq[0].astype(np.int64), k)


def test_act_quantize_ties_go_away_from_zero():
    """With d = 1 (amax = 127): values j + 1/2 are exact ties and go away from zero (62.5 -> 63, -0.5 -> -1); ties to
    even would give 62 and 0."""
    vals = [127.0, 62.5, -62.5, 0.5, -0.5, 1.5, -2.5, 126.5] + [0.0] * 24
    xq, xd = oracle.quantize_act(_act_block(vals))
    assert float(xd[0, 0]) == 1.0
    assert list(xq[0, :8]) == [127, 63, -63, 1, -1, 2, -3, 127]


def test_act_quantize_zero_and_nonfinite_blocks():
    """A block of (signed) zeros gives d = 0 and codes 0; a block holding inf or NaN gives d = NaN and codes 0; the
    other blocks of the row are unaffected."""
    x = np.zeros((3, 64), dtype=np.uint16)
    x[0, :32] = np.uint16(0x8000)
    x[1, 3] = np.uint16(0x7F80)       # +inf
    x[2, 40] = np.uint16(0x7FC0)      # NaN
    x[1, 32:] = _act_block(np.arange(32) - 16.0)
    xq, xd = oracle.quantize_act(x)
    assert xd[0, 0] == 0.0 and not np.signbit(xd[0, 0]) and np.all(xq[0] == 0)
    assert np.isnan(xd[1, 0]) and np.all(xq[1, :32] == 0)
    assert np.isnan(xd[2, 1]) and np.all(xq[2, 32:] == 0)
    assert float(xd[1, 1]) == float(np.float32(16.0) / np.float32(127.0))
    assert xq[1, 32] == -127


@pytest.mark.parametrize("scale", [1.0, 1e-30, 1e-38, 1e30])
def test_act_quantize_against_exact_rational_rounding(scale):
    """Random blocks (N(0,1) times `scale`, so that d is normal, tiny or subnormal): every d and every code equals the
    rule evaluated in exact rational arithmetic with binary32 rounding written out (d = round32(amax / 127),
    q = half-away(round32(x / d)))."""
    rng = np.random.default_rng(int(abs(np.log10(scale))) + 17)
    x = si.f32_to_bf16_bits((rng.standard_normal((4, 96)) * scale).astype(np.float32)).reshape(4, 96)
    xq, xd = oracle.quantize_act(x)
    xf = si.bf16_bits_to_f32(x.reshape(-1)).reshape(4, 96)
    for r in range(4):
        for b in range(3):
            blk = [Fraction(float(v)) for v in xf[r, 32 * b:32 * b + 32]]
            amax = max(abs(v) for v in blk)
            d = _fp32_round(amax / 127)
            assert Fraction(float(xd[r, b])) == d
            for i, v in enumerate(blk):
                assert int(xq[r, 32 * b + i]) == max(-127, min(127, _half_away(_fp32_round(v / d))))


def test_act_quantize_invariants_over_every_bf16_magnitude():
    """For every positive finite bf16 value a as a block's amax (with -a, a/3 and a small value beside it): the code
    at +-a is +-127, every code lies in [-127, 127], and every value is within d/2 (plus the fp32 quotient's
    rounding) of q d."""
    mags = np.arange(1, 0x7F80, dtype=np.uint16)
    n = mags.size
    x = np.zeros((n, 32), dtype=np.uint16)
    x[:, 0] = mags
    x[:, 1] = mags | np.uint16(0x8000)
    third = si.bf16_bits_to_f32(mags) / np.float32(3.0)
    x[:, 2] = si.f32_to_bf16_bits(third.astype(np.float32))
    x[:, 3] = np.uint16(1)
    xq, xd = oracle.quantize_act(x)
    assert np.all(xq[:, 0] == 127) and np.all(xq[:, 1] == -127)
    assert np.abs(xq.astype(np.int64)).max() <= 127
    xf = si.bf16_bits_to_f32(x.reshape(-1)).reshape(n, 32).astype(np.float64)
    d = xd[:, 0].astype(np.float64)[:, None]
    err = np.abs(xf - xq.astype(np.float64) * d)
    assert np.all(err <= d * (0.5 + 2.0 ** -9) + 2.0 ** -149)


def _exact_q8act(xq, xd, q, s, r, n):
    K = xq.shape[1]
    y = Fraction(0)
    for b in range(K // 32):
        inner = sum(int(xq[r, 32 * b + i]) * int(q[32 * b + i, n]) for i in range(32))
        y += Fraction(float(s[b, n])) * Fraction(float(xd[r, b])) * inner
    return y


@pytest.mark.parametrize("K,N,m", [(32, 1, 1), (32, 3, 2), (64, 2, 3), (96, 33, 1)])
def test_q8act_product_brute_force(K, N, m):
    """Exact rational y = sum_b s d sum_i xq q for every output; the oracle's fp64 result is within a few ulps."""
    x, q, s = si.case(m, K, N, 300 + K + N)
    xq, xd = oracle.quantize_act(x)
    y, a = oracle.gemv_q8act(xq, xd, q, s)
    for r in range(m):
        for n in range(q.shape[1]):
            ref = _exact_q8act(xq, xd, q, s, r, n)
            assert abs(Fraction(float(y[r, n])) - ref) <= Fraction(2) ** -50 * Fraction(float(a[r, n]))


def test_q8act_integer_case_and_one_hot():
    """s = d = 1: y is the integer dot sum_k xq[k] q[k, n] exactly (Python integers); a one-hot xq = c e_k gives
    y[n] = s[k/32, n] d c q[k, n]."""
    rng = np.random.default_rng(8)
    K, N = 2048, 64
    xq = rng.integers(-127, 128, size=(2, K)).astype(np.int8)
    q = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    ones_s = np.ones((K // 32, N), dtype=np.float32)
    ones_d = np.ones((2, K // 32), dtype=np.float32)
    y, _ = oracle.gemv_q8act(xq, ones_d, q, ones_s)
    for r in range(2):
        for n in (0, 17, 63):
            assert y[r, n] == sum(int(xq[r, k]) * int(q[k, n]) for k in range(K))
    _, q2, s2 = si.case(1, 256, 40, 9)
    oh = np.zeros((1, 256), dtype=np.int8)
    oh[0, 77] = -93
    d = np.full((1, 8), 0.375, dtype=np.float32)
    y2, _ = oracle.gemv_q8act(oh, d, q2, s2)
    expect = s2[77 // 32].astype(np.float64) * 0.375 * -93 * q2[77].astype(np.float64)
    assert np.array_equal(y2[0], expect)


@pytest.mark.parametrize("m,K,N", [(4, 1024, 96), (16, 256, 33)])
def test_q8act_dense_fp64_matmul(m, K, N):
    """y = (xq d) @ (q s), the dequantized activation and weight multiplied by numpy's fp64 matmul: within 1e-12 A."""
    x, q, s = si.case(m, K, N, 410 + m)
    xq, xd = oracle.quantize_act(x)
    y, a = oracle.gemv_q8act(xq, xd, q, s)
    xdq = xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1)
    ref = xdq @ oracle.dequantize(q, s)
    assert np.all(np.abs(y - ref) <= 1e-12 * a)


def test_q8act_close_to_the_bf16_product():
    """The quantized numerics differ from the bf16 product by at most the quantization error carried through the
    weight: |y_q8 - y_bf16| <= sum_b |s| sum_i |x - d xq| |q| (+ fp64 rounding)."""
    x, q, s = si.case(3, 512, 70, 420)
    xq, xd = oracle.quantize_act(x)
    y8, a8 = oracle.gemv_q8act(xq, xd, q, s)
    y, a = oracle.gemv(x, q, s)
    xf = si.bf16_bits_to_f32(x.reshape(-1)).reshape(x.shape).astype(np.float64)
    dx = np.abs(xf - xq.astype(np.float64) * np.repeat(xd.astype(np.float64), 32, axis=1))
    bound = dx @ np.abs(oracle.dequantize(q, s))
    assert np.all(np.abs(y8 - y) <= bound + 1e-12 * (a + a8))
    assert np.all(bound <= 0.02 * a + 1e-30)


@pytest.mark.parametrize("wrong", ["row_scale_of_other_row", "no_act_scale", "block_scale_shifted", "round_to_even"])
def test_q8act_pins_catch_planted_mistakes(wrong, monkeypatch):
    """Wrong quantized numerics planted in the oracle fail the pins."""
    good_q, good_p = oracle.quantize_act, oracle.gemv_q8act

    def bad_product(xq, xd, q, s, cols=None):
        xd = np.asarray(xd, dtype=np.float32)
        if wrong == "row_scale_of_other_row":
            xd = xd[::-1].copy()
        elif wrong == "no_act_scale":
            xd = np.ones_like(xd)
        elif wrong == "block_scale_shifted":
            xd = np.roll(xd, 1, axis=1)
        return good_p(xq, xd, q, s, cols)

    def bad_quantize(x_bits):
        xq, xd = good_q(x_bits)
        xf = si.bf16_bits_to_f32(np.asarray(x_bits).reshape(-1)).reshape(xq.shape).astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            v = xf / np.repeat(xd.astype(np.float64), 32, axis=1)
        return np.where(np.isfinite(v), np.clip(np.round(v), -127, 127), 0).astype(np.int8), xd

    if wrong == "round_to_even":
        monkeypatch.setattr(oracle, "quantize_act", bad_quantize)
    else:
        monkeypatch.setattr(oracle, "gemv_q8act", bad_product)
    failed = 0
    for pin in (test_act_quantize_ties_go_away_from_zero, lambda: test_q8act_product_brute_force(64, 2, 3),
                lambda: test_q8act_dense_fp64_matmul(4, 1024, 96)):
        try:
            pin()
        except AssertionError:
            failed += 1
    assert failed >= 1
