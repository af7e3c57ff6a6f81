"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, element by element.

Bar (the product's stated bound): |y_gpu - y_oracle| <= 1e-5 * A for every output, A = sum_b |s| sum_i |x q|; where
A = 0 the GPU value must be exactly 0.  Arg-max: the oracle's first maximum wherever its gap to every other column
exceeds the two columns' bounds, otherwise one of the columns within the bound; constructed ties go to the lowest
index.  Sizes span several column tiles, K splits and a ragged last tile; the largest shapes are checked on sampled
columns in the launch configuration the benchmark uses.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

TOL = 1e-5


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    return torch


def _to_dev(torch, x, q, s):
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    return xd, torch.from_numpy(np.ascontiguousarray(q)).cuda(), torch.from_numpy(np.ascontiguousarray(s)).cuda()


def _gemv(torch, x, q, s, N, variant="auto"):
    """One call through the C ABI; variant "tiled" first rearranges the weight with q8_tile_device."""
    import q8_block_quantized_gemv_gb300 as q8
    xd, qd, sd = _to_dev(torch, x, q, s)
    if variant == "tiled":
        qt, st = q8.tile_device(qd, sd, N)
        y = q8.gemv(xd, qt, st, N, tiled=True)
    else:
        y = q8.gemv(xd, qd, sd, N, variant=variant)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _assert_close(y_gpu, y_o, a_o, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_o)
    bad = err > TOL * a_o
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of bound; first at ({r},{c}): gpu {y_gpu[r, c]!r} "
                             f"oracle {y_o[r, c]!r} A {a_o[r, c]!r}")


def _variants(m):
    import q8_block_quantized_gemv_gb300 as q8
    out = ["auto", "mma", "tma", "tiled"]
    if m in (1, 2, 3, 4, 8):
        out.append("simt")
    return out


# --------------------------------------------------------------------------------------------------------------------
# element-by-element parity
# --------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("m", list(range(1, 17)))
def test_single_gemv_1024(dev, m):
    """The single 1024 x 1024 GEMV workload (x bf16 N(0,1), q uniform int8 with a +-127 per block, s = 2^u/127),
    every row count 1..16, every kernel family."""
    x, q, s = si.case(m, 1024, 1024, si.case_seed(0, m))
    y_o, a_o = oracle.gemv(x, q, s)
    for v in _variants(m):
        _assert_close(_gemv(dev, x, q, s, 1024, v), y_o, a_o, f"m={m} {v}")


@pytest.mark.parametrize("N", [40, 3000, 6144])
def test_ragged_tp_shapes(dev, N):
    """Ragged tensor-parallel shapes, K = 5120, m = 3, zero-padded last tile; pads written as exactly 0."""
    x, q, s = si.case(3, 5120, N, si.case_seed(3, 3, N))
    y_o, a_o = oracle.gemv(x, q, s)
    for v in _variants(3):
        y = _gemv(dev, x, q, s, N, v)
        _assert_close(y, y_o, a_o, f"N={N} {v}")
        assert np.all(y[:, N:] == 0.0)


@pytest.mark.parametrize("K", [768, 2176])
@pytest.mark.parametrize("m", [1, 2, 16])
def test_pages_row_split_tails(dev, K, m):
    """The pages' row-split weights (768 and 2,176 rows: K not whole 1,024-row blocks) at a width of 40."""
    x, q, s = si.case(m, K, 40, 500 + K + m)
    y_o, a_o = oracle.gemv(x, q, s)
    for v in _variants(m):
        _assert_close(_gemv(dev, x, q, s, 40, v), y_o, a_o, f"K={K} m={m} {v}")


@pytest.mark.parametrize("m,K,N", [(1, 32, 1), (16, 32, 1), (3, 32, 33), (5, 64, 2), (16, 14336, 32),
                                   (1, 14336, 64), (8, 4096, 96), (2, 256, 100000)])
def test_edge_shapes(dev, m, K, N):
    """One block; one column; narrow N with deep K (the cluster split of K); very wide N with few blocks."""
    x, q, s = si.case(m, K, N, 700 + m + K + N)
    cols = None if N <= 6144 else np.r_[0:64, N - 64:oracle.padded_n(N)]
    y_o, a_o = oracle.gemv(x, q, s, cols)
    for v in _variants(m):
        y = _gemv(dev, x, q, s, N, v)
        _assert_close(y if cols is None else y[:, cols], y_o, a_o, f"m={m} K={K} N={N} {v}")


@pytest.mark.parametrize("m", [1, 4, 16])
def test_attention_projection_4096(dev, m):
    """The 7B-class attention projection, K = N = 4096, m = 1, 4, 16: every output, row-major and tiled."""
    x, q, s = si.case(m, 4096, 4096, si.case_seed(1, m))
    y_o, a_o = oracle.gemv(x, q, s)
    for v in ("auto", "tiled"):
        _assert_close(_gemv(dev, x, q, s, 4096, v), y_o, a_o, f"m={m} {v}")


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_ffn_projections_sampled(dev, K, N, m):
    """FFN up/gate (4096 x 14336) and down (14336 x 4096) at full size, m = 1, 2, 4, 8, 16, in the benchmark's
    launch configuration (tiled) and row-major; checked on 384 sampled columns (tile edges, the last columns and
    random ones)."""
    x, q, s = si.case(m, K, N, si.case_seed(2, m, 1 if K > N else 0))
    rng = np.random.default_rng(m)
    cols = np.unique(np.r_[0:32, 120:136, 248:264, 504:520, N - 32:N, rng.integers(0, N, 256)])
    y_o, a_o = oracle.gemv(x, q, s, cols)
    for v in ("auto", "tiled"):
        y = _gemv(dev, x, q, s, N, v)
        _assert_close(y[:, cols], y_o, a_o, f"K={K} N={N} m={m} {v}")


# --------------------------------------------------------------------------------------------------------------------
# activation magnitude ranges (the tiled path's exact fp16 scaling and its bf16 alternative)
# --------------------------------------------------------------------------------------------------------------------

def _bits(v):
    a = np.asarray(v, dtype=np.float32)
    return si.f32_to_bf16_bits(a).reshape(a.shape)


def _ranged_case(m, kinds=tuple(range(14)), nb_each=2, N=300, seed=4242):
    """Activations built block by block (all rows of a 32-row block share a kind), every kind twice:
    0 N(0,1); 1 N(0,1) * 1e30; 2 N(0,1) * 1e-30; 3 N(0,1) * 1e-36 (below the scalable range); 4 rows alternating
    1e10 and 1e-10 (a 66-binade span); 5 one 1.0 per row and 1e-12 * N(0,1) elsewhere, with the weight row of the
    1.0 zeroed in 150 columns (the large activation meets zero weights); 6 signed powers 2^-26 .. 2^3 with random
    mantissas, both ends present (a 29-binade span: the widest exact fp16 scaling); 7 as 6 plus one 2^-27 (one binade
    more); 8 N(0,1) with a few bf16 subnormals; 9 zeros and negative zeros; 10 zeros with a few N(0,1) values;
    11 values +-1.9921875 * 2^k, k in -10..9 (the largest bf16 mantissa in the top binade: 65280 after scaling);
    12 signed values m * 2^e, e in -14..15, with 2^-14 and 1.9921875 * 2^15 = 65280 present (the widest range that is
    already fp16 normal, so that no scaling is needed); 13 as 12 plus one -1.5 * 2^-15 (one binade below it).
    Blocks cycle through `kinds`."""
    nb = len(kinds) * nb_each
    K = 32 * nb
    rng = np.random.default_rng(seed)
    x = np.zeros((m, K), dtype=np.uint16)
    _, q, s = si.case(1, K, N, seed)
    for b in range(nb):
        kind = kinds[b % len(kinds)]
        sl = slice(32 * b, 32 * b + 32)
        g = rng.standard_normal((m, 32)).astype(np.float32)
        if kind == 0:
            v = _bits(g)
        elif kind == 1:
            v = _bits(g * np.float32(1e30))
        elif kind == 2:
            v = _bits(g * np.float32(1e-30))
        elif kind == 3:
            v = _bits(g * np.float32(1e-36))
        elif kind == 4:
            f = np.where(np.arange(m)[:, None] % 2 == 0, np.float32(1e10), np.float32(1e-10))
            v = _bits(g * f)
        elif kind == 5:
            v = _bits(g * np.float32(1e-12))
            v[:, 0] = _bits(np.float32(1.0))
            q[32 * b, :150] = 0
        elif kind in (6, 7):
            e = rng.integers(-26, 4, size=(m, 32))
            e[:, 0], e[:, 1] = 3, -26
            mant = 1.0 + rng.integers(0, 128, size=(m, 32)) / 128.0
            sign = np.where(rng.integers(0, 2, size=(m, 32)) == 1, -1.0, 1.0)
            v = _bits((sign * mant * np.exp2(e)).astype(np.float32))
            if kind == 7:
                v[m - 1, 5] = _bits(np.float32(-1.5 * 2.0 ** -27))
        elif kind == 8:
            v = _bits(g)
            v[:, 3] = np.uint16(0x0041)
            v[0, 7] = np.uint16(0x8005)
        elif kind == 9:
            v = np.where(rng.integers(0, 2, size=(m, 32)) == 1, np.uint16(0x8000), np.uint16(0)).astype(np.uint16)
        elif kind in (12, 13):
            e = rng.integers(-14, 16, size=(m, 32))
            mant = 1.0 + rng.integers(0, 128, size=(m, 32)) / 128.0
            e[:, 0], mant[:, 0] = 15, 1.9921875
            e[:, 1] = -14
            sign = np.where(rng.integers(0, 2, size=(m, 32)) == 1, -1.0, 1.0)
            v = _bits((sign * mant * np.exp2(e)).astype(np.float32))
            if kind == 13:
                v[m // 2, 9] = _bits(np.float32(-1.5 * 2.0 ** -15))
        elif kind == 10:
            v = np.zeros((m, 32), dtype=np.uint16)
            v[:, 4] = _bits(g[:, 4])
            v[0, 31] = _bits(g[0, 31])
        else:
            k = rng.integers(-10, 10, size=(m, 32))
            k[:, 0] = 9
            v = _bits((1.9921875 * np.exp2(k) * np.sign(g + 0.5)).astype(np.float32))
        x[:, sl] = v
    return x, q, s, N


@pytest.mark.parametrize("kinds", [tuple(range(14))] + [(k,) for k in range(14)], ids=lambda k: "-".join(map(str, k)))
@pytest.mark.parametrize("m", [5, 16])
def test_activation_magnitude_ranges(dev, m, kinds):
    """Every activation range the scaled fp16 operands must either represent exactly or hand to bf16 operands: the
    bound holds for every output of every kernel family, all kinds mixed and each kind alone (so that the bound is
    set by that kind's own magnitudes), including the columns whose large activations meet zero weights (A is then
    set by the 1e-12 values alone)."""
    x, q, s, N = _ranged_case(m, kinds, nb_each=max(2, 24 // len(kinds)))
    y_o, a_o = oracle.gemv(x, q, s)
    for v in _variants(m):
        _assert_close(_gemv(dev, x, q, s, N, v), y_o, a_o, f"m={m} kinds={kinds} {v}")


@pytest.mark.parametrize("m", [3, 12])
def test_nonfinite_activations_propagate(dev, m):
    """inf, -inf and NaN activations give the oracle's NaN / +-inf pattern in the outputs (IEEE: inf * 0 and
    inf - inf are NaN); every finite output meets the bound."""
    K, N = 512, 260
    x, q, s = si.case(m, K, N, 515 + m)
    x[0, 40] = np.uint16(0x7F80)           # +inf
    x[m - 1, 300] = np.uint16(0xFF80)      # -inf
    x[1, 77] = np.uint16(0x7FC0)           # NaN
    y_o, a_o = oracle.gemv(x, q, s)
    for v in _variants(m):
        y = _gemv(dev, x, q, s, N, v).astype(np.float64)[:, :N]
        yo, ao = y_o[:, :N], a_o[:, :N]
        assert np.array_equal(np.isnan(y), np.isnan(yo)), v
        inf = np.isinf(yo)
        assert np.array_equal(np.isinf(y), inf) and np.array_equal(y[inf], yo[inf]), v
        fin = np.isfinite(yo)
        assert np.all(np.abs(y[fin] - yo[fin]) <= TOL * ao[fin]), v


# --------------------------------------------------------------------------------------------------------------------
# properties
# --------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("m", [1, 3, 9, 16])
def test_deterministic_and_sign_symmetric(dev, m):
    """Repeated calls give identical bits; y(-x) = -y(x) bit for bit (every rounding is sign-symmetric)."""
    x, q, s = si.case(m, 4096, 1000, 900 + m)
    for v in _variants(m):
        y1 = _gemv(dev, x, q, s, 1000, v)
        y2 = _gemv(dev, x, q, s, 1000, v)
        yn = _gemv(dev, x ^ np.uint16(0x8000), q, s, 1000, v)
        assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32)), v
        assert np.array_equal(yn, -y1), v


def test_batch_rows_match_single_rows(dev):
    x, q, s = si.case(7, 2048, 700, 77)
    y7 = _gemv(dev, x, q, s, 700)
    y_o, a_o = oracle.gemv(x, q, s)
    for r in range(7):
        y1 = _gemv(dev, x[r:r + 1], q, s, 700)
        _assert_close(y1, y_o[r:r + 1], a_o[r:r + 1], f"row {r}")
        assert np.all(np.abs(y1[0].astype(np.float64) - y7[r]) <= 2 * TOL * a_o[r])


def test_guards_and_dirty_pads(dev):
    """Nothing outside y[m, Np] is written; garbage in the pad columns of q and s does not reach real columns and
    the pad outputs are still exactly 0."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    m, K, N = 5, 1024, 3000
    x, q, s = si.case(m, K, N, 31)
    y_o, a_o = oracle.gemv(x, q, s)
    q2, s2 = q.copy(), s.copy()
    q2[:, N:] = 99
    s2[:, N:] = 3.0
    xd, qd, sd = _to_dev(torch, x, q2, s2)
    Np = oracle.padded_n(N)
    guard = 4096
    buf = torch.full((m * Np + 2 * guard,), 12345.0, dtype=torch.float32, device="cuda")
    y = buf[guard:guard + m * Np].view(m, Np)
    for v in _variants(m):
        if v == "tiled":
            qt, st = q8.tile_device(qd, sd, N)
            q8.gemv(xd, qt, st, N, y=y, tiled=True)
        else:
            q8.gemv(xd, qd, sd, N, y=y, variant=v)
        torch.cuda.synchronize()
        host = buf.cpu().numpy()
        assert np.all(host[:guard] == 12345.0) and np.all(host[guard + m * Np:] == 12345.0)
        yy = host[guard:guard + m * Np].reshape(m, Np)
        assert np.all(yy[:, N:] == 0.0)
        _assert_close(yy[:, :N], y_o[:, :N], a_o[:, :N], v)


# --------------------------------------------------------------------------------------------------------------------
# arg-max
# --------------------------------------------------------------------------------------------------------------------

def _argmax_ok(idx, y_o, a_o, N):
    """The acceptance rule: exact where the oracle's winner clears every other column's bound, else within it."""
    for r in range(y_o.shape[0]):
        best = int(oracle.argmax(y_o[r:r + 1], N)[0])
        close = (y_o[r, best] - y_o[r, :N]) <= TOL * (a_o[r, best] + a_o[r, :N])
        close[best] = True
        if close.sum() == 1:
            assert idx[r] == best, (r, idx[r], best)
        else:
            assert close[idx[r]], (r, idx[r], best)


def _argmax(torch, x, q, s, N, with_logits=True, tiled=False):
    import q8_block_quantized_gemv_gb300 as q8
    xd, qd, sd = _to_dev(torch, x, q, s)
    logits = torch.empty((x.shape[0], q.shape[1]), dtype=torch.float32, device="cuda") if with_logits else None
    if tiled:
        qd, sd = q8.tile_device(qd, sd, N)
    idx = q8.gemv_argmax(xd, qd, sd, N, logits=logits, tiled=tiled)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), (logits.cpu().numpy() if with_logits else None)


@pytest.mark.parametrize("m", [1, 2])
def test_argmax_tied_head_full(dev, m):
    """The tied head, K = 4096, N = 128256, every logit against the oracle; the fused arg-max under the rule."""
    x, q, s = si.case(m, 4096, 128256, si.case_seed(4, m))
    y_o, a_o = oracle.gemv(x, q, s)
    idx, logits = _argmax(dev, x, q, s, 128256)
    _assert_close(logits, y_o, a_o, "head logits")
    _argmax_ok(idx, y_o, a_o, 128256)
    # the fused arg-max is exactly the first maximum of the logits the same call wrote
    for r in range(m):
        assert idx[r] == int(np.flatnonzero(logits[r, :128256] == logits[r, :128256].max())[0])
    idx2, _ = _argmax(dev, x, q, s, 128256, with_logits=False)
    assert np.array_equal(idx, idx2)
    idx3, logits3 = _argmax(dev, x, q, s, 128256, tiled=True)
    _assert_close(logits3, y_o, a_o, "head logits, tiled")
    _argmax_ok(idx3, y_o, a_o, 128256)


def test_argmax_head_m16_every_row(dev):
    """The tied head at m = 16 (K = 4096, N = 128256): every logit of every row against the oracle, and each row's
    fused arg-max under the rule -- on the row-major and the tiled storage."""
    x, q, s = si.case(16, 4096, 128256, si.case_seed(4, 16))
    y_o, a_o = oracle.gemv(x, q, s)
    for tiled in (False, True):
        idx, logits = _argmax(dev, x, q, s, 128256, tiled=tiled)
        _assert_close(logits, y_o, a_o, f"head logits, tiled={tiled}")
        _argmax_ok(idx, y_o, a_o, 128256)
        for r in range(16):
            assert idx[r] == int(np.flatnonzero(logits[r, :128256] == logits[r, :128256].max())[0])


@pytest.mark.parametrize("m", [1, 5, 16])
def test_argmax_planted_ties_and_pads(dev, m):
    K, N = 1024, 3000
    x, q, s = si.case(m, K, N, 1300 + m)
    xf = si.bf16_bits_to_f32(x)
    # a planted winner for row 0: column 1234 aligned with the signs of row 0's activations
    q[:, 1234] = np.where(xf[0] >= 0, 127, -127).astype(np.int8)
    s[:, 1234] = s[:, :N].max()
    # ties: copies of the winner further right
    for c in (1500, 2999):
        q[:, c] = q[:, 1234]
        s[:, c] = s[:, 1234]
    y_o, a_o = oracle.gemv(x, q, s)
    for tiled in (False, True):
        idx, _ = _argmax(dev, x, q, s, N, tiled=tiled)
        assert idx[0] == 1234
        _argmax_ok(idx, y_o, a_o, N)
    # every real logit negative: the pad columns (exactly 0) must not win
    xa = si.f32_to_bf16_bits(np.abs(xf))
    qn = -np.abs(q.astype(np.int16)).astype(np.int8)
    qn[:, 0] = -1                         # keep every column strictly negative
    qn[:, N:] = 0
    y_o, a_o = oracle.gemv(xa, qn, s)
    assert np.all(y_o[:, :N] < 0)
    idx, _ = _argmax(dev, xa, qn, s, N)
    assert np.all(idx < N)
    _argmax_ok(idx, y_o, a_o, N)


@pytest.mark.parametrize("m", [1, 3, 16])
def test_argmax_nonfinite_logits(dev, m):
    """Activations holding inf or NaN make the logits +-inf and NaN (inf * 0 is NaN).  The arg-max follows the
    oracle's reading exactly: a NaN of either sign ranks above every number (the first NaN wins), +inf above every
    finite logit (the first +inf wins); the other rows as usual."""
    K, N = 512, 700
    x, q, s = si.case(m, K, N, 1400 + m)
    x[0, 40] = np.uint16(0x7F80)          # row 0: +inf meets q[40, n]: +-inf, NaN where q[40, n] = 0
    q[40, [100, 300]] = 0
    if m > 1:
        x[1, 41] = np.uint16(0x7F80)      # row 1: +inf, every q[41, n] nonzero: +-inf only, the first +inf wins
        q[41, :N][q[41, :N] == 0] = 1
        x[2, 7] = np.uint16(0xFFC0)       # row 2: a negative NaN activation: every real logit NaN
    y_o, a_o = oracle.gemv(x, q, s)
    want = oracle.argmax(y_o, N)
    assert want[0] == int(np.flatnonzero(q[40, :N] == 0)[0])
    special = [0] if m == 1 else [0, 1, 2]
    for tiled in (False, True):
        idx, logits = _argmax(dev, x, q, s, N, tiled=tiled)
        assert np.array_equal(np.isnan(logits[:, :N]), np.isnan(y_o[:, :N])), tiled
        for r in special:
            assert idx[r] == want[r], (tiled, r, idx[r], want[r])
        rest = [r for r in range(m) if r not in special]
        if rest:
            _argmax_ok(idx[rest], y_o[rest], a_o[rest], N)


def test_argmax_scratch_contents_do_not_matter(dev):
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s = si.case(4, 1024, 2000, 55)
    xd, qd, sd = _to_dev(torch, x, q, s)
    idx = torch.full((4,), -1, dtype=torch.int64, device="cuda")
    a = q8.gemv_argmax(xd, qd, sd, 2000, idx=idx).cpu().numpy()
    idx.fill_(2**62)
    b = q8.gemv_argmax(xd, qd, sd, 2000, idx=idx).cpu().numpy()
    assert np.array_equal(a, b)
    y_o, a_o = oracle.gemv(x, q, s)
    _argmax_ok(a, y_o, a_o, 2000)


@pytest.mark.parametrize("ks", [1, 2, 3, 5, 8])
def test_tma_every_cluster_split(dev, ks, tune):
    """The pipelined kernel at every K split across a cluster (the planner's choice forced), m = 1 and 16, against
    the oracle; the device fault word stays clear (no bounded wait ran out)."""
    import q8_block_quantized_gemv_gb300 as q8
    tune(ksplit=ks)
    for m in (1, 16):
        x, q, s = si.case(m, 2048, 1000, 1700 + ks + m)
        y_o, a_o = oracle.gemv(x, q, s)
        for v in ("tma", "tiled"):
            _assert_close(_gemv(dev, x, q, s, 1000, v), y_o, a_o, f"ks={ks} m={m} {v}")
    assert q8.device_fault() == 0


@pytest.mark.parametrize("m", [1, 2, 3, 9, 16])
def test_single_tile_sixteen_rank_cluster(dev, m):
    """One column tile (N = 40, K = 5120) on the tiled storage: the planner splits K over a cluster of up to 16 CTAs
    (above the portable 8 when the residency query allows), whose epilogue loads the ranks' partials in groups of
    eight and sums them in rank order -- every output against the oracle, the pads exactly 0, and the same bits on a
    second call."""
    x, q, s = si.case(m, 5120, 40, 7300 + m)
    y_o, a_o = oracle.gemv(x, q, s)
    y1 = _gemv(dev, x, q, s, 40, "tiled")
    _assert_close(y1, y_o, a_o, f"m={m}")
    assert np.all(y1[:, 40:] == 0)
    y2 = _gemv(dev, x, q, s, 40, "tiled")
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_no_device_fault_after_suite(dev):
    import q8_block_quantized_gemv_gb300 as q8
    assert q8.device_fault(clear=True) == 0


@pytest.mark.parametrize("tiled", [False, True])
@pytest.mark.parametrize("m", [1, 16])
def test_graph_chain_with_constant_weights(dev, m, tiled):
    """Back-to-back calls captured in a CUDA graph and replayed, weights declared constant (programmatic dependent
    launch lets each call start streaming its weights before the previous call ends) -- the benchmark's launch
    configuration -- each output against the oracle; the last call reads the first call's output as its activation
    (a true dependency through x)."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    shapes = [(1024, 2048), (2048, 1024), (1024, 4096), (4096, 1024)]
    host = [si.case(m, K, N, 3100 + 10 * i + m) for i, (K, N) in enumerate(shapes)]
    devs = [_to_dev(torch, *h) for h in host]
    if tiled:
        devs = [(xd,) + q8.tile_device(qd, sd, N) for (xd, qd, sd), (_, N) in zip(devs, shapes)]
    ys = [torch.empty((m, N), dtype=torch.float32, device="cuda") for _, N in shapes]
    xdep = torch.empty((m, 2048), dtype=torch.bfloat16, device="cuda")

    def run():
        for i, (K, N) in enumerate(shapes):
            xd, qd, sd = devs[i]
            if i == 1:
                xd = xdep
            q8.gemv(xd, qd, sd, N, y=ys[i], constant_weights=True, tiled=tiled)
            if i == 0:
                xdep.copy_(ys[0].to(torch.bfloat16))   # a torch kernel between two calls, on the same stream

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        for y in ys:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        for i, (K, N) in enumerate(shapes):
            x, q, s_ = host[i]
            if i == 1:
                x = xdep.view(torch.int16).cpu().numpy().view(np.uint16)
            y_o, a_o = oracle.gemv(x, q, s_)
            _assert_close(ys[i].cpu().numpy(), y_o, a_o, f"call {i} m={m}")
    assert q8.device_fault() == 0


@pytest.mark.parametrize("K,N", [(64, 40), (1024, 3000), (4096, 128256)])
def test_tile_device_matches_host(dev, K, N):
    """q8_tile_device writes exactly the bytes q8_tile writes (the host transform is pinned on the CPU)."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    _, q, s = si.case(1, K, N, 4400 + N)
    q[:, N:] = 3
    qt, st = q8.tile(q, s, N)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    qtd, std = q8.tile_device(qd, sd, N)
    torch.cuda.synchronize()
    assert np.array_equal(qtd.cpu().numpy(), qt) and np.array_equal(std.cpu().numpy(), st)


@pytest.mark.parametrize("tiled", [True, False])
@pytest.mark.parametrize("m", [1, 3, 16])
def test_gemv_parts(dev, m, tiled, tune):
    """Several weights of one activation in one call (q/k/v-style widths and a ragged one): each output against the
    oracle, and -- with the K split pinned, so that both calls sum in the same order -- bit-identical to the
    single-weight call on the same layout."""
    tune(ksplit=2)
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K = 2048
    Ns = [1024, 3000, 512, 40]
    x, _, _ = si.case(m, K, 32, 5100 + m)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    ws, devw = [], []
    for i, N in enumerate(Ns):
        _, q, s = si.case(1, K, N, 5200 + 10 * i)
        ws.append((q, s))
        qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
        if tiled:
            qd, sd = q8.tile_device(qd, sd, N)
        devw.append((qd, sd, N))
    ys = q8.gemv_parts(xd, devw, tiled=tiled, constant_weights=True)
    torch.cuda.synchronize()
    for i, N in enumerate(Ns):
        q, s = ws[i]
        y_o, a_o = oracle.gemv(x, q, s)
        got = ys[i].cpu().numpy()
        _assert_close(got, y_o, a_o, f"part {i} N={N}")
        assert np.all(got[:, N:] == 0.0)
        single = q8.gemv(xd, devw[i][0], devw[i][1], N, tiled=tiled).cpu().numpy()
        if tiled:
            assert np.array_equal(single.view(np.uint32), got.view(np.uint32))


@pytest.mark.parametrize("m", [1, 16])
@pytest.mark.parametrize("Ns", [(4096, 4096, 4096), (14336, 14336)])
def test_chain_parts_full_size_sampled(dev, m, Ns):
    """The decode chain's multi-projection launches as the benchmark makes them -- q/k/v (3 x 4096) and gate/up
    (2 x 14336) over K = 4096, tiled, constant weights, the planner's own K split -- at m = 1 and 16: 160 sampled
    columns of every part (tile edges, the last columns, random ones) against the oracle."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K = 4096
    x, _, _ = si.case(m, K, 32, si.case_seed(4, m, 90))
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    ws, devw = [], []
    for i, N in enumerate(Ns):
        _, q, s = si.case(1, K, N, si.case_seed(4, m, 91 + i))
        ws.append((q, s))
        devw.append(q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N) + (N,))
    ys = q8.gemv_parts(xd, devw, tiled=True, constant_weights=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(m + len(Ns))
    for i, N in enumerate(Ns):
        cols = np.unique(np.r_[0:16, 120:136, N - 16:N, rng.integers(0, N, 112)])
        y_o, a_o = oracle.gemv(x, ws[i][0], ws[i][1], cols)
        _assert_close(ys[i].cpu().numpy()[:, cols], y_o, a_o, f"m={m} part {i} of {Ns}")


# --------------------------------------------------------------------------------------------------------------------
# the gated pair (plan.rs `Launch::GemvGlu`, SwiGLU)
# --------------------------------------------------------------------------------------------------------------------

def _glu_bound(g_o, u_o, a_g, a_u, out_o):
    """The product's bound carried through silu(g) * u: |silu'| <= 1.1, so an error e_g in g moves the output by at
    most 1.1 |e_g| |u| and e_u by |silu(g)| |e_u|; plus a few fp32 ulps of the output for expf, the division and the
    product."""
    return (TOL * (1.1 * a_g * np.abs(u_o) + np.abs(oracle.silu(g_o)) * a_u) + 1.1 * TOL * TOL * a_g * a_u
            + 1e-6 * np.abs(out_o))


def _glu_run(torch, x, qg, sg, qu, su, N, want=("f32", "bf16")):
    import q8_block_quantized_gemv_gb300 as q8
    xd, qgd, sgd = _to_dev(torch, x, qg, sg)
    _, qud, sud = _to_dev(torch, x, qu, su)
    gate = q8.tile_device(qgd, sgd, N)
    up = q8.tile_device(qud, sud, N)
    out, outb = q8.gemv_glu(xd, gate, up, N, want=want)
    torch.cuda.synchronize()
    return (out.cpu().numpy() if out is not None else None,
            outb.view(torch.int16).cpu().numpy().view(np.uint16) if outb is not None else None)


def _glu_check(out, outb, x, qg, sg, qu, su, N, cols=None, what="", act=None):
    out_o, g_o, u_o, a_g, a_u = oracle.glu(x, qg, sg, qu, su, cols, act=act)
    got = out if cols is None else out[:, cols]
    err = np.abs(got.astype(np.float64) - out_o)
    bound = _glu_bound(g_o, u_o, a_g, a_u, out_o)
    bad = err > bound
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of bound; first at ({r},{c}): gpu {got[r, c]!r} "
                             f"oracle {out_o[r, c]!r} bound {bound[r, c]!r}")
    if outb is not None:
        assert np.array_equal(outb, si.f32_to_bf16_bits(out)), f"{what}: bf16 output is not the fp32 output rounded"
    if cols is None:
        assert np.all(out[:, N:] == 0.0) and (outb is None or np.all(outb[:, N:] == 0))


@pytest.mark.parametrize("m", [1, 2, 3, 8, 9, 16])
def test_glu_small(dev, m):
    """The gated pair on K = 1024, N = 1000 (8 column tiles, a ragged last one), every output: fp32 against the oracle
    within the carried bound, the bf16 copy equal to the fp32 output rounded to nearest even, pads exactly 0."""
    x, qg, sg = si.case(m, 1024, 1000, 2100 + m)
    _, qu, su = si.case(m, 1024, 1000, 2200 + m)
    out, outb = _glu_run(dev, x, qg, sg, qu, su, 1000)
    _glu_check(out, outb, x, qg, sg, qu, su, 1000, what=f"m={m}")


@pytest.mark.parametrize("m", [1, 2, 4, 8, 16])
def test_glu_ffn_gate_up_sampled(dev, m):
    """The FFN's gate and up projections (4096 x 14336) as one gated-pair launch, in the benchmark's configuration;
    384 sampled columns."""
    x, qg, sg = si.case(m, 4096, 14336, si.case_seed(2, m, 7))
    _, qu, su = si.case(m, 4096, 14336, si.case_seed(2, m, 8))
    rng = np.random.default_rng(50 + m)
    cols = np.unique(np.r_[0:32, 120:136, 248:264, 14304:14336, rng.integers(0, 14336, 290)])
    out, outb = _glu_run(dev, x, qg, sg, qu, su, 14336)
    _glu_check(out, outb, x, qg, sg, qu, su, 14336, cols, what=f"m={m}")


@pytest.mark.parametrize("ks", [1, 2, 3, 4])
@pytest.mark.parametrize("m", [2, 16])
def test_glu_every_cluster_split(dev, ks, m, tune):
    """Every K split of the gated pair's clusters (2 x ks CTAs): K = 4096 over 3 column tiles, every output."""
    tune(ksplit=ks)
    x, qg, sg = si.case(m, 4096, 300, 2300 + 10 * ks + m)
    _, qu, su = si.case(m, 4096, 300, 2400 + 10 * ks + m)
    out, outb = _glu_run(dev, x, qg, sg, qu, su, 300)
    _glu_check(out, outb, x, qg, sg, qu, su, 300, what=f"ks={ks} m={m}")


@pytest.mark.parametrize("want", [("f32",), ("bf16",)])
def test_glu_single_output_and_determinism(dev, want):
    """Either output alone is written correctly; repeated calls give identical bits."""
    x, qg, sg = si.case(5, 512, 200, 2501)
    _, qu, su = si.case(5, 512, 200, 2502)
    a = _glu_run(dev, x, qg, sg, qu, su, 200, want)
    b = _glu_run(dev, x, qg, sg, qu, su, 200, want)
    if want == ("f32",):
        assert a[1] is None and np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))
        _glu_check(a[0], None, x, qg, sg, qu, su, 200, what="f32 only")
    else:
        assert a[0] is None and np.array_equal(a[1], b[1])
        ref, _ = _glu_run(dev, x, qg, sg, qu, su, 200, ("f32",))
        assert np.array_equal(a[1], si.f32_to_bf16_bits(ref))


# --------------------------------------------------------------------------------------------------------------------
# residual add + RMS norm folded after a projection (plan.rs `Launch::Fold` / `gemv_norm_epilogue`)
# --------------------------------------------------------------------------------------------------------------------

def _norm_inputs(m, K, N, seed):
    x, q, s = si.case(m, K, N, seed)
    rng = np.random.default_rng(seed)
    Np = oracle.padded_n(N)
    res = np.zeros((m, Np), dtype=np.float32)
    res[:, :N] = rng.standard_normal((m, N)).astype(np.float32)
    gamma = (0.5 + rng.random(Np)).astype(np.float32)
    return x, q, s, res, gamma


def _norm_run(torch, x, q, s, res, gamma, eps, N, in_place=False):
    import q8_block_quantized_gemv_gb300 as q8
    xd, qd, sd = _to_dev(torch, x, q, s)
    qt, st = q8.tile_device(qd, sd, N)
    rd = torch.from_numpy(res).cuda()
    gd = torch.from_numpy(gamma).cuda()
    h, out = q8.gemv_residual_norm(xd, qt, st, N, rd, gd, eps, h=rd if in_place else None)
    torch.cuda.synchronize()
    return h.cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16)


def _norm_check(h, outb, x, q, s, res, gamma, eps, N, what="", act=None):
    h_o, out_o, _, a_o = oracle.residual_norm(x, q, s, res, gamma, eps, N, act=act)
    tol_h = TOL * a_o + 2.0 ** -24 * np.abs(h_o)
    bad = np.abs(h.astype(np.float64) - h_o) > tol_h
    assert not bad.any(), f"{what}: h out of bound at {np.argwhere(bad)[0]}"
    assert np.all(h[:, N:] == 0.0)
    bound = oracle.rmsnorm_bound(h_o, out_o, tol_h, gamma, eps, N)
    got = si.bf16_bits_to_f32(outb).astype(np.float64)
    bad = np.abs(got - out_o) > bound
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: out of bound at ({r},{c}): gpu {got[r, c]!r} oracle {out_o[r, c]!r}")
    assert np.all(outb[:, N:] == 0)


@pytest.mark.parametrize("m", [1, 2, 8, 16])
@pytest.mark.parametrize("K", [4096, 14336])
def test_residual_norm_hidden_width(dev, m, K):
    """The attention output (K = 4096) and FFN down (K = 14336) projections onto the 4096-wide residual stream,
    followed by the residual add and the following RMS norm; every output of h and of the normed bf16 rows."""
    x, q, s, res, gamma = _norm_inputs(m, K, 4096, 3100 + m + K)
    h, out = _norm_run(dev, x, q, s, res, gamma, 1e-6, 4096)
    _norm_check(h, out, x, q, s, res, gamma, 1e-6, 4096, what=f"m={m} K={K}")


@pytest.mark.parametrize("route", ["fold", "launch"])
@pytest.mark.parametrize("ks", [1, 2, 3, 8])
def test_residual_norm_every_cluster_split_and_in_place(dev, ks, route, tune):
    """Ragged width (N = 300, three column tiles) under each K split, with h written over the residual in place; the
    norm in the product's last CTA (tuning norm_fold = 1) and as a launch of its own."""
    tune(ksplit=ks)
    tune(norm_fold=int(route == "fold"))
    x, q, s, res, gamma = _norm_inputs(5, 1024, 300, 3200 + ks)
    h, out = _norm_run(dev, x, q, s, res.copy(), gamma, 0.5, 300, in_place=True)
    _norm_check(h, out, x, q, s, res, gamma, 0.5, 300, what=f"ks={ks}")


@pytest.mark.parametrize("route", ["fold", "launch"])
def test_residual_norm_counters_reused_and_deterministic(dev, route, tune):
    """More calls than the 64 completion counters, back to back: every call's result is bit-identical (the last CTA's
    fixed-order mean square does not depend on which CTA is last; nor, with the norm as a launch of its own, on
    anything but the row) and within the bound."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    tune(norm_fold=int(route == "fold"))
    x, q, s, res, gamma = _norm_inputs(3, 2048, 4096, 3300)
    xd, qd, sd = _to_dev(torch, x, q, s)
    qt, st = q8.tile_device(qd, sd, 4096)
    rd, gd = torch.from_numpy(res).cuda(), torch.from_numpy(gamma).cuda()
    outs = []
    for _ in range(70):
        h, out = q8.gemv_residual_norm(xd, qt, st, 4096, rd, gd, 1e-5, constant_weights=True)
        outs.append((h, out))
    torch.cuda.synchronize()
    h0, o0 = outs[0][0].cpu().numpy(), outs[0][1].view(torch.int16).cpu().numpy().view(np.uint16)
    for h, out in outs[1:]:
        assert np.array_equal(h.cpu().numpy().view(np.uint32), h0.view(np.uint32))
        assert np.array_equal(out.view(torch.int16).cpu().numpy().view(np.uint16), o0)
    _norm_check(h0, o0, x, q, s, res, gamma, 1e-5, 4096, what="repeated")


@pytest.mark.parametrize("m,K,N", [(1, 1024, 4096), (5, 1024, 300), (16, 2048, 5000), (33, 1024, 4096)])
def test_residual_norm_both_routes(dev, m, K, N, tune):
    """The norm in the product's last CTA (tuning norm_fold = 1) and as a launch of its own, one CTA per row
    (norm_fold = 0): ragged widths, a row wider than the 4096 columns a CTA keeps in registers (N = 5000), row
    groups (m = 33).  Both within the bound, one in place; h bit-identical (the same product and add)."""
    x, q, s, res, gamma = _norm_inputs(m, K, N, 3250 + m + N)
    got = {}
    for route in ("fold", "launch"):
        tune(norm_fold=int(route == "fold"))
        got[route] = _norm_run(dev, x, q, s, res.copy(), gamma, 1e-5, N, in_place=(route == "launch"))
        _norm_check(*got[route], x, q, s, res, gamma, 1e-5, N, what=f"m={m} N={N} route {route}")
    assert np.array_equal(got["fold"][0].view(np.uint32), got["launch"][0].view(np.uint32))
