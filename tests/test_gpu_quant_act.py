"""Parity of the quantized-activation path (q8_quantize_act and every product under Q8_FLAG_Q8_ACT) with the oracle.

The quantizer's codes and scales are integer / binary32 decisions taken in the same precision on both sides (IEEE fp32
quotients, rounding half away from zero), so they must match bit for bit.  The products are judged by the product's
bound, |y_gpu - y_oracle| <= 1e-5 * A with A = sum_b |s d| sum_i |xq q|; where s = d = 1 and the integer sums stay
below 2^24 the result must be the exact integer.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si
from test_gpu_parity import TOL, _assert_close, _glu_check, _norm_check, _norm_inputs, _to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    return torch


def _x_dev(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _quantize_dev(torch, x):
    """GPU quantized form of bf16 bits x -> (xq int8, xd fp32) numpy arrays and the QuantAct."""
    import q8_block_quantized_gemv_gb300 as q8
    xa = q8.quantize_act(_x_dev(torch, x))
    torch.cuda.synchronize()
    return xa.values().cpu().numpy(), xa.scales().cpu().numpy(), xa


def _act_from(torch, xq, xd):
    """A QuantAct holding given codes and scales (the oracle's), for product parity independent of the quantizer."""
    import q8_block_quantized_gemv_gb300 as q8
    m, K = xq.shape
    raw = np.concatenate([np.ascontiguousarray(xq).view(np.uint8).reshape(-1),
                          np.ascontiguousarray(xd, dtype=np.float32).view(np.uint8).reshape(-1)])
    return q8.QuantAct(torch.from_numpy(raw).cuda(), m, K)


def _kinds(m, K, seed):
    """bf16 activations whose blocks cycle through: N(0,1); x 1e30; x 1e-30; x 1e-38 (subnormal d); bf16 subnormals
    only; zeros and -0; d = 1 ties (127 and j + 1/2 values); one inf; one NaN; a single nonzero value."""
    rng = np.random.default_rng(seed)
    nb = K // 32
    x = np.zeros((m, K), dtype=np.uint16)
    for b in range(nb):
        kind = b % 10
        g = rng.standard_normal((m, 32)).astype(np.float32)
        if kind == 0:
            v = si.f32_to_bf16_bits(g).reshape(m, 32)
        elif kind in (1, 2, 3):
            f = {1: 1e30, 2: 1e-30, 3: 1e-38}[kind]
            v = si.f32_to_bf16_bits((g * np.float32(f)).astype(np.float32)).reshape(m, 32)
        elif kind == 4:
            v = rng.integers(1, 0x80, size=(m, 32)).astype(np.uint16) | np.where(g < 0, 0x8000, 0).astype(np.uint16)
        elif kind == 5:
            v = np.where(g < 0, np.uint16(0x8000), np.uint16(0)).astype(np.uint16)
        elif kind == 6:
            j = rng.integers(-127, 127, size=(m, 32)).astype(np.float32) + np.float32(0.5)
            j[:, 0] = 127.0
            v = si.f32_to_bf16_bits(j).reshape(m, 32)
        elif kind == 7:
            v = si.f32_to_bf16_bits(g).reshape(m, 32)
            v[m - 1, 11] = np.uint16(0x7F80 | (0x8000 if b % 20 == 7 else 0))
        elif kind == 8:
            v = si.f32_to_bf16_bits(g).reshape(m, 32)
            v[0, 30] = np.uint16(0x7FC0)
        else:
            v = np.zeros((m, 32), dtype=np.uint16)
            v[:, 13] = si.f32_to_bf16_bits(g[:, 13]).reshape(m)
        x[:, 32 * b:32 * b + 32] = v
    return x


@pytest.mark.parametrize("m,K", [(1, 320), (3, 640), (16, 4096), (300, 1024), (16, 14336)])
def test_quantize_act_bit_exact(dev, m, K):
    """Codes and scales equal the oracle's bit for bit (NaN scales where the oracle has NaN), every value kind."""
    x = _kinds(m, K, 40 + m + K)
    xq, xd, _ = _quantize_dev(dev, x)
    xq_o, xd_o = oracle.quantize_act(x)
    assert np.array_equal(xq, xq_o)
    nan = np.isnan(xd_o)
    assert np.array_equal(np.isnan(xd), nan)
    assert np.array_equal(xd[~nan].view(np.uint32), xd_o[~nan].view(np.uint32))


def test_quantize_act_sign_symmetry(dev):
    """-x gives the negated codes and the same scales (rounding half away from zero is symmetric)."""
    x, _, _ = si.case(7, 2048, 32, 41)
    xq, xd, _ = _quantize_dev(dev, x)
    xqn, xdn, _ = _quantize_dev(dev, x ^ np.uint16(0x8000))
    assert np.array_equal(xqn.astype(np.int16), -xq.astype(np.int16)) and np.array_equal(xdn, xd)


def _product(torch, act, q, s, N):
    import q8_block_quantized_gemv_gb300 as q8
    qd, sd = torch.from_numpy(np.ascontiguousarray(q)).cuda(), torch.from_numpy(np.ascontiguousarray(s)).cuda()
    qt, st = q8.tile_device(qd, sd, N)
    y = q8.gemv(act, qt, st, N, tiled=True)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("m", list(range(1, 17)))
def test_product_1024(dev, m):
    """K = N = 1024, every row count: the product of the oracle's quantized form, and the full chain (GPU quantizer,
    then the product), both within the bound; the chain equals the product of the oracle's form bit for bit."""
    x, q, s = si.case(m, 1024, 1024, si.case_seed(0, m, 5))
    xq, xd = oracle.quantize_act(x)
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s)
    y1 = _product(dev, _act_from(dev, xq, xd), q, s, 1024)
    _assert_close(y1, y_o, a_o, f"m={m}")
    _, _, xa = _quantize_dev(dev, x)
    y2 = _product(dev, xa, q, s, 1024)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("m,K,N", [(1, 32, 1), (16, 32, 1), (3, 32, 33), (5, 64, 2), (16, 14336, 32), (1, 14336, 64),
                                   (8, 4096, 96), (3, 5120, 40), (3, 5120, 3000), (2, 256, 100000), (9, 768, 40)])
def test_product_edge_and_ragged_shapes(dev, m, K, N):
    """One block; one column; narrow N with deep K (the cluster split); ragged widths; a very wide N (sampled)."""
    x, q, s = si.case(m, K, N, 750 + m + K + N)
    xq, xd = oracle.quantize_act(x)
    cols = None if N <= 6144 else np.r_[0:64, N - 64:oracle.padded_n(N)]
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s, cols)
    y = _product(dev, _act_from(dev, xq, xd), q, s, N)
    _assert_close(y if cols is None else y[:, cols], y_o, a_o, f"m={m} K={K} N={N}")
    if cols is None:
        assert np.all(y[:, N:] == 0.0)


@pytest.mark.parametrize("m", [1, 8, 16])
def test_integer_sums_are_exact(dev, m):
    """s = d = 1, K = 1024 (every partial sum below 2^24): each output is the exact integer dot product."""
    rng = np.random.default_rng(60 + m)
    K, N = 1024, 384
    xq = rng.integers(-127, 128, size=(m, K)).astype(np.int8)
    q = np.zeros((K, N), dtype=np.int8)
    q[:] = rng.integers(-127, 128, size=(K, N))
    s = np.ones((K // 32, N), dtype=np.float32)
    xd = np.ones((m, K // 32), dtype=np.float32)
    y = _product(dev, _act_from(dev, xq, xd), q, s, N)
    exact = xq.astype(np.int64) @ q.astype(np.int64)
    assert np.array_equal(y.astype(np.int64), exact) and np.all(y == exact)


@pytest.mark.parametrize("K,N", [(4096, 14336), (14336, 4096)])
@pytest.mark.parametrize("m", [1, 4, 16])
def test_ffn_projections_sampled(dev, K, N, m):
    """FFN up/gate and down at full size under the quantized numerics (GPU quantizer), 384 sampled columns."""
    x, q, s = si.case(m, K, N, si.case_seed(2, m, 5 if K > N else 6))
    xq, xd, xa = _quantize_dev(dev, x)
    rng = np.random.default_rng(m + 3)
    cols = np.unique(np.r_[0:32, 120:136, 248:264, N - 32:N, rng.integers(0, N, 256)])
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s, cols)
    y = _product(dev, xa, q, s, N)
    _assert_close(y[:, cols], y_o, a_o, f"K={K} N={N} m={m}")


def test_nonfinite_blocks_poison_their_rows(dev):
    """A block holding inf or NaN has d = NaN, so every real output of its row is NaN (the pad columns stay exactly
    0); the other rows meet the bound."""
    x, q, s = si.case(4, 512, 200, 61)
    x[1, 70] = np.uint16(0x7F80)
    x[3, 500] = np.uint16(0xFFC0)
    xq, xd, xa = _quantize_dev(dev, x)
    y = _product(dev, xa, q, s, 200)
    assert np.all(np.isnan(y[[1, 3], :200])) and np.all(y[:, 200:] == 0.0)
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s)
    _assert_close(y[[0, 2]], y_o[[0, 2]], a_o[[0, 2]], "finite rows")


@pytest.mark.parametrize("m", [1, 4, 16])
def test_argmax_head(dev, m):
    """The tied-head shape (K = 4096, N = 32000 here) with a planted winner per row: exact index; the logits within
    the bound."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, N = 4096, 32000
    x, q, s = si.case(m, K, N, 770 + m)
    xq, xd = oracle.quantize_act(x)
    win = (np.arange(m) * 7919 + 123) % N
    for r in range(m):
        # the winner's column equals the row's codes' signs at full scale: its logit is far above every other
        q[:, win[r]] = np.where(xq[r] >= 0, 127, -127)
    cols = np.unique(np.r_[win, 0:64, N - 64:N])
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s, cols)
    qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
    qt, st = q8.tile_device(qd, sd, N)
    logits = torch.empty((m, oracle.padded_n(N)), dtype=torch.float32, device="cuda")
    idx = q8.gemv_argmax(_act_from(torch, xq, xd), qt, st, N, logits=logits, tiled=True)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), win)
    _assert_close(logits.cpu().numpy()[:, cols], y_o, a_o, f"m={m}")


def test_parts(dev):
    """q, k and v of one quantized activation in one launch; each part within the bound."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    m, K = 5, 2048
    x, _, _ = si.case(m, K, 32, 780)
    xq, xd = oracle.quantize_act(x)
    act = _act_from(torch, xq, xd)
    ws, refs = [], []
    for i, N in enumerate([1024, 256, 300]):
        _, q, s = si.case(1, K, N, 781 + i)
        qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N)
        ws.append((qt, st, N))
        refs.append(oracle.gemv_q8act(xq, xd, q, s))
    ys = q8.gemv_parts(act, ws, tiled=True)
    torch.cuda.synchronize()
    for i, (y, (y_o, a_o)) in enumerate(zip(ys, refs)):
        _assert_close(y.cpu().numpy(), y_o, a_o, f"part {i}")


@pytest.mark.parametrize("m", [1, 8, 16])
def test_glu(dev, m):
    """The gated pair over a quantized activation (K = 1024, N = 1000): silu(g) u within the carried bound, the bf16
    copy the fp32 output rounded."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, qg, sg = si.case(m, 1024, 1000, 2600 + m)
    _, qu, su = si.case(m, 1024, 1000, 2700 + m)
    xq, xd = oracle.quantize_act(x)
    _, qgd, sgd = _to_dev(torch, x, qg, sg)
    _, qud, sud = _to_dev(torch, x, qu, su)
    out, outb = q8.gemv_glu(_act_from(torch, xq, xd), q8.tile_device(qgd, sgd, 1000), q8.tile_device(qud, sud, 1000),
                            1000, want=("f32", "bf16"))
    torch.cuda.synchronize()
    _glu_check(out.cpu().numpy(), outb.view(torch.int16).cpu().numpy().view(np.uint16), x, qg, sg, qu, su, 1000,
               what=f"m={m}", act=(xq, xd))


@pytest.mark.parametrize("m,K", [(1, 4096), (16, 14336)])
def test_residual_norm(dev, m, K):
    """The residual add and RMS norm after a projection of a quantized activation (hidden width 4096)."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s, res, gamma = _norm_inputs(m, K, 4096, 3400 + m)
    xq, xd = oracle.quantize_act(x)
    qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), 4096)
    h, out = q8.gemv_residual_norm(_act_from(torch, xq, xd), qt, st, 4096, torch.from_numpy(res).cuda(),
                                   torch.from_numpy(gamma).cuda(), 1e-6)
    torch.cuda.synchronize()
    _norm_check(h.cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), x, q, s, res, gamma, 1e-6,
                4096, what=f"m={m} K={K}", act=(xq, xd))


def test_deterministic(dev):
    """Repeated calls give identical bits."""
    x, q, s = si.case(11, 4096, 1000, 790)
    _, _, xa = _quantize_dev(dev, x)
    y1 = _product(dev, xa, q, s, 1000)
    y2 = _product(dev, xa, q, s, 1000)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


# --------------------------------------------------------------------------------------------------------------------
# producers that write the quantized form in their epilogue (the gated pair, the residual norm)
# --------------------------------------------------------------------------------------------------------------------

def _assert_form_of(torch, qa, bf16_out, what):
    """The epilogue's quantized form equals q8_quantize_act's rule (the oracle) applied to its own bf16 output."""
    bits = bf16_out.view(torch.int16).cpu().numpy().view(np.uint16)
    xq_o, xd_o = oracle.quantize_act(bits)
    xq, xd = qa.values().cpu().numpy(), qa.scales().cpu().numpy()
    assert np.array_equal(xq, xq_o), what
    nan = np.isnan(xd_o)
    assert np.array_equal(np.isnan(xd), nan) and np.array_equal(xd[~nan].view(np.uint32),
                                                                xd_o[~nan].view(np.uint32)), what


@pytest.mark.parametrize("ks", [1, 2, 3, 4])
@pytest.mark.parametrize("m", [1, 8, 16, 40])
def test_glu_writes_its_quantized_form(dev, m, ks, tune):
    """The gated pair's out_q8 is the quantized form of its bf16 output, for every K split (32-column slices) and row
    groups; the bf16 output itself stays within the bound."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    tune(ksplit=ks)
    x, qg, sg = si.case(m, 1024, 1000, 2800 + m)
    _, qu, su = si.case(m, 1024, 1000, 2900 + m)
    _, qgd, sgd = _to_dev(torch, x, qg, sg)
    _, qud, sud = _to_dev(torch, x, qu, su)
    out, outb, qa = q8.gemv_glu(_x_dev(torch, x), q8.tile_device(qgd, sgd, 1000), q8.tile_device(qud, sud, 1000),
                                1000, want=("f32", "bf16", "q8"))
    torch.cuda.synchronize()
    _glu_check(out.cpu().numpy(), outb.view(torch.int16).cpu().numpy().view(np.uint16), x, qg, sg, qu, su, 1000,
               what=f"m={m} ks={ks}")
    _assert_form_of(torch, qa, outb, f"m={m} ks={ks}")


@pytest.mark.parametrize("route", ["fold", "launch"])
@pytest.mark.parametrize("m", [1, 16, 40])
def test_residual_norm_writes_its_quantized_form(dev, m, route, tune):
    """The residual norm's out_q8 is the quantized form of its bf16 rows; asked for alone, it is the same bytes.  The
    norm in the product's last CTA (tuning norm_fold = 1) and as a launch of its own."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    tune(norm_fold=int(route == "fold"))
    x, q, s, res, gamma = _norm_inputs(m, 2048, 4096, 3500 + m)
    qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), 4096)
    xd, gd = _x_dev(torch, x), torch.from_numpy(gamma).cuda()
    h, outb, qa = q8.gemv_residual_norm(xd, qt, st, 4096, torch.from_numpy(res).cuda(), gd, 1e-6,
                                        want=("bf16", "q8"))
    h2, none, qa2 = q8.gemv_residual_norm(xd, qt, st, 4096, torch.from_numpy(res).cuda(), gd, 1e-6, want=("q8",))
    torch.cuda.synchronize()
    assert none is None
    _norm_check(h.cpu().numpy(), outb.view(torch.int16).cpu().numpy().view(np.uint16), x, q, s, res, gamma, 1e-6,
                4096, what=f"m={m}")
    _assert_form_of(torch, qa, outb, f"m={m}")
    assert torch.equal(qa.buf, qa2.buf) and torch.equal(h, h2)


def test_fused_form_feeds_the_next_projection(dev):
    """The gated pair's quantized output read by the down projection (Q8_FLAG_Q8_ACT) gives the same bits as
    quantizing its bf16 output with q8_quantize_act first."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    m, D, F = 4, 1024, 2048
    x, qg, sg = si.case(m, D, F, 3600)
    _, qu, su = si.case(m, D, F, 3601)
    _, qd, sd = si.case(m, F, D, 3602)
    _, qgd, sgd = _to_dev(torch, x, qg, sg)
    _, qud, sud = _to_dev(torch, x, qu, su)
    down = q8.tile_device(torch.from_numpy(qd).cuda(), torch.from_numpy(sd).cuda(), D)
    _, hb, hq = q8.gemv_glu(_x_dev(torch, x), q8.tile_device(qgd, sgd, F), q8.tile_device(qud, sud, F), F,
                            want=("bf16", "q8"))
    y1 = q8.gemv(hq, down[0], down[1], D, tiled=True)
    y2 = q8.gemv(q8.quantize_act(hb), down[0], down[1], D, tiled=True)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
