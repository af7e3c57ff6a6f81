"""Parity of calls with more than 16 activation rows (the tiled storage's row groups of 16, up to 512 rows a call)
with the fp64 oracle, through every tiled entry point and both activation forms.

Bar as for the 16-row product: |y_gpu - y_oracle| <= 1e-5 * A per output; arg-max exact where planted; the gated
pair and the residual norm within their carried bounds.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si
from test_gpu_parity import _assert_close, _glu_check, _norm_check, _norm_inputs, _to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    return torch


def _tiled(torch, q, s, N):
    import q8_block_quantized_gemv_gb300 as q8
    return q8.tile_device(torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                          torch.from_numpy(np.ascontiguousarray(s)).cuda(), N)


def _x(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _act_from(torch, xq, xd):
    import q8_block_quantized_gemv_gb300 as q8
    m, K = xq.shape
    raw = np.concatenate([np.ascontiguousarray(xq).view(np.uint8).reshape(-1),
                          np.ascontiguousarray(xd, dtype=np.float32).view(np.uint8).reshape(-1)])
    return q8.QuantAct(torch.from_numpy(raw).cuda(), m, K)


@pytest.mark.parametrize("m", [17, 24, 31, 32, 33, 48, 64, 100, 128])
def test_product_rows(dev, m):
    """K = 1024, N = 1000 (a ragged last tile), every output, bf16 activations."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s = si.case(m, 1024, 1000, 5000 + m)
    y_o, a_o = oracle.gemv(x, q, s)
    qt, st = _tiled(torch, q, s, 1000)
    y = q8.gemv(_x(torch, x), qt, st, 1000, tiled=True)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    _assert_close(y, y_o, a_o, f"m={m}")
    assert np.all(y[:, 1000:] == 0.0)


@pytest.mark.parametrize("m,K,N", [(512, 4096, 4096), (300, 14336, 4096), (77, 4096, 14336)])
def test_product_prefill_chunks_sampled(dev, m, K, N):
    """Prefill-sized chunks up to the 512-row maximum on the decode layer's shapes; 160 sampled columns, every
    row."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s = si.case(m, K, N, 5100 + m)
    rng = np.random.default_rng(m)
    cols = np.unique(np.r_[0:16, 120:136, N - 16:N, rng.integers(0, N, 112)])
    y_o, a_o = oracle.gemv(x, q, s, cols)
    qt, st = _tiled(torch, q, s, N)
    y = q8.gemv(_x(torch, x), qt, st, N, tiled=True, constant_weights=True)
    torch.cuda.synchronize()
    _assert_close(y.cpu().numpy()[:, cols], y_o, a_o, f"m={m} K={K} N={N}")


@pytest.mark.parametrize("m", [17, 40, 128])
def test_quantized_activation_rows(dev, m):
    """The quantized numerics with row groups: K = 2048, N = 700."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s = si.case(m, 2048, 700, 5200 + m)
    xq, xd = oracle.quantize_act(x)
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s)
    qt, st = _tiled(torch, q, s, 700)
    y = q8.gemv(_act_from(torch, xq, xd), qt, st, 700, tiled=True)
    xa = q8.quantize_act(_x(torch, x))
    y2 = q8.gemv(xa, qt, st, 700, tiled=True)
    torch.cuda.synchronize()
    _assert_close(y.cpu().numpy(), y_o, a_o, f"m={m}")
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))


def test_parts_rows(dev):
    """q, k, v of 40 rows in one launch."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    m, K = 40, 1024
    x, _, _ = si.case(m, K, 32, 5300)
    ws, refs = [], []
    for i, N in enumerate([512, 128, 300]):
        _, q, s = si.case(1, K, N, 5301 + i)
        ws.append(_tiled(torch, q, s, N) + (N,))
        refs.append(oracle.gemv(x, q, s))
    ys = q8.gemv_parts(_x(torch, x), ws, tiled=True)
    torch.cuda.synchronize()
    for i, (y, (y_o, a_o)) in enumerate(zip(ys, refs)):
        _assert_close(y.cpu().numpy(), y_o, a_o, f"part {i}")


@pytest.mark.parametrize("m", [20, 64])
def test_argmax_rows(dev, m):
    """A planted winner in every row of a 32000-wide head: exact indices across the row groups."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, N = 1024, 32000
    x, q, s = si.case(m, K, N, 5400 + m)
    xf = si.bf16_bits_to_f32(x.reshape(-1)).reshape(m, K)
    win = (np.arange(m) * 4099 + 77) % N
    for r in range(m):
        q[:, win[r]] = np.where(xf[r] >= 0, 127, -127)
    cols = np.unique(np.r_[win, 0:32, N - 32:N])
    y_o, a_o = oracle.gemv(x, q, s, cols)
    qt, st = _tiled(torch, q, s, N)
    logits = torch.empty((m, oracle.padded_n(N)), dtype=torch.float32, device="cuda")
    idx = q8.gemv_argmax(_x(torch, x), qt, st, N, logits=logits, tiled=True)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), win)
    _assert_close(logits.cpu().numpy()[:, cols], y_o, a_o, f"m={m}")


@pytest.mark.parametrize("m", [17, 33, 64])
def test_glu_rows(dev, m):
    """The gated pair with row groups (K = 1024, N = 1000)."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, qg, sg = si.case(m, 1024, 1000, 5500 + m)
    _, qu, su = si.case(m, 1024, 1000, 5600 + m)
    out, outb = q8.gemv_glu(_x(torch, x), _tiled(torch, qg, sg, 1000), _tiled(torch, qu, su, 1000), 1000,
                            want=("f32", "bf16"))
    torch.cuda.synchronize()
    _glu_check(out.cpu().numpy(), outb.view(torch.int16).cpu().numpy().view(np.uint16), x, qg, sg, qu, su, 1000,
               what=f"m={m}")


@pytest.mark.parametrize("route", ["fold", "launch"])
@pytest.mark.parametrize("m,in_place", [(17, False), (40, True), (100, False)])
def test_residual_norm_rows(dev, m, in_place, route, tune):
    """The residual add and RMS norm with row groups: each group's last CTA norms its own rows (the one-launch fold,
    tuning norm_fold = 1), or a launch of its own norms every row (norm_fold = 0)."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    tune(norm_fold=int(route == "fold"))
    x, q, s, res, gamma = _norm_inputs(m, 1024, 4096, 5700 + m)
    qt, st = _tiled(torch, q, s, 4096)
    rd = torch.from_numpy(res.copy()).cuda()
    h, out = q8.gemv_residual_norm(_x(torch, x), qt, st, 4096, rd, torch.from_numpy(gamma).cuda(), 1e-6,
                                   h=rd if in_place else None)
    torch.cuda.synchronize()
    _norm_check(h.cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16), x, q, s, res, gamma, 1e-6,
                4096, what=f"m={m}")


def test_residual_norm_rows_counters_reused(dev, tune):
    """Calls of 200 rows (13 groups) back to back with the norm in each group's last CTA, more groups in all than the
    64 counters: identical bits."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    tune(norm_fold=1)
    m = 200
    x, q, s, res, gamma = _norm_inputs(m, 1024, 4096, 5800)
    qt, st = _tiled(torch, q, s, 4096)
    xd, rd, gd = _x(torch, x), torch.from_numpy(res).cuda(), torch.from_numpy(gamma).cuda()
    outs = [q8.gemv_residual_norm(xd, qt, st, 4096, rd, gd, 1e-5, constant_weights=True) for _ in range(7)]
    torch.cuda.synchronize()
    h0, o0 = outs[0][0].cpu().numpy(), outs[0][1].view(torch.int16).cpu().numpy().view(np.uint16)
    for h, o in outs[1:]:
        assert np.array_equal(h.cpu().numpy().view(np.uint32), h0.view(np.uint32))
        assert np.array_equal(o.view(torch.int16).cpu().numpy().view(np.uint16), o0)
    _norm_check(h0, o0, x, q, s, res, gamma, 1e-5, 4096, what="repeated")


def test_rows_match_single_groups(dev, tune):
    """Each 16-row group of a 50-row call gives the same bits as a call of those rows alone (one K split for both)."""
    tune(ksplit=4)
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    x, q, s = si.case(50, 2048, 600, 5900)
    qt, st = _tiled(torch, q, s, 600)
    y = q8.gemv(_x(torch, x), qt, st, 600, tiled=True).cpu().numpy()
    for r0 in range(0, 50, 16):
        r1 = min(r0 + 16, 50)
        yg = q8.gemv(_x(torch, np.ascontiguousarray(x[r0:r1])), qt, st, 600, tiled=True)
        torch.cuda.synchronize()
        yg = yg.cpu().numpy()
        if r1 - r0 > 8:  # the same 16-row kernel and K split: identical bits
            assert np.array_equal(yg.view(np.uint32), y[r0:r1].view(np.uint32)), (r0, r1)
        else:
            y_o, a_o = oracle.gemv(x[r0:r1], q, s)
            _assert_close(y[r0:r1], y_o, a_o, f"rows {r0}..{r1}")
