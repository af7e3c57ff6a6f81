"""The residual norm for callers that cannot allocate device memory: q8_gemv_residual_norm_noalloc, called through the
C ABI, against the existing entry point q8_gemv_residual_norm on the same inputs.

Some callers may not allocate device memory at all -- a real-time loop, a plugin whose host framework owns every
device buffer, a step that must not synchronise the device -- so this entry point keeps its only scratch, one
completion counter per group of 16 rows, in a static array of the library, clears it at every call and allocates
nothing.  The test runs it twice in a row on the same stream (the second call reuses the counters the first one
left) and compares both results with the existing entry point's: h exactly (the same product and add), the normed
bf16 rows bit for bit with the existing one-launch fold and within one bf16 unit of the default route (whose sums of
squares run in another order), and both against the oracle's bound.  This file is collected last.
"""
import ctypes

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


def _inputs(m, K, N, seed):
    x, q, s = si.case(m, K, N, seed)
    rng = np.random.default_rng(seed)
    Np = oracle.padded_n(N)
    res = np.zeros((m, Np), dtype=np.float32)
    res[:, :N] = rng.standard_normal((m, N)).astype(np.float32)
    gamma = (0.5 + rng.random(Np)).astype(np.float32)
    return x, q, s, res, gamma


def _bf16_ulp(v):
    """One unit in the last place of bf16 at each |v| (8 significant bits), for normal values."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def _oracle_bound(h, outb, x, q, s, res, gamma, eps, N):
    """h within the product's bound plus one fp32 rounding of the add; the normed rows within the bound of
    oracle.rmsnorm_bound (half a bf16 unit, the h error carried through the norm, the fp32 arithmetic's roundings)."""
    h_o, out_o, _, a_o = oracle.residual_norm(x, q, s, res, gamma, eps, N)
    tol_h = TOL * a_o + 2.0 ** -24 * np.abs(h_o)
    assert np.all(np.abs(h.astype(np.float64) - h_o) <= tol_h)
    bound = oracle.rmsnorm_bound(h_o, out_o, tol_h, gamma, eps, N)
    assert np.all(np.abs(si.bf16_bits_to_f32(outb).astype(np.float64) - out_o) <= bound)


@pytest.mark.parametrize("m,K,N", [(3, 1024, 4096), (40, 2048, 1000)])
def test_noalloc_matches_residual_norm(dev, m, K, N, tune):
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    lib = q8.lib()
    eps = 1e-5
    x, q, s, res, gamma = _inputs(m, K, N, 7700 + m)
    Np = oracle.padded_n(N)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N)
    rd = torch.from_numpy(res).cuda()
    gd = torch.from_numpy(gamma).cuda()

    # the existing entry point: its default route (the norm as a launch of its own) and its one-launch fold
    h_ref, o_ref = q8.gemv_residual_norm(xd, qt, st, N, rd, gd, eps)
    tune(norm_fold=1)
    h_fold, o_fold = q8.gemv_residual_norm(xd, qt, st, N, rd, gd, eps)
    tune(norm_fold=0)

    # the entry point that allocates nothing, twice in a row through the C ABI
    stream = torch.cuda.current_stream().cuda_stream
    got = []
    for _ in range(2):
        h = torch.full((m, Np), float("nan"), dtype=torch.float32, device="cuda")
        o = torch.full((m, Np), -1.0, dtype=torch.bfloat16, device="cuda")
        status = lib.q8_gemv_residual_norm_noalloc(xd.data_ptr(), qt.data_ptr(), st.data_ptr(), rd.data_ptr(),
                                                   gd.data_ptr(), ctypes.c_float(eps), h.data_ptr(), o.data_ptr(),
                                                   m, K, N, q8.FLAG_TILED, stream)
        assert status == 0, q8.status_string(status)
        got.append((h, o))
    torch.cuda.synchronize()

    h_ref = h_ref.cpu().numpy()
    ob_ref = o_ref.view(torch.int16).cpu().numpy().view(np.uint16)
    ob_fold = o_fold.view(torch.int16).cpu().numpy().view(np.uint16)
    for h, o in got:
        hh = h.cpu().numpy()
        ob = o.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(hh.view(np.uint32), h_ref.view(np.uint32))
        assert np.array_equal(ob, ob_fold)
        a, b = si.bf16_bits_to_f32(ob).astype(np.float64), si.bf16_bits_to_f32(ob_ref).astype(np.float64)
        assert np.all(np.abs(a - b) <= _bf16_ulp(b))
        assert np.all(ob[:, N:] == 0)
        _oracle_bound(hh, ob, x, q, s, res, gamma, eps, N)
