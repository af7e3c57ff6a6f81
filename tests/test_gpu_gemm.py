"""Parity of the prefill GEMM (tcgen05; tiled storage, bf16 activations, m >= 128 rows) with the fp64 oracle.

An integer case (small integer activations, s = 1) must come out exact: every product and every partial sum is an
integer below 2^24, so any slip in the operands' shared-memory layouts shows as a wrong integer.  The rest is judged
by the product's bound, |y_gpu - y_oracle| <= 1e-5 * A, and compared with the row-group path on the same inputs.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si
from test_gpu_parity import _assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gemm_whatever_the_width(tune):
    """Narrow weights would otherwise take the row groups; these tests are about the GEMM."""
    tune(gemm=1)


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    return torch


def _run(torch, x, q, s, N):
    import q8_block_quantized_gemv_gb300 as q8
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    qt, st = q8.tile_device(torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                            torch.from_numpy(np.ascontiguousarray(s)).cuda(), N)
    y = q8.gemv(xd, qt, st, N, tiled=True)
    torch.cuda.synchronize()
    assert q8.device_fault(clear=True) == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("m,K,N", [(128, 32, 128), (128, 64, 256), (130, 96, 128), (200, 1024, 384)])
def test_integer_case_is_exact(dev, m, K, N):
    """x small integers, q int8, s = 1: y is the integer matmul, bit for bit."""
    rng = np.random.default_rng(m + K + N)
    xi = rng.integers(-8, 9, size=(m, K)).astype(np.float32)
    x = si.f32_to_bf16_bits(xi).reshape(m, K)
    q = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    s = np.ones((K // 32, N), dtype=np.float32)
    y = _run(dev, x, q, s, N)
    exact = xi.astype(np.int64) @ q.astype(np.int64)
    bad = np.argwhere(y != exact)
    assert bad.size == 0, f"{len(bad)} wrong; first {bad[0]}: gpu {y[tuple(bad[0])]} exact {exact[tuple(bad[0])]}"


@pytest.mark.parametrize("m,K,N", [(128, 1024, 1000), (131, 512, 300), (128, 2048, 128), (129, 1024, 640),
                                   (256, 4096, 512), (512, 1024, 1024), (140, 14336, 256)])
def test_matches_oracle(dev, m, K, N):
    """The workload's value distributions, ragged rows and columns; every output within the bound, pads exactly 0."""
    x, q, s = si.case(m, K, N, 6000 + m + K + N)
    y_o, a_o = oracle.gemv(x, q, s)
    y = _run(dev, x, q, s, N)
    _assert_close(y, y_o, a_o, f"m={m} K={K} N={N}")
    assert np.all(y[:, N:] == 0.0)


def test_same_as_row_groups_within_bound(dev, tune):
    """The GEMM and the row groups (tuning gemm = 0) agree with the oracle on the same 160-row call."""
    x, q, s = si.case(160, 2048, 500, 6100)
    y_o, a_o = oracle.gemv(x, q, s)
    y_g = _run(dev, x, q, s, 500)
    tune(gemm=0)
    y_r = _run(dev, x, q, s, 500)
    _assert_close(y_g, y_o, a_o, "gemm")
    _assert_close(y_r, y_o, a_o, "row groups")


def test_parts(dev):
    """q, k and v of a 128-row chunk in one GEMM launch."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    m, K = 128, 1024
    x, _, _ = si.case(m, K, 32, 6200)
    ws, refs = [], []
    for i, N in enumerate([512, 128, 384]):
        _, q, s = si.case(1, K, N, 6201 + i)
        ws.append(q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N) + (N,))
        refs.append(oracle.gemv(x, q, s))
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()
    ys = q8.gemv_parts(xd, ws, tiled=True)
    torch.cuda.synchronize()
    for i, (y, (y_o, a_o)) in enumerate(zip(ys, refs)):
        _assert_close(y.cpu().numpy(), y_o, a_o, f"part {i}")


def test_deterministic(dev):
    x, q, s = si.case(160, 2048, 640, 6300)
    y1 = _run(dev, x, q, s, 640)
    y2 = _run(dev, x, q, s, 640)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("ks", [1, 2, 3, 4])
def test_every_k_split(dev, ks, tune):
    """Each cluster split of K (ranks summed through distributed shared memory in rank order): K = 4096 (128 blocks,
    uneven thirds), 130 rows, 3 column tiles, every output; the integer case stays exact."""
    tune(ksplit=ks)
    x, q, s = si.case(130, 4096, 300, 6400 + ks)
    y_o, a_o = oracle.gemv(x, q, s)
    y = _run(dev, x, q, s, 300)
    _assert_close(y, y_o, a_o, f"ks={ks}")
    assert np.all(y[:, 300:] == 0.0)
    rng = np.random.default_rng(ks)
    xi = rng.integers(-8, 9, size=(128, 1024)).astype(np.float32)
    qi = rng.integers(-127, 128, size=(1024, 256)).astype(np.int8)
    yi = _run(dev, si.f32_to_bf16_bits(xi).reshape(128, 1024), qi, np.ones((32, 256), np.float32), 256)
    assert np.array_equal(yi, (xi.astype(np.int64) @ qi.astype(np.int64)).astype(np.float32))
