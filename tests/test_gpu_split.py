"""The two-launch split of plain products (q8_api.cu `plan_split`): a store or arg-max product of at most 16 rows whose
column tiles do not fill the SMs evenly runs as a first launch over one tile per SM (or over whole waves) and a
second over the remaining tiles with K split across a cluster.

Checked here, through the C ABI, against the fp64 oracle under the product's bound (|y - y_oracle| <= 1e-5 * A):
  - the planner's choice (q8_plan_launches) for the decode chain's launches and for the shapes below;
  - both forms (split on and off), every output, for both split cases, tiled and row-major weights, every kernel family
    (1, 2, 4 and 16 rows), and the arg-max;
  - repeated calls are bit-identical (the split is fixed by the shape);
  - stream order around the pair: a later launch that reads the split product's output (the residual of a residual
    norm) or overwrites its input (the norm's bf16 output written over the product's activation) sees both launches
    complete, eagerly and replayed from a CUDA graph.
"""
import numpy as np
import pytest

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

TOL = 1e-5

# (K, Ns) of the two split cases on a GPU of 152 SMs (two CTAs per SM for 1 and 9..16 rows, one for 2..8):
#   co:    160 tiles, between the SMs and the resident slots: 152 tiles one CTA per SM, then 8 tiles with K split
#   waves: 330 tiles, above the slots: the whole waves, then the rest with K split
CASES = {"co": (512, (10240, 10240)), "waves": (256, (42240,))}


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q8_block_quantized_gemv_gb300 import build
    build.build()
    return torch


@pytest.fixture(scope="module")
def sms(dev):
    return dev.cuda.get_device_properties(0).multi_processor_count


def _x_dev(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _weights(torch, K, Ns, seed, tiled):
    import q8_block_quantized_gemv_gb300 as q8
    host, devw = [], []
    for i, N in enumerate(Ns):
        _, q, s = si.case(1, K, N, seed + i)
        host.append((q, s))
        qd, sd = torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda()
        if tiled:
            qd, sd = q8.tile_device(qd, sd, N)
        devw.append((qd, sd, N))
    return host, devw


def _assert_close(y_gpu, y_o, a_o, what=""):
    err = np.abs(y_gpu.astype(np.float64) - y_o)
    bad = err > TOL * a_o
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs out of bound; first at ({r},{c}): gpu {y_gpu[r, c]!r} "
                             f"oracle {y_o[r, c]!r} A {a_o[r, c]!r}")


def test_planner_splits_the_chains_uneven_launches(dev, sms):
    """On 152 SMs, where every stream kernel runs two CTAs per SM: the gate/up pair (224 tiles) and the tied head
    (1002 tiles) split in two at every row count and on both storages; q/k/v, o and down keep one launch (their K
    split already fills the SMs).  Switched off, or under a forced K split, every call is one launch."""
    import q8_block_quantized_gemv_gb300 as q8
    if sms != 152:
        pytest.skip("expectations for a 152-SM GB300")
    shapes = {"qkv": (4096, (4096, 4096, 4096)), "o": (4096, (4096,)), "gateup": (4096, (14336, 14336)),
              "down": (14336, (4096,)), "head": (4096, (128256,))}
    for m in (1, 2, 4, 8, 16):
        for tiled in (True, False):
            for name, (K, Ns) in shapes.items():
                got = q8.plan_launches(m, K, Ns, tiled=tiled)
                assert got == (2 if name in ("gateup", "head") else 1), (m, tiled, name, got)
    with q8.tuning(split=0):
        assert q8.plan_launches(16, 4096, (14336, 14336)) == 1 and q8.plan_launches(1, 4096, (128256,)) == 1
    with q8.tuning(ksplit=2):
        assert q8.plan_launches(16, 4096, (14336, 14336)) == 1
    assert q8.plan_launches(17, 4096, (14336, 14336)) == 1  # row groups: one launch


@pytest.mark.parametrize("tiled", [True, False], ids=["tiled", "rowmajor"])
@pytest.mark.parametrize("m", [1, 2, 4, 16])
@pytest.mark.parametrize("case", sorted(CASES))
def test_split_products_match_the_oracle(dev, sms, case, m, tiled, tune):
    """Every output of both split cases, split and unsplit, against the oracle; the split form twice, bit-identical."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, Ns = CASES[case]
    x, _, _ = si.case(m, K, 32, si.case_seed(11, m, len(Ns)))
    host, devw = _weights(torch, K, Ns, si.case_seed(12, m, K), tiled)
    xd = _x_dev(torch, x)
    if sms == 152:
        assert q8.plan_launches(m, K, Ns, tiled=tiled) == 2, (case, m)
    runs = []
    for split in (1, 1, 0):
        tune(split=split)
        ys = q8.gemv_parts(xd, devw, tiled=tiled, constant_weights=True)
        torch.cuda.synchronize()
        runs.append([y.cpu().numpy() for y in ys])
    for i, (q, s) in enumerate(host):
        N = Ns[i]
        y_o, a_o = oracle.gemv(x, q, s)
        for r, label in ((0, "split"), (2, "one launch")):
            _assert_close(runs[r][i][:, :N], y_o[:, :N], a_o[:, :N], f"{case} m={m} part {i} {label}")
            assert np.all(runs[r][i][:, N:] == 0.0)
        assert np.array_equal(runs[0][i].view(np.uint32), runs[1][i].view(np.uint32)), "split not reproducible"


@pytest.mark.parametrize("m", [1, 16])
def test_split_argmax_matches_the_oracle(dev, m):
    """The arg-max over the waves case (330 tiles): both launches fold into the row keys; logits and indices against
    the oracle."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, (N,) = CASES["waves"]
    x, q, s = si.case(m, K, N, si.case_seed(13, m))
    y_o, a_o = oracle.gemv(x, q, s)
    qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N)
    logits = torch.full((m, oracle.padded_n(N)), float("nan"), dtype=torch.float32, device="cuda")
    idx = q8.gemv_argmax(_x_dev(torch, x), qt, st, N, logits=logits, tiled=True, constant_weights=True)
    torch.cuda.synchronize()
    lg, ix = logits.cpu().numpy(), idx.cpu().numpy()
    _assert_close(lg[:, :N], y_o[:, :N], a_o[:, :N], f"m={m} logits")
    for r in range(m):
        best = int(oracle.argmax(y_o[r:r + 1], N)[0])
        close = (y_o[r, best] - y_o[r, :N]) <= TOL * (a_o[r, best] + a_o[r, :N])
        close[best] = True
        assert (ix[r] == best) if close.sum() == 1 else close[ix[r]], (r, ix[r], best)


def _norm_after(torch, m, K2, N, seed):
    """A residual norm over a fresh product (K2 x N, tiled): h = residual + x2 . W2."""
    import q8_block_quantized_gemv_gb300 as q8
    x2, q2, s2 = si.case(m, K2, N, seed)
    qt, st = q8.tile_device(torch.from_numpy(q2).cuda(), torch.from_numpy(s2).cuda(), N)
    gamma = torch.ones(oracle.padded_n(N), dtype=torch.float32, device="cuda")
    return (x2, q2, s2), (_x_dev(torch, x2), qt, st, gamma)


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("m", [1, 16])
def test_launch_after_the_pair_reads_its_output(dev, sms, m, graph):
    """A residual norm whose residual is the split product's output (the up part, written by both launches): its h
    must hold the finished product.  The output starts as NaN before every run, so a read before either launch had
    written would show."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, Ns = 4096, (10240, 10240)  # 160 tiles: the co case
    x, _, _ = si.case(m, K, 32, si.case_seed(14, m))
    host, devw = _weights(torch, K, Ns, si.case_seed(15, m), True)
    xd = _x_dev(torch, x)
    if sms == 152:
        assert q8.plan_launches(m, K, Ns) == 2
    Np = oracle.padded_n(Ns[1])
    ys = [torch.empty((m, oracle.padded_n(N)), dtype=torch.float32, device="cuda") for N in Ns]
    (x2, q2, s2), (x2d, q2t, s2t, gamma) = _norm_after(torch, m, 256, Ns[1], si.case_seed(16, m))
    h = torch.empty((m, Np), dtype=torch.float32, device="cuda")
    outb = torch.empty((m, Np), dtype=torch.bfloat16, device="cuda")

    def step():
        for y in ys:
            y.fill_(float("nan"))
        q8.gemv_parts(xd, devw, ys=ys, tiled=True, constant_weights=True)
        q8.gemv_residual_norm(x2d, q2t, s2t, Ns[1], ys[1], gamma, 1e-6, h=h, out_bf16=outb, constant_weights=True)

    if graph:
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
    else:
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    y_o, a_o = oracle.gemv(x, host[1][0], host[1][1])
    y2_o, a2_o = oracle.gemv(x2, q2, s2)
    hh = h.cpu().numpy().astype(np.float64)
    N = Ns[1]
    bound = TOL * (a_o + a2_o) + 2.0 ** -23 * np.abs(y_o + y2_o)
    bad = ~(np.abs(hh[:, :N] - (y_o + y2_o)[:, :N]) <= bound[:, :N])
    assert not bad.any(), f"h wrong at {np.argwhere(bad)[0]} ({bad.sum()} outputs)"


@pytest.mark.parametrize("graph", [False, True], ids=["eager", "graph"])
@pytest.mark.parametrize("m", [1, 16])
def test_launch_after_the_pair_overwrites_its_input(dev, sms, m, graph):
    """A residual norm whose bf16 output is the split product's activation: it may overwrite x only after both launches
    have read it.  x is restored before every run; the product must equal the oracle's over the original x."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    K, Ns = 4096, (20480,)  # 160 tiles: the co case; the norm's width is K
    x, _, _ = si.case(m, K, 32, si.case_seed(17, m))
    host, devw = _weights(torch, K, Ns, si.case_seed(18, m), True)
    x0 = _x_dev(torch, x)
    xd = x0.clone()
    if sms == 152:
        assert q8.plan_launches(m, K, Ns) == 2
    y = torch.empty((m, oracle.padded_n(Ns[0])), dtype=torch.float32, device="cuda")
    res = torch.zeros((m, K), dtype=torch.float32, device="cuda")
    _, (x2d, q2t, s2t, gamma) = _norm_after(torch, m, 1024, K, si.case_seed(19, m))
    h = torch.empty((m, K), dtype=torch.float32, device="cuda")

    def step():
        xd.copy_(x0)
        q8.gemv_parts(xd, devw, ys=[y], tiled=True, constant_weights=True)
        q8.gemv_residual_norm(x2d, q2t, s2t, K, res, gamma, 1e-6, h=h, out_bf16=xd, constant_weights=True)

    if graph:
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(3):
            g.replay()
    else:
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    y_o, a_o = oracle.gemv(x, host[0][0], host[0][1])
    _assert_close(y.cpu().numpy()[:, :Ns[0]], y_o[:, :Ns[0]], a_o[:, :Ns[0]], f"m={m} product over the original x")
    assert not torch.equal(xd, x0), "the norm did not write its output over x"


@pytest.mark.parametrize("m", [1, 4, 16])
def test_split_gated_pair_matches_the_oracle(dev, sms, m, tune):
    """The gated pair over 80 column tiles (160 CTAs, two a tile): split in two on 152 SMs (one tile pair per two SMs,
    then the rest with K split over clusters of 2 x ks), every fp32 output against the oracle's silu(g) * u within the
    carried bound, the bf16 copy the fp32 output rounded; split and unsplit both, the split twice bit-identical."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    from test_gpu_parity import _glu_check, _to_dev
    K, N = 512, 10240
    x, qg, sg = si.case(m, K, N, si.case_seed(20, m))
    _, qu, su = si.case(1, K, N, si.case_seed(21, m))
    xd, qgd, sgd = _to_dev(torch, x, qg, sg)
    _, qud, sud = _to_dev(torch, x, qu, su)
    gate, up = q8.tile_device(qgd, sgd, N), q8.tile_device(qud, sud, N)
    if sms == 152:
        assert q8.plan_glu_launches(m, K, N) == 2, m
    runs = []
    for split in (1, 1, 0):
        tune(split=split)
        if split == 0:
            assert q8.plan_glu_launches(m, K, N) == 1
        out, outb = q8.gemv_glu(xd, gate, up, N, want=("f32", "bf16"), constant_weights=True)
        torch.cuda.synchronize()
        runs.append((out.cpu().numpy(), outb.view(torch.int16).cpu().numpy().view(np.uint16)))
    for r, label in ((0, "split"), (2, "one launch")):
        _glu_check(runs[r][0], runs[r][1], x, qg, sg, qu, su, N, what=f"m={m} {label}")
    assert np.array_equal(runs[0][0].view(np.uint32), runs[1][0].view(np.uint32)), "split not reproducible"


@pytest.mark.parametrize("m", [1, 2, 4, 16])
@pytest.mark.parametrize("case", sorted(CASES))
def test_split_quantized_activations_match_the_oracle(dev, sms, case, m, tune):
    """Both split cases over quantized activations (Q8_FLAG_Q8_ACT: the dp4a CUDA-core kernel at 1 and 2 rows, the
    integer-exact tensor-core kernels above): every output against the oracle's quantized product, split and
    unsplit, the split twice bit-identical."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    from test_gpu_quant_act import _act_from
    K, Ns = CASES[case]
    x, _, _ = si.case(m, K, 32, si.case_seed(22, m, len(Ns)))
    xq, xd = oracle.quantize_act(x)
    host, devw = _weights(torch, K, Ns, si.case_seed(23, m, K), True)
    xa = _act_from(torch, xq, xd)
    if sms == 152:
        assert q8.plan_launches(m, K, Ns, q8_act=True) == 2, (case, m)
    runs = []
    for split in (1, 1, 0):
        tune(split=split)
        ys = q8.gemv_parts(xa, devw, tiled=True, constant_weights=True)
        torch.cuda.synchronize()
        runs.append([y.cpu().numpy() for y in ys])
    for i, (q, s) in enumerate(host):
        N = Ns[i]
        y_o, a_o = oracle.gemv_q8act(xq, xd, q, s)
        for r, label in ((0, "split"), (2, "one launch")):
            _assert_close(runs[r][i][:, :N], y_o[:, :N], a_o[:, :N], f"{case} m={m} part {i} {label}")
            assert np.all(runs[r][i][:, N:] == 0.0)
        assert np.array_equal(runs[0][i].view(np.uint32), runs[1][i].view(np.uint32)), "split not reproducible"


@pytest.mark.parametrize("m", [1, 16])
def test_split_argmax_quantized_activations(dev, sms, m):
    """The arg-max over the waves case with quantized activations and a planted winner per row (one in each launch of
    the split): exact indices, the logits within the bound."""
    torch = dev
    import q8_block_quantized_gemv_gb300 as q8
    from test_gpu_quant_act import _act_from
    K, (N,) = CASES["waves"]
    x, q, s = si.case(m, K, N, si.case_seed(24, m))
    xq, xd = oracle.quantize_act(x)
    # winners spread over the first launch's tiles and the second's (tiles 304 .. 329 hold columns 38912 ..)
    win = np.where(np.arange(m) % 2 == 0, (np.arange(m) * 7919 + 123) % 38912, 38912 + (np.arange(m) * 131) % 3328)
    for r in range(m):
        # the winner's column: the row's code signs at full scale and the weight's largest block scale (with K = 256,
        # eight blocks, a random column with large scales could otherwise beat a planted one with small ones)
        q[:, win[r]] = np.where(xq[r] >= 0, 127, -127)
        s[:, win[r]] = s.max()
    y_o, a_o = oracle.gemv_q8act(xq, xd, q, s)
    assert np.array_equal(oracle.argmax(y_o, N), win)
    if sms == 152:
        assert q8.plan_launches(m, K, (N,), q8_act=True) == 2
    qt, st = q8.tile_device(torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), N)
    logits = torch.empty((m, oracle.padded_n(N)), dtype=torch.float32, device="cuda")
    idx = q8.gemv_argmax(_act_from(torch, xq, xd), qt, st, N, logits=logits, tiled=True, constant_weights=True)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), win)
    _assert_close(logits.cpu().numpy()[:, :N], y_o[:, :N], a_o[:, :N], f"m={m}")
