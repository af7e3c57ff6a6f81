"""The C ABI on the CPU: the library loads and exports every declared symbol; host entry points agree with the oracle;
device entry points reject bad arguments before touching CUDA (no compute call runs here)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth_inputs as si
import q8_block_quantized_gemv_gb300 as q8
from q8_block_quantized_gemv_gb300 import build as q8build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8_gemv.h")


@pytest.fixture(scope="module")
def lib():
    q8build.build()
    return q8.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(q8_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 9
    for name in names:
        assert hasattr(lib, name), name
    assert set(names) == set(q8.SIGNATURES), "binding signatures and header disagree"


def test_padded_n(lib):
    for n, want in [(1, 32), (32, 32), (33, 64), (40, 64), (3000, 3008), (6144, 6144), (128256, 128256),
                    (0, -1), (-7, -1), (2**31 - 1, -1)]:
        assert q8.padded_n(n) == want, n
        if n > 0 and want > 0:
            assert want == oracle.padded_n(n)


def test_status_strings(lib):
    for code in range(6):
        assert q8.status_string(code)
    assert q8.status_string(99) == "unknown status"
    assert lib.q8_version() >= 10000


# --------------------------------------------------------------------------------------------------------------------
# host entry points against the oracle
# --------------------------------------------------------------------------------------------------------------------

@pytest.mark.parametrize("K,N,seed", [(256, 40, 1), (1024, 96, 2), (64, 1, 3)])
def test_quantize_matches_oracle(lib, K, N, seed):
    _, q, s = si.case(1, K, N, seed)
    w = oracle.dequantize(q[:, :N], s[:, :N])
    gq, gs = q8.quantize(w)
    oq, os_ = oracle.quantize(w)
    assert np.array_equal(gq[:, :N], oq) and np.array_equal(gs[:, :N], os_)
    assert np.all(gq[:, N:] == 0) and np.all(gs[:, N:] == 0)
    assert np.array_equal(gq, q) and np.array_equal(gs, s)


def test_quantize_rejections_match_oracle(lib):
    _, q, s = si.case(1, 64, 4, 18)
    w = oracle.dequantize(q[:, :4], s[:, :4])
    w[5, 2] = np.nextafter(w[5, 2], np.inf)
    assert oracle.quantize(w) is None
    with pytest.raises(q8.Q8Error) as e:
        q8.quantize(w)
    assert e.value.status == 4
    one = np.zeros((32, 1))
    one[0, 0] = 1.0                      # d = 1/127 is not an fp32
    assert oracle.quantize(one) is None
    with pytest.raises(q8.Q8Error):
        q8.quantize(one)
    d = 2.0 ** -10
    half = np.zeros((32, 1))
    half[0, 0], half[1, 0] = 127 * d, 63.5 * d
    with pytest.raises(q8.Q8Error):
        q8.quantize(half)
    for bad in (np.nan, np.inf):
        w2 = np.zeros((32, 2))
        w2[3, 1] = bad
        with pytest.raises(q8.Q8Error):
            q8.quantize(w2)
    zero = np.zeros((64, 3))
    gq, gs = q8.quantize(zero)
    assert not gq.any() and not gs.any()


def test_quantize_shape_errors(lib):
    with pytest.raises(q8.Q8Error) as e:
        q8.quantize(np.zeros((33, 2)))
    assert e.value.status == 2


def _blocks(q, s, N):
    K = q.shape[0]
    nb = K // 32
    rec = np.zeros((N, nb, 36), dtype=np.uint8)
    rec[:, :, :4] = s[:, :N].T.astype("<f4").copy().view(np.uint8).reshape(N, nb, 4)
    rec[:, :, 4:] = q[:, :N].T.reshape(N, nb, 32).view(np.uint8)
    return rec.tobytes()


@pytest.mark.parametrize("K,N", [(128, 40), (64, 3000), (32, 1)])
def test_repack_matches_oracle(lib, K, N):
    _, q, s = si.case(1, K, N, K + N)
    blk = _blocks(q, s, N)
    gq, gs = q8.repack(blk, K, N)
    oq, os_ = oracle.repack(blk, K, N)
    assert np.array_equal(gq, oq) and np.array_equal(gs, os_)
    assert np.array_equal(gq, q) and np.array_equal(gs, s)


def test_repack_rejects(lib):
    _, q, s = si.case(1, 64, 8, 5)
    q2 = q.copy()
    q2[7, 3] = -128
    with pytest.raises(q8.Q8Error) as e:
        q8.repack(_blocks(q2, s, 8), 64, 8)
    assert e.value.status == 4
    s2 = s.copy()
    s2[1, 2] = np.inf
    with pytest.raises(q8.Q8Error):
        q8.repack(_blocks(q, s2, 8), 64, 8)


def _f16_blocks(q, d_bits, N):
    K = q.shape[0]
    rec = np.zeros((N, K // 32, 34), dtype=np.uint8)
    rec[:, :, 0:2] = np.ascontiguousarray(d_bits.T).astype("<u2").view(np.uint8).reshape(N, K // 32, 2)
    rec[:, :, 2:] = np.ascontiguousarray(q.T).reshape(N, K // 32, 32).view(np.uint8)
    return rec.tobytes()


@pytest.mark.parametrize("K,N", [(32, 1), (96, 40), (512, 300)])
def test_repack_f16_matches_oracle(lib, K, N):
    """GGML-style blocks: every finite binary16 scale class (normals, subnormals, zeros of both signs) widened as the
    oracle (numpy's float16) widens it, bit for bit; the values in place."""
    rng = np.random.default_rng(K + N)
    q = rng.integers(-127, 128, size=(K, N)).astype(np.int8)
    d_bits = rng.integers(0, 0x7C00, size=(K // 32, N)).astype(np.uint16)
    d_bits |= (rng.integers(0, 2, size=d_bits.shape) << 15).astype(np.uint16)
    special = np.array([0x0001, 0x83FF, 0x0000, 0x8000], dtype=np.uint16)
    flat = d_bits.reshape(-1)
    flat[:min(4, flat.size)] = special[:min(4, flat.size)]
    blk = _f16_blocks(q, d_bits, N)
    gq, gs = q8.repack(blk, K, N, scale="f16")
    oq, os_ = oracle.repack_f16(blk, K, N)
    assert np.array_equal(gq, oq) and np.array_equal(gs.view(np.uint32), os_.view(np.uint32))


def test_repack_f16_every_half_pattern(lib):
    """All 63,488 finite binary16 patterns as scales: the library's widening equals numpy's for every one."""
    pats = np.array([b for b in range(0x10000) if (b >> 10) & 0x1F != 0x1F], dtype=np.uint16)
    N = 128
    nb = -(-pats.size // N)
    d_bits = np.zeros(nb * N, dtype=np.uint16)
    d_bits[:pats.size] = pats
    d_bits = d_bits.reshape(N, nb).T
    q = np.ones((32 * nb, N), dtype=np.int8)
    gq, gs = q8.repack(_f16_blocks(q, d_bits, N), 32 * nb, N, scale="f16")
    want = d_bits.view(np.float16).astype(np.float32)
    assert np.array_equal(gs[:, :N].view(np.uint32), want.view(np.uint32))


def test_repack_f16_rejects(lib):
    q = np.ones((64, 8), dtype=np.int8)
    d = np.full((2, 8), 0x3C00, dtype=np.uint16)
    q2 = q.copy()
    q2[5, 1] = -128
    for qq, dd in ((q2, d), (q, np.where(np.arange(16).reshape(2, 8) == 9, 0x7C00, d).astype(np.uint16)),
                   (q, np.where(np.arange(16).reshape(2, 8) == 3, 0xFE00, d).astype(np.uint16))):
        with pytest.raises(q8.Q8Error) as e:
            q8.repack(_f16_blocks(qq, dd, 8), 64, 8, scale="f16")
        assert e.value.status == 4


# --------------------------------------------------------------------------------------------------------------------
# device entry points: argument errors come back before any CUDA call
# --------------------------------------------------------------------------------------------------------------------

A16 = 0x10000      # fake, 16-byte aligned addresses: never dereferenced, the calls fail their checks first
B16 = 0x20000
C16 = 0x30000
D16 = 0x40000


@pytest.mark.parametrize("args,want", [
    ((None, B16, C16, D16, 1, 32, 32), 1),          # null x
    ((A16, None, C16, D16, 1, 32, 32), 1),          # null q
    ((A16, B16, None, D16, 1, 32, 32), 1),          # null s
    ((A16, B16, C16, None, 1, 32, 32), 1),          # null y
    ((A16, B16, C16, D16, 0, 32, 32), 2),           # m = 0
    ((A16, B16, C16, D16, 17, 32, 32), 2),          # m > 16
    ((A16, B16, C16, D16, 1, 0, 32), 2),            # K = 0
    ((A16, B16, C16, D16, 1, 48, 32), 2),           # K % 32 != 0
    ((A16, B16, C16, D16, 1, 32, 0), 2),            # N = 0
    ((A16, B16, C16, D16, 1, 32, 2**31 - 1), 2),    # Np overflows
    ((A16 + 2, B16, C16, D16, 1, 32, 32), 3),       # misaligned x
    ((A16, B16 + 8, C16, D16, 1, 32, 32), 3),       # misaligned q
    ((A16, B16, C16 + 4, D16, 1, 32, 32), 3),       # misaligned s
    ((A16, B16, C16, D16 + 4, 1, 32, 32), 3),       # misaligned y
    ((A16, B16, C16, B16, 1, 32, 32), 1),           # y overlaps q
])
def test_gemv_argument_errors(lib, args, want):
    assert lib.q8_gemv(*args, None) == want
    assert lib.q8_gemv_ex(*args, 0, 0, None) == want


def test_gemv_ex_rejects_unknown_variant(lib):
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 32, 4, 0, None) == 1
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 32, -1, 0, None) == 1
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 32, 0, 4, None) == 1       # unknown flag


@pytest.mark.parametrize("args,want", [
    ((A16, B16, C16, None, D16, 1, 32, 32), 1),     # null idx
    ((A16, B16, C16, D16 + 4, None, 1, 32, 32), 3),  # misaligned idx
    ((A16, B16, C16, D16, 0x50004, 1, 32, 32), 3),  # misaligned logits
    ((A16, B16, C16, D16, None, 0, 32, 32), 2),
    ((A16, B16, C16, D16, None, 1, 31, 32), 2),
    ((A16, B16, C16, D16, B16, 1, 32, 32), 1),      # logits overlap q
])
def test_argmax_argument_errors(lib, args, want):
    assert lib.q8_gemv_argmax(*args, None) == want


def test_device_fault_rejects_null(lib):
    assert lib.q8_device_fault(None, 0) == 1


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    x = torch.zeros((1, 32), dtype=torch.bfloat16)
    q = torch.zeros((32, 32), dtype=torch.int8)
    s = torch.zeros((1, 32), dtype=torch.float32)
    with pytest.raises(ValueError):
        q8.gemv(x, q, s, 32)


# --------------------------------------------------------------------------------------------------------------------
# the tiled storage order (q8_tile): checked against the index map written out independently here
# --------------------------------------------------------------------------------------------------------------------

def _tile_reference(q, s, N):
    """The documented tiled order, written as the index map of the header: the byte of weight row 32b + 16s + 4u + k
    in column 128t + 8(4h + w) + g sits at 512(4s + h) + 16(4g + u) + 4w + k of unit (t, b), stored as q + 128;
    columns >= N hold byte 128 (q = 0) and scale 0."""
    K = q.shape[0]
    nb, Nt = K // 32, -(-N // 128) * 128
    T = Nt // 128
    qt = np.full((T, nb, 4096), 128, dtype=np.uint8)
    st = np.zeros((T, nb, 128), dtype=np.float32)
    for t in range(T):
        for b in range(nb):
            for r in range(32):
                step, u, k = r // 16, (r % 16) // 4, r % 4
                for c in range(128):
                    n = 128 * t + c
                    if n < N:
                        j, g = c // 8, c % 8
                        at = 512 * (4 * step + j // 4) + 16 * (4 * g + u) + 4 * (j % 4) + k
                        qt[t, b, at] = int(q[32 * b + r, n]) + 128
            for c in range(128):
                if 128 * t + c < N:
                    st[t, b, c] = s[b, 128 * t + c]
    return qt.reshape(-1).view(np.int8), st.reshape(-1)


@pytest.mark.parametrize("K,N", [(64, 40), (96, 300), (32, 128)])
def test_tile_host_matches_index_map(lib, K, N):
    _, q, s = si.case(1, K, N, 77 + N)
    q[:, N:] = 5          # dirty pads must not reach the tiled form
    qt, st = q8.tile(q, s, N)
    rq, rs = _tile_reference(q, s, N)
    assert np.array_equal(qt, rq) and np.array_equal(st, rs)
    assert q8.tiled_n(N) == -(-N // 128) * 128


def test_tile_argument_errors(lib):
    assert lib.q8_tile(None, C16, 32, 32, A16, B16) == 1
    assert lib.q8_tile(A16, C16, 33, 32, A16, B16) == 2
    assert lib.q8_tile_device(A16 + 1, C16, 32, 32, B16, D16, None) == 3
    assert lib.q8_tiled_n(0) == -1 and lib.q8_tiled_n(1) == 128 and lib.q8_tiled_n(129) == 256
    # tiled flag only with the pipelined kernel
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 32, 1, 2, None) == 1
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 32, 3, 2, None) == 1
    assert lib.q8_gemv_argmax_ex(A16, B16, C16, D16, None, 1, 32, 32, 4, None) == 1


def test_gemv_glu_argument_errors(lib):
    G, GS, U, US = B16, C16, 0x50000, 0x60000
    F32, BF = D16, 0x70000
    assert lib.q8_gemv_glu(None, G, GS, U, US, F32, BF, 1, 32, 64, 2, None) == 1      # null x
    assert lib.q8_gemv_glu(A16, G, GS, None, US, F32, BF, 1, 32, 64, 2, None) == 1    # null up weight
    assert lib.q8_gemv_glu(A16, G, GS, U, US, None, None, 1, 32, 64, 2, None) == 1    # no output
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF, 1, 32, 64, 0, None) == 1       # not tiled
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF, 1, 32, 64, 8 | 2, None) == 1   # unknown flag
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF, 513, 32, 64, 2, None) == 2     # m > 512 (tiled)
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF, 1, 33, 64, 2, None) == 2       # K % 32
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF, 1, 32, 0, 2, None) == 2        # N = 0
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32 + 4, BF, 1, 32, 64, 2, None) == 3   # misaligned out
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, BF + 2, 1, 32, 64, 2, None) == 3   # misaligned bf16 out
    assert lib.q8_gemv_glu(A16, G, GS, U, US, F32, F32, 1, 32, 64, 2, None) == 1      # outputs overlap
    assert lib.q8_gemv_glu(A16, G, GS, U, US, A16, None, 1, 32, 64, 2, None) == 1     # output over x


def test_gemv_residual_norm_argument_errors(lib):
    import ctypes
    R, G, H, O = 0x50000, 0x60000, 0x70000, 0x80000
    f = ctypes.c_float
    ok = (A16, B16, C16, R, G, f(1e-6), H, O, 2, 64, 96, 2, None)
    def call(**kw):
        args = list(ok)
        names = ["x", "q", "s", "res", "gamma", "eps", "h", "out", "m", "K", "N", "flags", "stream"]
        for k, v in kw.items():
            args[names.index(k)] = v
        return lib.q8_gemv_residual_norm(*args)
    assert call(x=None) == 1
    assert call(res=None) == 1
    assert call(gamma=None) == 1
    assert call(h=None) == 1
    assert call(out=None) == 1
    assert call(flags=0) == 1                  # not tiled
    assert call(flags=2 | 8) == 1              # unknown flag
    assert call(eps=f(-1.0)) == 1
    assert call(eps=f(float("inf"))) == 1
    assert call(eps=f(float("nan"))) == 1
    assert call(m=513) == 2
    assert call(K=33) == 2
    assert call(N=0) == 2
    assert call(h=H + 4) == 3                  # misaligned h
    assert call(out=O + 2) == 3                # misaligned bf16 out
    assert call(res=R + 2) == 3                # misaligned residual
    assert call(h=R + 16) == 1                 # h partly over the residual
    assert call(out=H) == 1                    # out over h
    assert call(h=A16) == 1                    # h over x


def test_gemv_parts_argument_errors(lib):
    import ctypes
    P = q8._Part
    good = (P * 2)(P(B16, C16, D16, 64), P(0x50000, 0x60000, 0x70000, 96))
    assert lib.q8_gemv_parts(None, ctypes.cast(good, ctypes.c_void_p), 2, 1, 32, 0, None) == 1   # null x
    assert lib.q8_gemv_parts(A16, None, 2, 1, 32, 0, None) == 1                                  # null parts
    assert lib.q8_gemv_parts(A16, ctypes.cast(good, ctypes.c_void_p), 0, 1, 32, 0, None) == 1     # no parts
    assert lib.q8_gemv_parts(A16, ctypes.cast(good, ctypes.c_void_p), 9, 1, 32, 0, None) == 1     # too many
    assert lib.q8_gemv_parts(A16, ctypes.cast(good, ctypes.c_void_p), 2, 17, 32, 0, None) == 2    # m > 16
    assert lib.q8_gemv_parts(A16, ctypes.cast(good, ctypes.c_void_p), 2, 1, 33, 0, None) == 2     # K % 32
    assert lib.q8_gemv_parts(A16, ctypes.cast(good, ctypes.c_void_p), 2, 1, 32, 8, None) == 1     # unknown flag
    bad = (P * 2)(P(B16, C16, D16, 64), P(0x50000, 0x60000, 0x70004, 96))
    assert lib.q8_gemv_parts(A16, ctypes.cast(bad, ctypes.c_void_p), 2, 1, 32, 0, None) == 3      # misaligned y
    clash = (P * 2)(P(B16, C16, D16, 64), P(0x50000, 0x60000, D16, 96))
    assert lib.q8_gemv_parts(A16, ctypes.cast(clash, ctypes.c_void_p), 2, 1, 32, 0, None) == 1    # outputs overlap
    zero = (P * 1)(P(B16, C16, D16, 0))
    assert lib.q8_gemv_parts(A16, ctypes.cast(zero, ctypes.c_void_p), 1, 1, 32, 0, None) == 2     # N = 0


def test_act_bytes(lib):
    assert lib.q8_act_bytes(1, 32) == 36
    assert lib.q8_act_bytes(3, 64) == 3 * 64 + 3 * 2 * 4
    assert lib.q8_act_bytes(16, 14336) == 16 * 14336 + 16 * 448 * 4
    assert lib.q8_act_bytes(0, 32) == -1 and lib.q8_act_bytes(1, 0) == -1 and lib.q8_act_bytes(1, 48) == -1


def test_quantize_act_argument_errors(lib):
    XA = 0x80000
    assert lib.q8_quantize_act(None, XA, 1, 32, None) == 1
    assert lib.q8_quantize_act(A16, None, 1, 32, None) == 1
    assert lib.q8_quantize_act(A16, XA, 0, 32, None) == 2
    assert lib.q8_quantize_act(A16, XA, 1, 33, None) == 2
    assert lib.q8_quantize_act(A16, XA, 1, 0, None) == 2
    assert lib.q8_quantize_act(A16 + 8, XA, 1, 32, None) == 3
    assert lib.q8_quantize_act(A16, XA + 4, 1, 32, None) == 3
    assert lib.q8_quantize_act(A16, A16 + 48, 1, 32, None) == 1     # output inside x (64 bytes)
    assert lib.q8_quantize_act(A16 + 16, A16, 1, 32, None) == 1     # x inside the output (36 bytes)


def test_quantized_activation_flag_rules(lib):
    """Q8_FLAG_Q8_ACT (4) needs Q8_FLAG_TILED on every product entry point; an output over the quantized form
    (whose size is q8_act_bytes, not 2 m K) is an overlap."""
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 1, 32, 64, 0, 4, None) == 1
    assert lib.q8_gemv_argmax_ex(A16, B16, C16, D16, None, 1, 32, 64, 4, None) == 1
    assert lib.q8_gemv_glu(A16, B16, C16, 0x50000, 0x60000, D16, None, 1, 32, 64, 4, None) == 1
    # m = 1, K = 64: 72 bytes of quantized form, so y at x + 64 overlaps it
    assert lib.q8_gemv_ex(A16, B16, C16, A16 + 64, 1, 64, 64, 0, 4 | 2, None) == 1
    assert lib.q8_gemv_parts(A16, None, 1, 1, 64, 4 | 2, None) == 1


def test_row_limits(lib):
    """m > 16 needs the tiled storage (row groups of 16, up to Q8_MAX_CHUNK = 512 rows); 513 rows never."""
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 17, 32, 64, 0, 0, None) == 2
    assert lib.q8_gemv_ex(A16, B16, C16, D16, 513, 32, 64, 0, 2, None) == 2
    assert lib.q8_gemv_argmax_ex(A16, B16, C16, D16, None, 17, 32, 64, 0, None) == 2
    assert lib.q8_gemv_argmax_ex(A16, B16, C16, D16, None, 513, 32, 64, 2, None) == 2


def test_quantized_output_argument_errors(lib):
    """The producers' _ex entry points: at least one output; out_q8 16-byte aligned and apart from the others."""
    import ctypes
    G, GS, U, US = B16, C16, 0x50000, 0x60000
    assert lib.q8_gemv_glu_ex(A16, G, GS, U, US, None, None, None, 1, 32, 64, 2, None) == 1
    assert lib.q8_gemv_glu_ex(A16, G, GS, U, US, None, None, 0x70004, 1, 32, 64, 2, None) == 3
    assert lib.q8_gemv_glu_ex(A16, G, GS, U, US, None, 0x70000, 0x70000, 1, 32, 64, 2, None) == 1
    f = ctypes.c_float
    R, GM, H = 0x50000, 0x60000, 0x70000
    assert lib.q8_gemv_residual_norm_ex(A16, B16, C16, R, GM, f(1e-6), H, None, None, 2, 64, 96, 2, None) == 1
    assert lib.q8_gemv_residual_norm_ex(A16, B16, C16, R, GM, f(1e-6), H, None, 0x80008, 2, 64, 96, 2, None) == 3
    assert lib.q8_gemv_residual_norm_ex(A16, B16, C16, R, GM, f(1e-6), H, 0x80000, 0x80000, 2, 64, 96, 2,
                                        None) == 1
    assert lib.q8_gemv_residual_norm_ex(A16, B16, C16, R, GM, f(1e-6), H, None, H, 2, 64, 96, 2, None) == 1


@pytest.mark.parametrize("env,want", [(None, (0, -1, 0, 1)), ({"Q8_NORM_LAUNCH": "0"}, (0, -1, 1, 1)),
                                      ({"Q8_NORM_LAUNCH": "1", "Q8_KSPLIT": "3", "Q8_GEMM": "1"}, (3, 1, 0, 1)),
                                      ({"Q8_KSPLIT": "9", "Q8_GEMM": "0", "Q8_SPLIT": "0"}, (0, 0, 0, 0)),
                                      ({"Q8_SPLIT": "1"}, (0, -1, 0, 1))])
def test_tuning_starts_from_the_environment(env, want):
    """The planner overrides start from Q8_KSPLIT, Q8_GEMM, Q8_NORM_LAUNCH and Q8_SPLIT, read once in a fresh process
    (an out-of-range K split is ignored); the binding's launch count of a residual-norm call follows the route."""
    import subprocess
    import sys
    e = {k: v for k, v in os.environ.items() if k not in ("Q8_NORM_LAUNCH", "Q8_KSPLIT", "Q8_GEMM", "Q8_SPLIT")}
    e.update(env or {})
    code = ("import q8_block_quantized_gemv_gb300 as q8; "
            "print(q8.get_tuning('ksplit'), q8.get_tuning('gemm'), q8.get_tuning('norm_fold'), "
            "q8.get_tuning('split'), q8.residual_norm_launches())")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=e, cwd=ROOT, timeout=120)
    assert out.returncode == 0, out.stderr
    got = tuple(int(v) for v in out.stdout.split())
    assert got == want + (1 if want[2] == 1 else 2,)


def test_tuning_set_get_and_rejects(lib):
    saved = [lib.q8_get_tuning(o) for o in range(4)]
    try:
        for opt, ok, bad in ((0, (0, 1, 8), (-1, 9)), (1, (-1, 0, 1), (-2, 2)), (2, (0, 1), (-1, 2)),
                             (3, (0, 1), (-1, 2))):
            for v in ok:
                assert lib.q8_set_tuning(opt, v) == 0 and lib.q8_get_tuning(opt) == v
            for v in bad:
                assert lib.q8_set_tuning(opt, v) == 1 and lib.q8_get_tuning(opt) == ok[-1]
        assert lib.q8_set_tuning(4, 0) == 1 and lib.q8_set_tuning(-1, 0) == 1
        assert lib.q8_get_tuning(4) == -2 and lib.q8_get_tuning(-1) == -2
        with q8.tuning(norm_fold=1, ksplit=5):
            assert q8.residual_norm_launches() == 1 and q8.get_tuning("ksplit") == 5
    finally:
        for o, v in enumerate(saved):
            lib.q8_set_tuning(o, v)
    assert [lib.q8_get_tuning(o) for o in range(4)] == saved


def test_plan_launches_argument_errors(lib):
    """q8_plan_launches rejects, before any device query, what q8_gemv_parts would reject; valid sizes give a count
    (1 or 2) on a GPU and -Q8_ERR_CUDA without one."""
    ns = (ctypes.c_int * 2)(4096, 4096)
    p = ctypes.cast(ns, ctypes.c_void_p)
    call = lib.q8_plan_launches
    assert call(1, 64, None, 1, 2) == -1
    assert call(1, 64, p, 0, 2) == -1 and call(1, 64, p, 9, 2) == -1
    assert call(1, 64, p, 1, 0x80) == -1
    assert call(0, 64, p, 1, 2) == -2 and call(17, 64, p, 1, 0) == -2 and call(513, 64, p, 1, 2) == -2
    assert call(1, 33, p, 1, 2) == -2 and call(1, 0, p, 1, 2) == -2
    bad = (ctypes.c_int * 1)(0)
    assert call(1, 64, ctypes.cast(bad, ctypes.c_void_p), 1, 2) == -2
    assert call(1, 64, p, 2, 2) in (-5, 1, 2)


def test_plan_glu_launches_argument_errors(lib):
    """q8_plan_glu_launches rejects what q8_gemv_glu_ex would (the tiled flag is required) before any device query."""
    call = lib.q8_plan_glu_launches
    assert call(1, 64, 96, 0) == -1 and call(1, 64, 96, 0x80 | 2) == -1
    assert call(0, 64, 96, 2) == -2 and call(513, 64, 96, 2) == -2 and call(1, 33, 96, 2) == -2
    assert call(1, 64, 0, 2) == -2
    assert call(1, 64, 96, 2) in (-5, 1, 2)


def test_residual_norm_noalloc_argument_errors(lib):
    """The entry point that allocates nothing rejects, before any CUDA call, rows beyond its static counters and the
    arguments the residual norm rejects."""
    f = ctypes.c_float
    X, W, S, R, GM, H, O = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000, 0x60000, 0x90000
    call = lib.q8_gemv_residual_norm_noalloc
    assert call(X, W, S, R, GM, f(1e-6), H, O, 513, 64, 96, 2, None) == 2      # m > 512: more groups than counters
    assert call(X, W, S, R, GM, f(1e-6), H, O, 0, 64, 96, 2, None) == 2
    assert call(X, W, S, R, GM, f(1e-6), H, None, 2, 64, 96, 2, None) == 1     # no bf16 output
    assert call(X, W, S, R, GM, f(1e-6), None, O, 2, 64, 96, 2, None) == 1     # no h
    assert call(X, W, S, R, GM, f(1e-6), H, O, 2, 64, 96, 0, None) == 1        # not tiled
    assert call(X, W, S, R, GM, f(-1.0), H, O, 2, 64, 96, 2, None) == 1        # eps < 0
    assert call(X, W, S, R, GM, f(1e-6), H + 4, O, 2, 64, 96, 2, None) == 3    # h not 16-byte aligned
    assert call(X, W, S, R, GM, f(1e-6), H, H, 2, 64, 96, 2, None) == 1        # output over h
    assert lib.q8_version() > 0  # the library still answers
