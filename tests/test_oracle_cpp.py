"""The C++ oracle against the numpy oracle (CPU only).

The two are written independently (oracle/q4_oracle.cpp, oracle/q4_oracle.py)
and are each pinned by tests/oracle_pins.py.  Here they must agree: codes,
scales, gathered bytes and argmax indices bit for bit; every floating result
within the rounding of the output format (the fp64 sums of both differ only
in summation order, so a C++ fp64 value rounds to the numpy fp32/fp16 value,
up to a tie)."""
import numpy as np
import pytest

from oracle import cpp_oracle
from oracle import q4_oracle as N


@pytest.fixture(scope="module")
def C():
    return cpp_oracle.oracle()


def _close32(c64, n32):
    """c64 (fp64) rounds to n32 (fp32): within half an fp32 step, plus fp64 noise."""
    c64 = np.asarray(c64, np.float64)
    n = np.asarray(n32, np.float32)
    step = np.spacing(np.abs(n)).astype(np.float64)
    assert np.all(np.abs(c64 - n.astype(np.float64)) <= 0.5 * step + 1e-12 * np.abs(c64) + 1e-300)


def _weights(rng, N_, K, scale=0.02):
    W = (rng.standard_normal((N_, K)) * scale).astype(np.float32)
    W[0, :32] = 0.0                                    # a zero block
    W[1, 32:64] = np.float32(0.5) * np.sign(rng.standard_normal(32)).astype(np.float32)   # ties in |w|
    return W


def test_quantize_bit_exact(C):
    rng = np.random.default_rng(1)
    for N_, K in ((3, 64), (17, 256), (64, 1536)):
        W = _weights(rng, N_, K)
        for a, b in zip(C.quantize_q4_0(W), N.quantize_q4_0(W)):
            assert a.dtype == b.dtype and np.array_equal(a, b)
    # blocks on the grid, subnormal and huge scales
    W = np.zeros((4, 32), np.float32)
    W[0] = np.arange(32) - 16.0
    W[1] = np.float32(1e-6) * (np.arange(32) - 8)
    W[2] = np.float32(6e-8)
    W[3, 5] = -3e4
    for a, b in zip(C.quantize_q4_0(W), N.quantize_q4_0(W)):
        assert np.array_equal(a, b)
    with pytest.raises(ValueError):
        C.quantize_q4_0(np.full((1, 32), np.inf, np.float32))


def test_gemv_and_head(C):
    rng = np.random.default_rng(2)
    W = _weights(rng, 300, 1536)
    codes, scales = N.quantize_q4_0(W)
    x = rng.standard_normal((3, 1536)).astype(np.float16)
    _close32(C.q4_gemv64(codes, scales, x, threads=4), N.q4_gemv(codes, scales, x))
    _close32(C.q4_gemv64(codes, scales, x[0]), N.q4_gemv(codes, scales, x[0]))
    assert np.array_equal(C.dequantize_q4_0(codes, scales), N.dequantize_q4_0(codes, scales))
    ci, c1, c2, cs = C.lmhead64(codes, scales, x, threads=3)
    ni, n1, n2, nm, ns = N.lmhead_softcap_argmax(codes, scales, x)
    assert np.array_equal(ci[nm >= 1e-9], ni[nm >= 1e-9])
    _close32(c1, n1)
    _close32(c2, n2)
    _close32(cs, ns)


def test_gemm_tile_mirror(C):
    rng = np.random.default_rng(3)
    codes, scales = N.quantize_q4_0(_weights(rng, 96, 512))
    X = rng.standard_normal((64, 512)).astype(np.float16)
    _close32(C.q4_gemm_chunk64(codes, scales, X, threads=4), N.q4_gemm_chunk(codes, scales, X))
    v = (rng.standard_normal(4096) * 10).astype(np.float32)
    assert np.array_equal(C.bf16_rne(v).view(np.uint32), N.bf16_rne(v).view(np.uint32))


def test_ple(C):
    rng = np.random.default_rng(4)
    V, L, ld, D, S = 50, 3, 256, 128, 7
    table = rng.integers(-127, 128, size=(V, L * ld)).astype(np.int8)
    row_scale = rng.uniform(0.001, 0.02, V).astype(np.float32)
    proj = (rng.standard_normal((L * ld, D)) * 0.02).astype(np.float32)
    hidden = rng.standard_normal((S, D)).astype(np.float16)
    norm_w = rng.uniform(0.5, 1.5, ld).astype(np.float32)
    ids = rng.integers(0, V, S).astype(np.int32)
    co, cg = C.ple64(ids, table, row_scale, proj, hidden, norm_w, L=L, ld=ld, threads=2)
    no, ng = N.ple_gather_project(ids, table, row_scale, proj, hidden, norm_w, L=L, ld=ld)
    assert np.array_equal(cg, ng)
    _close32(co, no)
    with pytest.raises(ValueError):
        C.ple_gather_project(np.array([V], np.int32), table, row_scale, proj, hidden[:1], norm_w, L=L, ld=ld)


def test_norm_gelu_softcap(C):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((6, 256)) * 3
    w = rng.uniform(0.5, 1.5, 256)
    assert np.allclose(C.rmsnorm(v, w), N.rmsnorm(v, w), rtol=1e-14, atol=0)
    x = np.linspace(-10, 10, 1001)
    # near x = -10 both are 1 + tanh(...) cancellations of two libm tanh: absolute agreement
    assert np.allclose(C.gelu_tanh(x), N.gelu_tanh(x), rtol=1e-14, atol=1e-14)
    assert np.allclose(C.softcap(x * 50), N.softcap(x * 50), rtol=1e-14, atol=0)
    h = rng.standard_normal(4096) * 100
    assert np.array_equal(C.to_f16(h).view(np.uint16), N.to_f16(h).view(np.uint16))
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    a, b = C.f16_from_bits(bits), N.f16_from_bits(bits)
    fin = np.isfinite(b)
    assert np.array_equal(a[fin], b[fin]) and np.array_equal(np.isnan(a), np.isnan(b))


def _layers(rng, H, shapes):
    out = []
    for Q, KV, I in shapes:
        def m(r, c):
            return N.quantize_q4_0((rng.standard_normal((r, c)) * 0.05).astype(np.float32))
        lw = {"q": m(Q, H), "o": m(H, Q), "g": m(I, H), "u": m(I, H), "d": m(H, I)}
        if KV:
            lw.update(k=m(KV, H), v=m(KV, H))
        out.append(lw)
    return out


def test_decode_layer_and_pass(C):
    rng = np.random.default_rng(6)
    H = 256
    layers = _layers(rng, H, [(512, 128, 1024), (1024, 0, 2048), (512, 128, 1024)])
    h0 = rng.standard_normal(H).astype(np.float16)
    cs = C.e2b_layer(h0, layers[0], threads=3)
    ns = N.e2b_layer(h0, layers[0])
    assert set(cs) == set(ns)
    for k in ns:
        assert cs[k].dtype == ns[k].dtype, k
        if ns[k].dtype == np.float16:      # one fp16 step at most (a tie of the fp64 sums)
            assert np.all(np.abs(cs[k].astype(np.float64) - ns[k].astype(np.float64))
                          <= np.spacing(np.abs(ns[k])).astype(np.float64)), k
        else:
            assert np.all(np.abs(cs[k].astype(np.float64) - ns[k].astype(np.float64))
                          <= np.spacing(np.abs(ns[k])).astype(np.float64)), k
    assert "k" not in C.e2b_layer(h0, layers[1])
    # the chain: both oracles' passes agree at the fp16 output (a tiny chain,
    # where one-step forks have not had room to grow)
    cp = C.e2b_pass(h0, layers[:2], threads=2)
    npass = N.e2b_pass(h0, layers[:2])
    assert np.max(np.abs(cp.astype(np.float64) - npass.astype(np.float64))) <= 2 * np.max(np.spacing(np.abs(npass)))
    # the threads split rows only
    assert np.array_equal(C.e2b_pass(h0, layers, threads=1), C.e2b_pass(h0, layers, threads=5))
