"""The C++ oracle's "next" rows -- the INT2 GEMV, the int8 per-block-32
weights and the PLE on them, the w4a8 activation pair -- against the numpy
oracles, and the numpy oracles' pins run on the C++ oracle (CPU only).

As for the main rows: codes, scales and the calibrated scale bit for bit,
floating results within the rounding of their output format (the fp64 sums
differ only in summation order)."""
import os

import numpy as np
import pytest

import test_a8_oracle as TA8
import test_q8_oracle as TQ8
from oracle import a8_oracle as A8
from oracle import cpp_oracle
from oracle import q2_oracle as Q2
from oracle import q4_oracle as O
from oracle import q8_oracle as Q8


@pytest.fixture(scope="module")
def C():
    return cpp_oracle.oracle()


def _same_fp32(c, n):
    """Two fp32 roundings of fp64 sums that differ only in order: equal, or one
    step apart at a tie."""
    c = np.asarray(c, np.float32)
    n = np.asarray(n, np.float32)
    assert np.all(np.abs(c.astype(np.float64) - n) <= np.spacing(np.abs(n)).astype(np.float64))


def test_q2_gemv(C):
    rng = np.random.default_rng(3)
    for N_, K in ((7, 64), (130, 1536), (5, 4096)):
        codes = rng.integers(0, 256, (N_, K // 4), dtype=np.uint8)
        scales = rng.uniform(1e-3, 2e-2, N_).astype(np.float32)
        x = rng.standard_normal((2, K)).astype(np.float16)
        c, n = C.q2_gemv(codes, scales, x, threads=3), Q2.q2_gemv(codes, scales, x)
        assert np.all(np.abs(c - n) <= 1e-12 * np.max(np.abs(n)))
        assert np.all(np.abs(C.q2_gemv(codes, scales, x[1]) - n[1]) <= 1e-12 * np.max(np.abs(n)))


def test_q8_quantize_bit_exact(C):
    rng = np.random.default_rng(4)
    W = (rng.standard_normal((40, 256)) * 0.02).astype(np.float32)
    W[0, :32] = 0.0                                             # a zero block
    W[1, 32:64] = np.float32(0.25) * np.sign(rng.standard_normal(32)).astype(np.float32)
    W[2, 64:96] = (np.arange(32) - 16) * np.float32(2.0 ** -7)  # on a grid
    for a, b in zip(C.quantize_q8_0(W), Q8.quantize_q8_0(W)):
        assert a.dtype == b.dtype and np.array_equal(a, b)
    codes, scales = Q8.quantize_q8_0(W)
    assert np.array_equal(C.dequantize_q8_0(codes, scales), Q8.dequantize_q8_0(codes, scales))
    with pytest.raises(ValueError):
        C.quantize_q8_0(np.full((1, 32), np.nan, np.float32))


def test_q8_ple(C):
    rng = np.random.default_rng(5)
    V, L, ld, D, S = 9, 2, 256, 128, 4
    proj = (rng.standard_normal((L * ld, D)) * 0.02).astype(np.float32)
    codes, scales = Q8.quantize_q8_0(proj)
    ids = rng.integers(0, V, S).astype(np.int32)
    table = rng.integers(-127, 128, (V, L * ld)).astype(np.int8)
    rs = rng.uniform(0.001, 0.02, V).astype(np.float32)
    hid = rng.standard_normal((S, D)).astype(np.float16)
    nw = rng.uniform(0.5, 1.5, ld).astype(np.float32)
    oc, gc = C.ple_gather_project_q8(ids, table, rs, codes, scales, hid, nw, L=L, ld=ld, threads=2)
    on, gn = Q8.ple_gather_project_q8(ids, table, rs, codes, scales, hid, nw, L=L, ld=ld)
    assert np.array_equal(gc, gn)
    _same_fp32(oc, on)


def test_a8_codes_calibration_and_products(C):
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((128, 1536)) * 3).astype(np.float16)
    s = A8.a8_calibrate(x)
    assert C.a8_calibrate(x) == s
    assert C.a8_calibrate(np.zeros(40, np.float16)) == np.float32(1.0)
    for sc in (s, np.float32(0.004), np.float32(2.0 ** -5)):
        assert np.array_equal(C.a8_quantize(x, sc), A8.a8_quantize(x, sc))
    W = (rng.standard_normal((96, 1536)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    _same_fp32(C.q4_gemv_a8(codes, scales, x[0], s, threads=3), A8.q4_gemv_a8(codes, scales, x[0], s))
    X = x[:64]
    _same_fp32(C.q4_gemm_chunk_a8(codes, scales, X, s, threads=3), A8.q4_gemm_chunk_a8(codes, scales, X, s))


# INT2 GEMV pins over any oracle object with q2_gemv (fixtures packed with
# the numpy oracle's pack_q2): what the pages fix about the format.
def pin_q2_bit_order_and_midpoint(M):
    """Byte 0b11100100 holds codes 0, 1, 2, 3 for columns 0..3 (the first code
    in bits [1:0]); column j alone gives scale * (code_j - 2)."""
    c = np.full((1, 1), 0xE4, dtype=np.uint8)
    s = np.array([0.5], dtype=np.float32)
    for j in range(4):
        x = np.zeros(4, np.float16)
        x[j] = 1.0
        assert float(M.q2_gemv(c, s, x)[0]) == 0.5 * (j - 2)


def pin_q2_constant_codes(M):
    """Codes all 2 give 0, all 3 give scale * sum(x), all 0 give -2 scale * sum(x)."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 64)).astype(np.float16)
    s = np.array([0.5, 3.0, 0.01], dtype=np.float32)
    sx = x.astype(np.float64).sum(axis=1)
    for code, factor in ((2, 0.0), (3, 1.0), (0, -2.0)):
        y = M.q2_gemv(Q2.pack_q2(np.full((3, 64), code, dtype=np.uint8)), s, x)
        assert np.allclose(y, factor * sx[:, None] * s.astype(np.float64)[None, :], rtol=0, atol=1e-12)


def pin_q2_row_scale_bruteforce(M):
    """One scale per row, on that row's sum only."""
    rng = np.random.default_rng(9)
    q = rng.integers(0, 4, size=(3, 8), dtype=np.uint8)
    s = np.array([2.0, -0.5, 0.25], dtype=np.float32)
    x = rng.standard_normal(8).astype(np.float16)
    y = M.q2_gemv(Q2.pack_q2(q), s, x)
    for n in range(3):
        acc = sum((int(q[n, k]) - 2) * float(x[k]) for k in range(8))
        assert abs(float(y[n]) - float(s[n]) * acc) <= 1e-12 * max(1.0, abs(acc))


Q2_PINS = [pin_q2_bit_order_and_midpoint, pin_q2_constant_codes, pin_q2_row_scale_bruteforce]


@pytest.mark.parametrize("pin", Q2_PINS, ids=[p.__name__ for p in Q2_PINS])
def test_q2_pins_on_both(C, pin):
    pin(Q2)
    pin(C)


@pytest.mark.parametrize("pin", TQ8.PINS, ids=[p.__name__ for p in TQ8.PINS])
def test_q8_pins_on_cpp(C, pin):
    pin(C)


@pytest.mark.parametrize("pin", TA8.PINS, ids=[p.__name__ for p in TA8.PINS])
def test_a8_pins_on_cpp(C, pin):
    pin(C)


# Planted mistakes in the C++ oracle's "next" rows (textual edits of a copy,
# compiled with the oracle's flags): some int8 or w4a8 pin must reject each.
NEXT_MUTANTS = [
    ("q2 last code in bits [1:0]", "(codes[(size_t)n * (K / 4) + k / 4] >> (2 * (k % 4))) & 3",
     "(codes[(size_t)n * (K / 4) + k / 4] >> (2 * (3 - k % 4))) & 3"),
    ("q2 midpoint 1", "acc += (double)(c - 2) * xv[(size_t)b * K + k];",
     "acc += (double)(c - 1) * xv[(size_t)b * K + k];"),
    ("q8 ties to even", "c = std::round((double)ratio);                // half away from zero",
     "c = std::nearbyint((double)ratio);"),
    ("q8 step max/128", "const float d32 = a / 127.0f;                     // IEEE fp32 quotient",
     "const float d32 = a / 128.0f;"),
    ("q8 ple on raw codes", "for (size_t i = 0; i < wd.size(); ++i) proj[i] = (float)wd[i];",
     "for (size_t i = 0; i < wd.size(); ++i) proj[i] = (float)codes[i];"),
    ("a8 ties away", "double c = std::nearbyint((double)r);               // round to nearest, ties to even",
     "double c = std::round((double)r);"),
    ("a8 clamp at -127", "if (c < -128.0) c = -128.0;", "if (c < -127.0) c = -127.0;"),
    ("a8 calibration over 128", "return amax > 0.0f ? amax / 127.0f : 1.0f;",
     "return amax > 0.0f ? amax / 128.0f : 1.0f;"),
    ("a8 gemv on raw x", "for (int k = 0; k < K; ++k) xd[k] = (double)q[k] * (double)s;",
     "for (int k = 0; k < K; ++k) xd[k] = f16_value(x[k]);"),
]


@pytest.mark.parametrize("mutant", NEXT_MUTANTS, ids=[m[0] for m in NEXT_MUTANTS])
def test_some_pin_rejects_next_row_cpp_mutant(mutant, tmp_path):
    _, old, new = mutant
    src = open(cpp_oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mut_src = os.path.join(tmp_path, "q4_oracle_mutant.cpp")
    with open(mut_src, "w") as f:
        f.write(src.replace(old, new))
    lib_path = cpp_oracle.build(force=True, src=mut_src, out=os.path.join(tmp_path, "libmutant.so"))
    mod = cpp_oracle.Oracle(cpp_oracle.load(lib_path))
    for pin in TQ8.PINS + TA8.PINS + Q2_PINS:
        try:
            pin(mod)
        except Exception:   # any failure or crash counts as the pin biting
            return
    pytest.fail(f"no pin rejects C++ mutant {mutant[0]!r}")
