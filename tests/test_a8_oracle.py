"""Pins of the w4a8 activation QDQ oracle against what the pages and the
mathematics fix (CPU only), and mutants of it that some pin must reject.

The pages name the pair (an int8 quantize/dequantize on every linear input,
calibrated) but print no worked value, so the pins are closed forms: the
grid's fixed points, hand-built ties, saturation, a quotient whose integer
only the fp32 division decides, the min-max calibration, and the GEMV / S=64
GEMM on activations already on the grid, where the QDQ is the identity and
the result must equal the pinned q4_0 oracles.
"""
import importlib.util
import inspect
import textwrap
from fractions import Fraction

import numpy as np
import pytest

from oracle import a8_oracle as A8_real
from oracle import q4_oracle as O4


def pin_grid_fixed_point(A, seed=3):
    """x = k s with s a power of two and |k| <= 127 (exact in fp16): x / s = k
    exactly, so q = k and x' = x."""
    rng = np.random.default_rng(seed)
    for e in (-9, -4, 0, 3):
        s = 2.0 ** e
        k = np.concatenate([np.arange(-128, 128), rng.integers(-128, 128, 200)])
        x = (k * s).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), k * s)
        assert np.array_equal(A.a8_quantize(x, s), k)
        assert np.array_equal(A.a8_qdq(x, s), k * s)


def pin_ties_half_to_even(A):
    """Exact ties (s = 2^-4): (k + 1/2) s rounds to the even neighbour."""
    s = 2.0 ** -4
    k2 = np.array([1, 3, 5, -1, -5, 253, -255])          # 2x the quotient
    x = (k2 * s / 2).astype(np.float16)
    assert np.array_equal(x.astype(np.float64), k2 * s / 2)
    assert A.a8_quantize(x, s).tolist() == [0, 2, 2, 0, -2, 126, -128]


def pin_saturation(A):
    """Quotients past the int8 range clamp to -128 and 127 (s = 1/2)."""
    x = np.array([63.75, 63.8125, 64.0, 1000.0, -64.0, -64.25, -64.375, -60000.0], np.float16)
    assert A.a8_quantize(x, 0.5).tolist() == [127, 127, 127, 127, -128, -128, -128, -128]


def _fp32_tie_case():
    """An fp16 x and an fp32 s whose IEEE fp32 quotient is exactly 2.5 while
    the exact quotient lies above it (so only the fp32 division gives 2)."""
    for xb in range(0x3C00, 0x4800):                      # fp16 x in [1, 8)
        x = float(np.uint16(xb).view(np.float16))
        s0 = np.float32(x / 2.5)
        for j in range(-6, 7):
            s = np.float32(s0)
            for _ in range(abs(j)):
                s = np.nextafter(s, np.float32(np.inf if j > 0 else -np.inf), dtype=np.float32)
            q32 = np.float32(np.float32(x) / s)
            exact = Fraction(x) / Fraction(float(s))
            if q32 == np.float32(2.5) and exact > Fraction(5, 2):
                return np.float16(x), s
    raise AssertionError("no fp32 tie case found")


def pin_fp32_quotient_decides(A):
    """The integer is decided on the IEEE fp32 quotient (reading A8-1): a case
    whose fp32 quotient is the tie 2.5 but whose exact quotient is above it."""
    x, s = _fp32_tie_case()
    assert int(A.a8_quantize(np.array([x]), s)[0]) == 2
    assert int(A.a8_quantize(np.array([-x]), s)[0]) == -2


def pin_calibration(A):
    """s = max |x| / 127 in fp32 over every sample; that element then sits at
    +-127; all-zero samples give s = 1."""
    samples = [np.array([0.5, -1.25, 2.0], np.float16), np.array([[0.25, -3.0], [1.0, 2.75]], np.float16)]
    s = A.a8_calibrate([np.concatenate([a.ravel() for a in samples])])
    assert s == np.float32(np.float32(3.0) / np.float32(127.0))
    assert A.a8_calibrate(np.concatenate([a.ravel() for a in samples])) == s
    assert A.a8_quantize(np.array([-3.0, 3.0], np.float16), s).tolist() == [-127, 127]
    assert A.a8_calibrate(np.zeros((4, 8), np.float16)) == np.float32(1.0)


def _q4_on_grid_weights(rng, N, K, exact_bf16):
    """q4_0 codes and fp16 scales (scales with <= 4 significant bits when
    exact_bf16, so that d (c - 8) is exact in bf16)."""
    codes = rng.integers(0, 256, (N, K // 2)).astype(np.uint8)
    if exact_bf16:
        d = (rng.integers(8, 16, (N, K // 32)) * 2.0 ** rng.integers(-12, -6, (N, K // 32))).astype(np.float16)
    else:
        d = rng.uniform(1e-3, 2e-2, (N, K // 32)).astype(np.float16)
    return codes, d.view(np.uint16)


def pin_gemv_on_grid_is_q4_gemv(A, seed=5):
    """Activations on the grid: the QDQ is the identity, so the w4a8 GEMV is
    the pinned q4_0 GEMV."""
    rng = np.random.default_rng(seed)
    N, K = 24, 160
    codes, scales = _q4_on_grid_weights(rng, N, K, False)
    s = 2.0 ** -5
    x = (rng.integers(-128, 128, K) * s).astype(np.float16)
    np.testing.assert_allclose(A.q4_gemv_a8(codes, scales, x, s), O4.q4_gemv(codes, scales, x), rtol=1e-6, atol=0)


def pin_gemm_on_grid_is_q4_gemm(A, seed=7):
    """The S=64 chunk on grid activations (exact in bf16) is the pinned
    q4_gemm_chunk, bf16 weight tile included."""
    rng = np.random.default_rng(seed)
    N, K = 16, 128
    codes, scales = _q4_on_grid_weights(rng, N, K, False)
    s = 2.0 ** -3
    X = (rng.integers(-128, 128, (64, K)) * s).astype(np.float16)
    np.testing.assert_allclose(A.q4_gemm_chunk_a8(codes, scales, X, s), O4.q4_gemm_chunk(codes, scales, X),
                               rtol=1e-6, atol=0)


def pin_gemv_bruteforce(A, seed=9):
    """Off the grid, against exact rational arithmetic: x' = s q with q from
    the fp32 quotient, y = sum_k d (c - 8) x'."""
    rng = np.random.default_rng(seed)
    N, K = 3, 64
    codes, scales = _q4_on_grid_weights(rng, N, K, False)
    x = rng.standard_normal(K).astype(np.float16)
    s = np.float32(0.0173)
    y = A.q4_gemv_a8(codes, scales, x, s)
    d = scales.view(np.float16)
    for n in range(N):
        tot = Fraction(0)
        for k in range(K):
            b = int(codes[n, k // 2])
            c = (b & 15) if k % 2 == 0 else (b >> 4)
            r = np.float32(np.float32(x[k]) / s)
            q = int(np.clip(np.rint(r), -128, 127))
            tot += Fraction(float(d[n, k // 32])) * (c - 8) * q * Fraction(float(s))
        assert abs(float(y[n]) - float(tot)) <= 1e-6 * max(1.0, abs(float(tot)))


PINS = [pin_grid_fixed_point, pin_ties_half_to_even, pin_saturation, pin_fp32_quotient_decides,
        pin_calibration, pin_gemv_on_grid_is_q4_gemv, pin_gemm_on_grid_is_q4_gemm, pin_gemv_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(A8_real)


MUTANTS = [
    ("ties away from zero", "a8_quantize", "np.rint(ratio)", "O.round_half_away(ratio)"),
    ("truncation", "a8_quantize", "np.rint(ratio)", "np.trunc(ratio)"),
    ("symmetric clamp to 127", "a8_quantize", "A8_QMIN, A8_QMAX)", "-A8_QMAX, A8_QMAX)"),
    ("no clamp", "a8_quantize", "np.clip(np.rint(ratio), A8_QMIN, A8_QMAX)", "np.rint(ratio)"),
    ("fp64 quotient", "a8_quantize", "(x / _scale32(s)).astype(np.float32)",
     "(x.astype(np.float64) / float(_scale32(s)))"),
    ("calibration over 128", "a8_calibrate", "amax / np.float32(A8_CAL_DIV)", "amax / np.float32(128.0)"),
    ("scale not applied", "a8_qdq", "* float(_scale32(s))", "* 1.0"),
    ("gemm without the bf16 tile", "q4_gemm_chunk_a8",
     "O.bf16_rne(O.dequantize_q4_0(codes, scales).astype(np.float32))", "O.dequantize_q4_0(codes, scales)"),
    ("gemv on raw x", "q4_gemv_a8", "a8_qdq(x_f16, s)", "np.asarray(x_f16, np.float16).astype(np.float64)"),
]


def _mutant(func, old, new):
    spec = importlib.util.spec_from_file_location("a8_oracle_mutant", A8_real.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    src = textwrap.dedent(inspect.getsource(getattr(A8_real, func)))
    assert old in src, f"mutation anchor not found in {func}: {old!r}"
    exec(compile(src.replace(old, new, 1), f"<mutant {func}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_rejects_mutant(mutant):
    mod = _mutant(*mutant[1:])
    for pin in PINS:
        try:
            pin(mod)
        except Exception:   # any failure or crash counts as the pin biting
            return
    pytest.fail(f"no pin rejects mutant {mutant[0]!r}")
