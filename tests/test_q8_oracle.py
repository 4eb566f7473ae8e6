"""Pins of the int8 per-block-32 (q8) oracle against what the pages and the
mathematics fix (CPU only), and mutants of it that some pin must reject.

The pages name the format (int8, per block of 32, signed) but print no worked
block, so the pins are closed forms: the grid's fixed points, the
reconstruction bound of a nearest-point rounding, hand-built ties, the zero
block, exact dequantisation, and the PLE on a projection that already lies on
the grid (where the int8 form must reproduce the f32 form's brute force).
"""
import importlib.util
import inspect
import math
import textwrap

import numpy as np
import pytest

from oracle import q4_oracle as O4
from oracle import q8_oracle as Q8_real


def _grid_block(rng, d_bits, lead):
    """Codes in [-127, 127] with code `lead` (+-127) at a random place."""
    c = rng.integers(-126, 127, 32)
    c[rng.integers(0, 32)] = lead
    d = np.uint16(d_bits).view(np.float16).astype(np.float64)
    return c, d


def pin_grid_fixed_point(Q, seed=3, nblocks=300):
    """A block built on the grid, w = d * c with fp16 d > 0 and one |c| = 127,
    re-quantises to the same codes and scale bits: max|w| = 127 d exactly, so
    max|w| / 127 = d, and every w / d = c exactly."""
    rng = np.random.default_rng(seed)
    W = np.empty((nblocks, 32), np.float32)
    C = np.empty((nblocks, 32), np.int64)
    D = np.empty(nblocks, np.uint16)
    for i in range(nblocks):
        bits = int(rng.integers(0x1400, 0x3C00))     # normal fp16 scales 2^-10 .. 1
        c, d = _grid_block(rng, bits, 127 if i % 2 else -127)
        W[i] = (c * d).astype(np.float32)            # exact: 19 significant bits
        C[i], D[i] = c, bits
    codes, scales = Q.quantize_q8_0(W)
    assert np.array_equal(codes.astype(np.int64), C)
    assert np.array_equal(scales.reshape(-1), D)
    assert np.array_equal(Q.dequantize_q8_0(codes, scales), W.astype(np.float64))


def pin_nearest_point_bound(Q, seed=5, N=40, K=256):
    """Rounding to the nearest grid point: every |w - w'| is at most half a step
    (plus the fp16 rounding of the stored step, at most 127 d 2^-11), and the
    largest-magnitude element of each block sits at code +-127."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = Q.quantize_q8_0(W)
    Wd = Q.dequantize_q8_0(codes, scales)
    d = O4.f16_from_bits(scales)                               # [N, K/32]
    step = np.repeat(d, 32, axis=1)
    err = np.abs(W.astype(np.float64) - Wd)
    assert np.all(err <= step * (0.5 + 127 * 2.0 ** -11) * (1 + 1e-6))
    blocks = np.abs(W).reshape(N, K // 32, 32)
    arg = np.argmax(blocks, axis=-1)
    lead = np.take_along_axis(codes.astype(np.int64).reshape(N, K // 32, 32), arg[..., None], -1)[..., 0]
    lead_sign = np.sign(np.take_along_axis(W.reshape(N, K // 32, 32), arg[..., None], -1)[..., 0])
    assert np.array_equal(lead, (127 * lead_sign).astype(np.int64))
    assert int(np.abs(codes.astype(np.int64)).max()) == 127


def pin_ties_away_from_zero(Q):
    """Hand-built exact ties: with max|w| = 127 d (d = 2^-6), w = 2.5 d and
    w = -3.5 d round away from zero to 3 and -4; 0.5 d to 1."""
    d = 2.0 ** -6
    w = np.zeros((1, 32), np.float32)
    w[0, :6] = np.array([127, 2.5, -3.5, 0.5, -0.5, 126.5]) * d
    codes, scales = Q.quantize_q8_0(w)
    assert codes[0, :6].tolist() == [127, 3, -4, 1, -1, 127]
    assert codes[0, 6:].tolist() == [0] * 26
    assert int(scales[0, 0]) == int(np.float16(d).view(np.uint16))


def pin_zero_block(Q):
    w = np.zeros((2, 64), np.float32)
    w[1, 32:] = np.linspace(-1, 1, 32, dtype=np.float32)
    codes, scales = Q.quantize_q8_0(w)
    assert np.all(codes[0] == 0) and np.all(codes[1, :32] == 0)
    assert scales[0].tolist() == [0, 0] and int(scales[1, 0]) == 0
    assert int(scales[1, 1]) == int(np.float16(np.float32(1.0) / np.float32(127.0)).view(np.uint16))
    assert codes[1, 32] == -127 and codes[1, 63] == 127


def pin_signed_storage(Q):
    """Codes are two's-complement int8 (signed, no midpoint): the byte 0x81 is
    -127 and dequantises to -127 d."""
    codes = np.array([[0x81, 0x7F, 0x00, 0xFF] + [0] * 28], dtype=np.uint8).view(np.int8)
    d = np.float16(0.25)
    scales = np.array([[d.view(np.uint16)]], dtype=np.uint16)
    assert Q.dequantize_q8_0(codes, scales)[0, :4].tolist() == [-31.75, 31.75, 0.0, -0.25]


def pin_dequant_block_scale(Q, seed=7):
    """Block b of a row takes scale b: scales 1, 2, 4, ... on all-one codes."""
    codes = np.ones((2, 128), np.int8)
    sc = np.array([[1.0, 2.0, 4.0, 8.0], [0.5, 0.25, 0.125, 3.0]], np.float16).view(np.uint16)
    Wd = Q.dequantize_q8_0(codes, sc)
    assert np.array_equal(Wd[0], np.repeat([1.0, 2.0, 4.0, 8.0], 32))
    assert np.array_equal(Wd[1], np.repeat([0.5, 0.25, 0.125, 3.0], 32))


def pin_ple_q8_on_grid_bruteforce(Q, seed=11):
    """A projection already on the int8 grid: the int8 PLE equals a brute-force
    evaluation of the f32 definition (fp64 sums, per-chunk RMSNorm, x16
    gathered term) on that projection."""
    rng = np.random.default_rng(seed)
    V, L, ld, D, S = 7, 2, 8, 64, 3
    c = rng.integers(-127, 128, (L * ld, D))
    c[:, ::32] = 127                               # every block reaches the grid's end
    d = rng.uniform(1e-4, 1e-3, (L * ld, D // 32)).astype(np.float16)
    proj = (c * np.repeat(d.astype(np.float64), 32, axis=1)).astype(np.float32)
    codes, scales = Q.quantize_q8_0(proj)
    ids = rng.integers(0, V, S).astype(np.int32)
    table = rng.integers(-127, 128, (V, L * ld)).astype(np.int8)
    rs = rng.uniform(0.001, 0.02, V).astype(np.float32)
    hid = rng.standard_normal((S, D)).astype(np.float16)
    nw = rng.uniform(0.5, 1.5, ld).astype(np.float32)
    out, gathered = Q.ple_gather_project_q8(ids, table, rs, codes, scales, hid, nw, L=L, ld=ld)
    for t, v in enumerate(ids):
        assert np.array_equal(gathered[t], table[v])
        p = [sum(float(proj[r, k]) * float(hid[t, k]) for k in range(D)) for r in range(L * ld)]
        for ch in range(L):
            seg = p[ch * ld:(ch + 1) * ld]
            r = 1.0 / math.sqrt(sum(e * e for e in seg) / ld + 1e-6)
            for j in range(ld):
                col = ch * ld + j
                g = float(np.float32(np.float32(float(table[v, col])) * rs[v]) * np.float32(16.0))
                want = seg[j] * r * float(nw[j]) + g
                assert abs(float(out[t, col]) - want) <= 1e-6 * max(1.0, abs(want))


PINS = [pin_grid_fixed_point, pin_nearest_point_bound, pin_ties_away_from_zero, pin_zero_block,
        pin_signed_storage, pin_dequant_block_scale, pin_ple_q8_on_grid_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(Q8_real)


MUTANTS = [
    ("step max/128", "quantize_q8_0", "a / np.float32(Q8_MAX)", "a / np.float32(128.0)"),
    ("round half to even", "quantize_q8_0", "O.round_half_away(ratio)", "np.round(ratio)"),
    ("truncating rounding", "quantize_q8_0", "O.round_half_away(ratio)", "np.trunc(ratio)"),
    ("codes negated", "quantize_q8_0", "q.reshape(N, K), scales", "(-q).reshape(N, K), scales"),
    ("clip to 126", "quantize_q8_0", "-Q8_MAX, Q8_MAX)", "-126, 126)"),
    ("offset-binary codes", "dequantize_q8_0", "np.int8).astype(np.int64)", "np.int8).view(np.uint8).astype(np.int64)"),
    ("scale of the next block", "dequantize_q8_0", "* d[..., None]", "* np.roll(d, -1, axis=1)[..., None]"),
    ("projection transposed rows", "ple_gather_project_q8", "proj = dequantize_q8_0(codes, scales).astype(np.float32)",
     "proj = dequantize_q8_0(codes, scales).astype(np.float32)[::-1].copy()"),
]


def _mutant(func, old, new):
    spec = importlib.util.spec_from_file_location("q8_oracle_mutant", Q8_real.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    src = textwrap.dedent(inspect.getsource(getattr(Q8_real, func)))
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
