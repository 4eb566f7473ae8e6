"""Pins of the INT2 oracle against what the pages and mathematics fix (CPU only)."""
import os

import numpy as np

from oracle import q2_oracle as Q

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q2_bytes_worked.txt")


def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f = line.split()
        rows.append((int(f[0], 16), [int(v) for v in f[1:5]], [int(v) for v in f[5:9]]))
    return rows


def test_worked_bytes():
    """Hand-decoded bytes: first code in bits[1:0], value = code - 2."""
    for byte, codes, values in _golden():
        b = np.array([[byte]], dtype=np.uint8)
        assert Q.unpack_q2(b)[0].tolist() == codes
        assert Q.q2_values(b)[0].tolist() == values


def test_matches_twos_complement_decode():
    """The pages' other storage: the same values in two's complement, decoded
    as (q ^ 2) - 2.  Re-encode every byte's values in two's complement and
    decode them that way: identical values for all 256 bytes."""
    b = np.arange(256, dtype=np.uint8)[:, None]
    vals = Q.q2_values(b)                                   # [256][4]
    twos = (vals & 3).astype(np.int64)                      # two's-complement 2-bit patterns
    assert np.array_equal(Q.q2_value_from_twos(twos), vals)
    assert set(np.unique(vals).tolist()) == {-2, -1, 0, 1}


def test_unpack_agrees_with_numpy_bit_unpacking():
    """An independent unpacking: numpy's little-endian bit order, bit pairs."""
    rng = np.random.default_rng(7)
    c = rng.integers(0, 256, size=(5, 12), dtype=np.uint8)
    bits = np.unpackbits(c, axis=-1, bitorder="little").reshape(5, 12, 4, 2)
    ref = (bits[..., 0] + 2 * bits[..., 1]).reshape(5, 48)
    assert np.array_equal(Q.unpack_q2(c), ref)
    assert np.array_equal(Q.unpack_q2(Q.pack_q2(ref)), ref)


def test_constant_codes_reduce_to_sums():
    """codes all 2 -> 0; all 3 -> scale * sum(x); all 0 -> -2 * scale * sum(x)."""
    rng = np.random.default_rng(8)
    x = rng.standard_normal((2, 64)).astype(np.float16)
    s = np.array([0.5, 3.0, 0.01], dtype=np.float32)
    sx = x.astype(np.float64).sum(axis=1)
    for code, factor in ((2, 0.0), (3, 1.0), (0, -2.0)):
        c = Q.pack_q2(np.full((3, 64), code, dtype=np.uint8))
        y = Q.q2_gemv(c, s, x)
        assert np.allclose(y, factor * sx[:, None] * s.astype(np.float64)[None, :], rtol=0, atol=1e-12)


def test_row_scale_brute_force():
    """Brute force on a tiny case: one scale per ROW, applied to that row only."""
    rng = np.random.default_rng(9)
    q = rng.integers(0, 4, size=(3, 8), dtype=np.uint8)
    s = np.array([2.0, -0.5, 0.25], dtype=np.float32)
    x = rng.standard_normal(8).astype(np.float16)
    y = Q.q2_gemv(Q.pack_q2(q), s, x)
    for n in range(3):
        acc = 0.0
        for k in range(8):
            acc += (int(q[n, k]) - 2) * float(x[k])
        assert abs(y[n] - float(s[n]) * acc) <= 1e-12 * max(1.0, abs(acc))
    # dequantise-then-dot is the same number
    assert np.allclose(Q.q2_dequantize(Q.pack_q2(q), s) @ x.astype(np.float64), y, rtol=1e-14, atol=1e-14)
