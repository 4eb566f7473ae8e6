"""CPU oracle for the INT2 per-row symmetric GEMV (the mixed-bit FFN / head format).

TEST INFRASTRUCTURE ONLY, like :mod:`oracle.q4_oracle`: only the test-suite,
the package smoke check and the benchmark's CPU legs use it; it shares no code
with the CUDA library and imports nothing from the package.

Source (page title, section):
  [MB]  "Gemma-4 E2B mobile mixed-bit QAT weights - extraction + Core AI
        transplant" (Core AI model zoo knowledge page)
        - "The decode recipe (Section 10)": FFN gating1/gating2/down of layers
          L15-L34 are INT2, [12288,1536] x 2 and [1536,12288]; the tied
          embed / lm_head is INT2 [262144,1536]; per-channel symmetric, all
          zero points 0, so dequant = code x scale[row].
        - same section, "Packing convention VERIFIED": 4 codes per byte, the
          first code in bits [1:0].
        - "P6 DONE": the official packing stores the UNSIGNED code minus its
          midpoint (int2: -2), so a code c in 0..3 stands for c - 2; the
          earlier extract stored the same values in two's complement.
        - "P3 DONE / Receiving-end design": the INT2 matvec decodes a
          two's-complement code q as (q ^ 2) - 2 and applies the per-row scale
          once, after the row's reduction.

Readings (the pages fix no more than this):
  Q2-1  scales are float32, one per output row ([V] f32 scale for the tied
        embed; the same for the FFN matrices);
  Q2-2  x is fp16 as in the q4_0 path; the sum is exact real arithmetic here
        (fp64), the scale multiplies the finished row sum;
  Q2-3  no quantiser: the weights come from QAT; synthetic tests draw codes
        and scales directly.
"""
from __future__ import annotations

import numpy as np

__all__ = ["unpack_q2", "pack_q2", "q2_values", "q2_dequantize", "q2_gemv", "q2_value_from_twos"]


def unpack_q2(codes) -> np.ndarray:
    """[N][K/4] bytes -> [N][K] unsigned codes 0..3; column 4b + j is bits
    [2j, 2j+2) of byte b ([MB] Packing convention: first code in bits[1:0])."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 4,), dtype=np.uint8)
    for j in range(4):
        out[..., j::4] = (c >> (2 * j)) & 3
    return out


def pack_q2(q) -> np.ndarray:
    """Inverse of :func:`unpack_q2` for codes 0..3 (test fixtures only)."""
    q = np.asarray(q, dtype=np.uint8)
    assert q.shape[-1] % 4 == 0 and int(q.max(initial=0)) <= 3
    out = np.zeros(q.shape[:-1] + (q.shape[-1] // 4,), dtype=np.uint8)
    for j in range(4):
        out |= (q[..., j::4] << (2 * j)).astype(np.uint8)
    return out


def q2_values(codes) -> np.ndarray:
    """Signed values c - 2 in {-2, -1, 0, 1} ([MB] P6: unsigned code minus midpoint)."""
    return unpack_q2(codes).astype(np.int64) - 2


def q2_value_from_twos(t) -> np.ndarray:
    """The pages' decode of a two's-complement 2-bit code t: (t ^ 2) - 2 ([MB] P3)."""
    t = np.asarray(t, dtype=np.int64)
    return (t ^ 2) - 2


def q2_dequantize(codes, scales) -> np.ndarray:
    """W[n][k] = (code - 2) * scale[n] in fp64 ([MB] Section 10: dequant = code x scale[row])."""
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    return q2_values(codes).astype(np.float64) * s[:, None]


def q2_gemv(codes, scales, x_f16) -> np.ndarray:
    """y[b][n] = scale[n] * sum_k (code[n][k] - 2) * x[b][k]: the integer-weighted
    row sum first, the per-row scale once after it ([MB] P3, reading Q2-2)."""
    v = q2_values(codes).astype(np.float64)
    x = np.asarray(x_f16, dtype=np.float16).astype(np.float64)
    x2 = np.atleast_2d(x)
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    y = (x2 @ v.T) * s[None, :]
    return y if x.ndim == 2 else y[0]
