"""CPU oracle for the int8 per-block-32 PLE projection (the q8 weight format).

TEST INFRASTRUCTURE ONLY, like :mod:`oracle.q4_oracle`: only the test-suite,
the package smoke check and the benchmark's CPU legs use it; it shares no code
with the CUDA library and imports nothing from the package.

Source (page title, section):
  [MB]  "Gemma-4 E2B mobile mixed-bit QAT weights - extraction + Core AI
        transplant"
        - "The decode recipe (Section 10)", mixed-bit map: the PLE gate/proj
          weights and the per-layer model projection [8960,1536] are INT8.
        - "Official checkpoint" equivalence notes: the PLE int8 weights are
          genuinely signed; the model projection ships as BF16 in the
          official checkpoint and the export re-quantises it to int8 per
          block of 32.
  [MC]  "visible-cx/gemma-4-E2B-CoreAI", The PLE gather-table sidecar: the
        projection is [L*ld = 8960 rows][D = 1536 columns]; everything after
        the projection (per-256 RMSNorm, the x16 gathered table term) is the
        f32 form's.

Readings (the pages name the format, not its grid):
  Q8-1  per block of 32 along K: a = max |w|; d = a / 127 as an IEEE fp32
        quotient; code = clamp(round(w / d), -127, 127) from the IEEE fp32
        quotient, rounding half away from zero (as the q4_0 reading R1); the
        stored scale is fp16(d), nearest-even.  Symmetric signed grid
        [-127, 127] (two's-complement bytes, no midpoint: "genuinely
        signed").  An all-zero block stores scale +0 and codes 0.
  Q8-2  planar layout as q4_0: codes int8 [N][K], scales fp16 bits [N][K/32].
  Q8-3  dequantisation w' = fp16(d) * code, exact (an 11-bit by 8-bit product).
  Q8-4  the PLE with an int8 projection is the f32 PLE with proj = w'.
"""
from __future__ import annotations

import numpy as np

from oracle import q4_oracle as O

__all__ = ["QK8", "Q8_MAX", "quantize_q8_0", "dequantize_q8_0", "ple_gather_project_q8"]

QK8 = 32        # weights per block
Q8_MAX = 127    # largest code magnitude


def quantize_q8_0(W) -> tuple[np.ndarray, np.ndarray]:
    """fp32 weights [N, K] -> (codes int8 [N, K], scales fp16 bits uint16 [N, K/32]).

    Readings Q8-1 and Q8-2: per 32-block, d = max|w| / 127 (fp32), code =
    clamp(round_half_away(w / d), -127, 127), scale = fp16(d).
    """
    W = np.asarray(W, dtype=np.float32)
    if W.ndim != 2 or W.shape[1] % QK8:
        raise ValueError("W must be [N, K] with K a multiple of 32")
    if not np.all(np.isfinite(W)):
        raise ValueError("non-finite weight")
    N, K = W.shape
    blocks = W.reshape(N, K // QK8, QK8)
    a = np.max(np.abs(blocks), axis=-1)                         # float32, exact
    d32 = (a / np.float32(Q8_MAX)).astype(np.float32)            # IEEE fp32 quotient
    if np.any(d32 > 65504.0):
        raise ValueError("block scale overflows fp16")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (blocks / d32[..., None]).astype(np.float32)    # IEEE fp32 quotient
    q = np.clip(O.round_half_away(ratio), -Q8_MAX, Q8_MAX)
    q = np.where(d32[..., None] == 0, 0, q).astype(np.int8)     # all-zero block: codes 0
    scales = d32.astype(np.float16).view(np.uint16)
    return q.reshape(N, K), scales


def dequantize_q8_0(codes, scales) -> np.ndarray:
    """w' = fp16(d) * code per 32-block, exact in fp64 (reading Q8-3)."""
    q = np.asarray(codes, dtype=np.int8).astype(np.int64)
    d = O.f16_from_bits(scales)
    N, K = q.shape
    return (q.reshape(N, K // QK8, QK8) * d[..., None]).reshape(N, K)


def ple_gather_project_q8(ids, table, row_scale, codes, scales, hidden_f16, norm_w,
                          L: int = 35, ld: int = 256,
                          embed_scale: float = O.PLE_EMBED_SCALE, eps: float = 1e-6):
    """The PLE input with an int8 per-block-32 projection (reading Q8-4):
    :func:`oracle.q4_oracle.ple_gather_project` on proj = w' (the dequantised
    int8 matrix, exact in fp32).  Returns (out f32 [S, L*ld], gathered int8)."""
    proj = dequantize_q8_0(codes, scales).astype(np.float32)    # exact: 19 significant bits
    return O.ple_gather_project(ids, table, row_scale, proj, hidden_f16, norm_w,
                                L=L, ld=ld, embed_scale=embed_scale, eps=eps)
