"""CPU oracle for the w4a8 activation quantise/dequantise pair (QDQ).

TEST INFRASTRUCTURE ONLY, like :mod:`oracle.q4_oracle`: only the test-suite
and the benchmark's CPU legs use it; it shares no code with the CUDA library
and imports nothing from the package.

Source (page title, section):
  [MC]  "visible-cx/gemma-4-E2B-CoreAI", About the w4a8 bundle: the same QAT
        int4 per-block-32 weights and graph as the int4 decode bundle; the
        difference is an int8 quantize/dequantize pair on the input of every
        linear layer, calibrated on 128 synthetic samples; built as a
        prefill / time-to-first-token lever.  The same section notes that
        the toolchain's fast path is int8 weights times int8 activations and
        that a floating-point weight path stays in floating point, which is
        why the product below is a floating-point one on the dequantised
        activations.

Readings (the pages name the pair and its calibration, not its grid):
  A8-1  per-tensor, symmetric, zero point 0: one fp32 scale s per linear
        input; q = clamp(rint(x / s), -128, 127), the quotient an IEEE fp32
        division and the rounding half to even (the int8 range of a
        zero-point-0 quantiser); the layer sees x' = s * q.
  A8-2  calibration, min-max over the samples: s = amax / 127 as an IEEE
        fp32 quotient, amax the largest |x| over every calibration sample;
        s = 1 when amax = 0 (every sample zero).
  A8-3  since q is an integer of at most 8 bits, exact in fp16 and in bf16,
        W' x' = s * (W' q): the weights multiply q and the row sum is scaled
        by s once.
  A8-4  decode GEMV (one token): the q4_0 GEMV on x' (exact dequantised
        weights, fp64 sums).  Prefill GEMM (64 tokens): the S=64 chunk's
        contraction, bf16(w') per weight, on x' per token.
"""
from __future__ import annotations

import numpy as np

from oracle import q4_oracle as O

__all__ = ["A8_QMIN", "A8_QMAX", "A8_CAL_DIV", "a8_calibrate", "a8_quantize", "a8_qdq",
           "q4_gemv_a8", "q4_gemm_chunk_a8"]

A8_QMIN, A8_QMAX = -128, 127   # reading A8-1
A8_CAL_DIV = 127.0             # reading A8-2


def _scale32(s) -> np.float32:
    s32 = np.float32(s)
    if not (np.isfinite(s32) and s32 > 0):
        raise ValueError("the activation scale must be finite and > 0")
    return s32


def a8_calibrate(samples) -> np.float32:
    """Reading A8-2: s = max |x| / 127 (fp32) over all calibration samples
    (any shape; fp16 values as the kernels see them); 1 when all are zero."""
    x = np.asarray(samples, dtype=np.float16).astype(np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite calibration sample")
    amax = np.float32(np.max(np.abs(x))) if x.size else np.float32(0.0)
    if amax == 0:
        return np.float32(1.0)
    return np.float32(amax / np.float32(A8_CAL_DIV))


def a8_quantize(x_f16, s) -> np.ndarray:
    """Reading A8-1: q = clamp(rint(x / s), -128, 127), x / s an IEEE fp32
    quotient, rint half to even; int64 array of x's shape."""
    x = np.asarray(x_f16, dtype=np.float16).astype(np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("non-finite activation")
    ratio = (x / _scale32(s)).astype(np.float32)
    return np.clip(np.rint(ratio), A8_QMIN, A8_QMAX).astype(np.int64)


def a8_qdq(x_f16, s) -> np.ndarray:
    """x' = s * q, exact in fp64 (an 8-bit integer times an fp32 scale)."""
    return a8_quantize(x_f16, s).astype(np.float64) * float(_scale32(s))


def q4_gemv_a8(codes, scales, x_f16, s) -> np.ndarray:
    """Reading A8-4 (decode): y[n] = sum_k w'[n, k] * x'[k], fp64, as fp32."""
    Wd = O.dequantize_q4_0(codes, scales)
    return (Wd @ a8_qdq(x_f16, s)).astype(np.float32)


def q4_gemm_chunk_a8(codes, scales, X_f16, s) -> np.ndarray:
    """Reading A8-4 (prefill): Y[t, n] = sum_k bf16(w'[n, k]) * x'[t, k], fp64,
    as fp32; X is fp16 [64][K]."""
    Wt = O.bf16_rne(O.dequantize_q4_0(codes, scales).astype(np.float32))
    return (a8_qdq(X_f16, s) @ Wt.astype(np.float64).T).astype(np.float32)
