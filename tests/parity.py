"""Comparison rule shared by the GPU parity tests.

Floats: elementwise |g - r| / max(|r|, rms(r)) <= 2e-3 (the stated tolerance
for fp32 accumulation with fp16/bf16 activations); integer, byte and index
outputs: bit-exact; argmax exempt where the oracle's top-2 margin is < 1e-3.
"""
import numpy as np

TOL = 2e-3
MARGIN_EXEMPT = 1e-3


def rel_err(g, r) -> float:
    g = np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    if r.size == 0:
        return 0.0
    den = np.maximum(np.abs(r), np.sqrt(np.mean(r * r)))
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(g - r) / den))


def assert_close(g, r, tol=TOL, what=""):
    e = rel_err(g, r)
    assert e <= tol, f"{what}: max rel err {e:.3e} > {tol:.1e}"
    return e
