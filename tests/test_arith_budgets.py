"""Error budgets of the tensor-core operand roundings (CPU only).

The PLE projection multiplies two fp16 pieces of each f32 weight (p1 = fp16(w),
p2 = fp16((w - p1) 2^11), 22 significant bits kept) and the batched LM head
rounds each dequantised weight once to fp16.  Both
budgets are checked here by feeding the rounded operand to the oracle (exact
fp64 arithmetic otherwise) and comparing with the oracle on the exact operand
under the parity rule, at the real row widths and vocabulary-scale samples.
The GPU parity tests then gate the kernels themselves against the exact
oracle.
"""
import numpy as np

from oracle import q4_oracle as O
from parity import MARGIN_EXEMPT, TOL, rel_err


def _fp16_pieces(a):
    """p1 + p2 2^-11 with p1 = fp16(w), p2 = fp16((w - p1) * 2^11) (what the
    tensor cores multiply), in fp64."""
    w = np.asarray(a, np.float32).astype(np.float64)
    p1 = w.astype(np.float16).astype(np.float64)
    p2 = ((w - p1) * 2048.0).astype(np.float16).astype(np.float64)
    return p1 + p2 / 2048.0


def test_fp16_pieces_projection_budget():
    rng = np.random.default_rng(71)
    S, L, ld, D, V = 16, 8, 256, 1536, 64
    proj = (rng.standard_normal((L * ld, D)) * 0.02).astype(np.float32)
    hidden = rng.standard_normal((S, D)).astype(np.float16)
    table = np.zeros((V, L * ld), np.int8)        # no gathered term: the projection alone
    row_scale = rng.uniform(0.001, 0.02, V).astype(np.float32)
    norm_w = rng.uniform(0.5, 1.5, ld).astype(np.float32)
    ids = rng.integers(0, V, S).astype(np.int32)
    # the pieces' sum reproduces the weight to 2^-22 relative (fp16 normal range)
    w = proj.astype(np.float64)
    pieces = _fp16_pieces(proj)
    normal = np.abs(w) >= 2.0 ** -14
    assert np.all(np.abs(pieces - w)[normal] <= 2.0 ** -22 * np.abs(w)[normal])
    assert np.all(np.abs(pieces - w)[~normal] <= 2.0 ** -36)
    exact, _ = O.ple_gather_project(ids, table, row_scale, proj, hidden, norm_w, L=L, ld=ld)
    # the oracle fed the pieces' sum (as f32, which holds its 22 bits exactly)
    split, _ = O.ple_gather_project(ids, table, row_scale, pieces.astype(np.float32), hidden, norm_w, L=L, ld=ld)
    e = rel_err(split, exact)
    assert e < 1e-5, e


def test_fp16_weight_tile_head_budget():
    rng = np.random.default_rng(73)
    V, K, b = 4096, 1536, 8
    W = (rng.standard_normal((V, K)) * 0.02).astype(np.float32)
    h = rng.standard_normal((b, K)).astype(np.float16)
    codes, scales = O.quantize_q4_0(W)
    _, r1, r2, margin, rs = O.lmhead_softcap_argmax(codes, scales, h)
    w16 = O.dequantize_q4_0(codes, scales).astype(np.float16).astype(np.float64)   # fp16(d (q - 8))
    z = h.astype(np.float64) @ w16.T
    s = O.softcap(z)
    assert rel_err(s, rs) < 0.75 * TOL
    gi = np.argmax(s, axis=1)
    ri = np.argmax(rs, axis=1)
    for i in range(b):
        assert gi[i] == ri[i] or margin[i] < MARGIN_EXEMPT


def test_fp16_tile_q8_projection_budget():
    """The int8 projection enters the tensor core as fp16(code * d), one
    rounding per weight (2^-11 relative); hidden fp16 is exact."""
    from oracle import q8_oracle as Q8
    rng = np.random.default_rng(79)
    S, L, ld, D, V = 16, 8, 256, 1536, 64
    proj = (rng.standard_normal((L * ld, D)) * 0.02).astype(np.float32)
    codes, scales = Q8.quantize_q8_0(proj)
    hidden = rng.standard_normal((S, D)).astype(np.float16)
    table = np.zeros((V, L * ld), np.int8)        # no gathered term: the projection alone
    row_scale = rng.uniform(0.001, 0.02, V).astype(np.float32)
    norm_w = rng.uniform(0.5, 1.5, ld).astype(np.float32)
    ids = rng.integers(0, V, S).astype(np.int32)
    exact, _ = Q8.ple_gather_project_q8(ids, table, row_scale, codes, scales, hidden, norm_w, L=L, ld=ld)
    tile = Q8.dequantize_q8_0(codes, scales).astype(np.float16).astype(np.float32)
    rounded, _ = O.ple_gather_project(ids, table, row_scale, tile, hidden, norm_w, L=L, ld=ld)
    e = rel_err(rounded, exact)
    assert 0 < e < 0.75 * TOL, e
