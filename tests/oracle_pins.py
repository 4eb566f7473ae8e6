"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle module ``O``
disagrees with a fact that does not come from the oracle itself: a value the
pages print, a hand-worked example of the pages' rule, a closed form, an
invariant, exact rational brute force on tiny inputs, or a library routine
that computes the same special case.  The mutant tests run the same pins on
deliberately broken copies of the oracle to show each pin bites.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _nib(codes, n, k):
    """Code of weight (n, k) read bit by bit: byte k//2, low nibble for even k."""
    byte = int(codes[n, k // 2])
    return (byte >> (4 * (k % 2))) & 0xF


def _scale(scales, n, k):
    return float(np.array(scales[n, k // 32], dtype=np.uint16).view(np.float16))


# --------------------------------------------------------------------------
# quantiser
# --------------------------------------------------------------------------
def pin_quantize_worked_block(O):
    rows = {r[0]: r[1:] for r in _read_golden("q4_block_worked.txt")}
    w = np.array([[float(v) for v in rows["w"]]], dtype=np.float32)
    codes, scales = O.quantize_q4_0(w)
    want_bytes = np.array([int(b, 16) for b in rows["bytes"]], dtype=np.uint8)
    assert codes.shape == (1, 16) and scales.shape == (1, 1)
    assert np.array_equal(codes[0], want_bytes), (codes[0], want_bytes)
    assert int(scales[0, 0]) == int(rows["d_bits"][0], 16)
    got_codes = [_nib(codes, 0, k) for k in range(32)]
    assert got_codes == [int(c) for c in rows["codes"]]


def pin_quantize_grid_fixed_point(O, seed=7, nblocks=400):
    """A block already on the grid (exactly one code 0, fp16 d != 0) re-quantises
    to the same codes and the same fp16 scale, bit for bit."""
    rng = np.random.default_rng(seed)
    K = 32
    c = rng.integers(1, 16, size=(nblocks, K))
    c[np.arange(nblocks), rng.integers(0, K, size=nblocks)] = 0
    mag = rng.uniform(1e-4, 2.0, size=nblocks).astype(np.float16)
    sign = np.where(rng.random(nblocks) < 0.5, -1.0, 1.0).astype(np.float16)
    d16 = (mag * sign).astype(np.float16)
    w = (d16.astype(np.float32)[:, None] * (c - 8).astype(np.float32)).astype(np.float32)
    codes, scales = O.quantize_q4_0(w)
    assert np.array_equal(scales[:, 0], d16.view(np.uint16))
    got = np.array([[_nib(codes, n, k) for k in range(K)] for n in range(nblocks)])
    assert np.array_equal(got, c)


def pin_quantize_nearest_grid(O, seed=11, N=24, K=256):
    """Brute force: every code is the grid point nearest w (over all 16 codes of
    the block's fp32 scale), ties away from zero; only the element equal to -m
    may sit at the clipped end.  Elements whose quotient lies within fp32
    rounding of a half-integer are skipped (the rule divides in fp32)."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    for n in range(N):
        for b in range(K // 32):
            blk = W[n, 32 * b: 32 * b + 32].astype(np.float64)
            j = int(np.argmax(np.abs(blk)))
            d = np.float32(np.float32(blk[j]) / np.float32(-8.0))
            assert _scale(scales, n, 32 * b) == float(np.float16(d))
            for i in range(32):
                w = blk[i]
                t = w / float(d)
                if abs(abs(t - math.floor(t)) - 0.5) < 1e-5:
                    continue
                dist = [abs(w - float(d) * (c - 8)) for c in range(16)]
                best = min(range(16), key=lambda c: (dist[c], -abs(c - 8)))
                assert _nib(codes, n, 32 * b + i) == best, (n, b, i, w, d)


def pin_quantize_zero_block(O):
    W = np.zeros((2, 64), np.float32)
    W[1, 32:] = np.linspace(-1, 1, 32, dtype=np.float32)
    codes, scales = O.quantize_q4_0(W)
    assert all(_nib(codes, 0, k) == 8 for k in range(64))
    assert all(_nib(codes, 1, k) == 8 for k in range(32))
    assert int(scales[0, 0]) == 0 and int(scales[0, 1]) == 0 and int(scales[1, 0]) == 0


def pin_dequant_affine(O, seed=3, N=16, K=128):
    """Dequant equals the pages' affine form d*q_u - 8*d evaluated in fp32 (both
    terms and their sum exact there), read back nibble by nibble."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    Wd = O.dequantize_q4_0(codes, scales)
    for n in range(N):
        for k in range(K):
            d = np.float32(_scale(scales, n, k))
            qu = np.float32(_nib(codes, n, k))
            aff = np.float32(d * qu) + np.float32(np.float32(-8.0) * d)
            assert Wd[n, k] == float(aff)


def pin_dequant_on_grid(O, seed=5, N=32, K=256):
    """Round trip: every dequantised value is d16 * j for an integer j in [-8, 7],
    and the error to the source weight is at most half a grid step (plus the
    clipped end and fp16 scale rounding)."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    Wd = O.dequantize_q4_0(codes, scales)
    d = np.repeat(scales.view(np.float16).astype(np.float64), 32, axis=1)
    j = Wd / d
    assert np.all(j == np.round(j)) and j.min() >= -8 and j.max() <= 7
    err = np.abs(Wd - W)
    assert np.all(err <= 1.0 * np.abs(d) * 1.001 + 1e-12)


# --------------------------------------------------------------------------
# GEMV
# --------------------------------------------------------------------------
def _exact_gemv(codes, scales, x):
    N = codes.shape[0]
    K = codes.shape[1] * 2
    out = []
    for n in range(N):
        acc = Fraction(0)
        for k in range(K):
            acc += Fraction(_scale(scales, n, k)) * (_nib(codes, n, k) - 8) * Fraction(float(x[k]))
        out.append(acc)
    return out


def pin_gemv_bruteforce(O, seed=13, N=3, K=96):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = rng.standard_normal(K).astype(np.float16)
    codes, scales = O.quantize_q4_0(W)
    y = O.q4_gemv(codes, scales, x)
    assert y.shape == (N,) and y.dtype == np.float32
    ex = _exact_gemv(codes, scales, x)
    for n in range(N):
        assert abs(float(y[n]) - float(ex[n])) <= 1e-6 * max(1.0, abs(float(ex[n])))


def pin_gemv_onehot(O, seed=17, N=5, K=64):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    for k in range(K):
        x = np.zeros(K, np.float16)
        x[k] = 1.0
        y = O.q4_gemv(codes, scales, x)
        for n in range(N):
            assert float(y[n]) == _scale(scales, n, k) * (_nib(codes, n, k) - 8)


def pin_gemv_batch_rows(O, seed=19, N=7, K=128, B=4):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((B, K)).astype(np.float16)
    codes, scales = O.quantize_q4_0(W)
    Y = O.q4_gemv(codes, scales, X)
    assert Y.shape == (B, N)
    for b in range(B):
        ex = _exact_gemv(codes, scales, X[b])
        for n in range(N):
            assert abs(float(Y[b, n]) - float(ex[n])) <= 1e-6 * max(1.0, abs(float(ex[n])))


# --------------------------------------------------------------------------
# head
# --------------------------------------------------------------------------
def pin_softcap_closed_forms(O):
    cap = 30.0
    assert float(O.softcap(np.array([0.0]))[0]) == 0.0
    z = np.linspace(-200, 200, 4001)
    s = O.softcap(z)
    assert np.all(np.abs(s) < cap)                     # strictly inside (-30, 30)
    assert np.all(np.diff(s) > 0)                      # monotone
    assert np.allclose(O.softcap(-z), -s, rtol=0, atol=0)   # odd
    # tanh(z/30)*30 = 15 exactly where z/30 = atanh(1/2)
    assert abs(float(O.softcap(np.array([30 * math.atanh(0.5)]))[0]) - 15.0) < 1e-12
    small = np.array([1e-3, 0.1, 0.5])
    taylor = small - small ** 3 / 2700.0 + 2 * small ** 5 / (15 * 30.0 ** 4)
    assert np.allclose(O.softcap(small), taylor, rtol=0, atol=1e-11)


def pin_head_argmax_ties(O):
    """One-hot h selects column k of W'; planted equal maxima go to the lowest
    row; top-2 equals top-1 when the maximum is shared."""
    N, K = 6, 32
    q = np.full((N, K), 8, np.uint8)
    q[:, 3] = [9, 15, 15, 2, 14, 0]          # column 3: values d*(q-8) with d = 0.5
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    scales = np.full((N, 1), np.float16(0.5).view(np.uint16), np.uint16)
    h = np.zeros((1, K), np.float16)
    h[0, 3] = 1.0
    idx, top1, top2, margin, s = O.lmhead_softcap_argmax(codes, scales, h)
    assert int(idx[0]) == 1
    assert float(top1[0]) == float(np.float32(30 * math.tanh(3.5 / 30)))
    assert float(top2[0]) == float(top1[0]) and float(margin[0]) == 0.0
    h[0, 3] = -1.0                              # now the most negative code wins
    idx, top1, top2, margin, s = O.lmhead_softcap_argmax(codes, scales, h)
    assert int(idx[0]) == 5 and abs(float(top1[0]) - 30 * math.tanh(4.0 / 30)) < 1e-6
    assert abs(float(top2[0]) - 30 * math.tanh(3.0 / 30)) < 1e-6


def pin_head_vs_sort(O, seed=23, V=300, K=64, B=3):
    """argmax / top-2 equal a stable sort of the exact softcapped logits."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((V, K)) * 0.02).astype(np.float32)
    h = rng.standard_normal((B, K)).astype(np.float16)
    codes, scales = O.quantize_q4_0(W)
    idx, top1, top2, margin, s = O.lmhead_softcap_argmax(codes, scales, h)
    for b in range(B):
        ex = _exact_gemv(codes, scales, h[b])
        sv = [30.0 * math.tanh(float(z) / 30.0) for z in ex]
        order = sorted(range(V), key=lambda i: (-sv[i], i))
        assert int(idx[b]) == order[0]
        assert abs(float(top1[b]) - sv[order[0]]) < 1e-6
        assert abs(float(top2[b]) - sv[order[1]]) < 1e-6


# --------------------------------------------------------------------------
# PLE
# --------------------------------------------------------------------------
def pin_ple_sidecar_sizes(O):
    g = {}
    for r in _read_golden("ple_sidecar.txt"):
        g[(r[0], r[1])] = r[2]
    V, D = int(g[("meta", "V")]), int(g[("meta", "D")])
    PLD, L, ld = int(g[("meta", "PLD")]), int(g[("meta", "L")]), int(g[("meta", "ld")])
    assert PLD == L * ld
    assert V * PLD == int(g[("file", "embed_per_layer.i8")])          # int8 table
    assert PLD * D * 4 == int(g[("file", "proj.f32")])                # f32 [8960,1536]
    assert V * 4 == int(g[("file", "embed_per_layer.scale.f32")])     # f32 per row
    assert ld * 4 == int(g[("file", "proj_norm.f32")])                # f32 [256]
    assert float(g[("meta", "embed_scale_pl")]) == math.sqrt(ld) == O.PLE_EMBED_SCALE


def _ple_small(seed, V=9, L=3, ld=8, D=16, S=4):
    rng = np.random.default_rng(seed)
    return dict(
        ids=rng.integers(0, V, S).astype(np.int32),
        table=rng.integers(-127, 128, (V, L * ld)).astype(np.int8),
        row_scale=rng.uniform(0.001, 0.02, V).astype(np.float32),
        proj=(rng.standard_normal((L * ld, D)) * 0.02).astype(np.float32),
        hidden_f16=rng.standard_normal((S, D)).astype(np.float16),
        norm_w=rng.uniform(0.5, 1.5, ld).astype(np.float32),
        L=L, ld=ld)


def pin_ple_gather_exact(O, seed=29):
    """proj = 0 makes the projection term vanish (RMSNorm(0) = 0), so the output
    is the gathered term alone: (float(q) * scale) * 16 in fp32, bit for bit."""
    a = _ple_small(seed)
    a["proj"] = np.zeros_like(a["proj"])
    out, gathered = O.ple_gather_project(**a)
    for t, v in enumerate(a["ids"]):
        assert np.array_equal(gathered[t], a["table"][v])
        for j in range(a["table"].shape[1]):
            want = np.float32(np.float32(float(a["table"][v, j])) * a["row_scale"][v]) * np.float32(16.0)
            assert out[t, j] == want


def pin_ple_bruteforce(O, seed=31):
    a = _ple_small(seed)
    out, _ = O.ple_gather_project(**a)
    L, ld = a["L"], a["ld"]
    D = a["proj"].shape[1]
    for t, v in enumerate(a["ids"]):
        p = [sum(float(a["proj"][r, c]) * float(a["hidden_f16"][t, c]) for c in range(D))
             for r in range(L * ld)]
        for c in range(L):
            seg = p[c * ld:(c + 1) * ld]
            r = 1.0 / math.sqrt(sum(e * e for e in seg) / ld + 1e-6)
            for j in range(ld):
                col = c * ld + j
                g = float(np.float32(np.float32(float(a["table"][v, col])) * a["row_scale"][v]) * np.float32(16.0))
                want = seg[j] * r * float(a["norm_w"][j]) + g
                assert abs(float(out[t, col]) - want) <= 1e-6 * max(1.0, abs(want))


def pin_ple_layer_chunks(O, seed=37):
    """Scaling the projection rows of layer chunk c by (c + 1) leaves the
    normalised term unchanged: the norm runs over each contiguous ld-chunk."""
    a = _ple_small(seed)
    a["proj"] = a["proj"] * np.float32(50.0)      # mean(p^2) >> eps
    out1, _ = O.ple_gather_project(**a)
    L, ld = a["L"], a["ld"]
    proj2 = a["proj"].copy()
    for c in range(L):
        proj2[c * ld:(c + 1) * ld] *= np.float32(c + 1)
    out2, _ = O.ple_gather_project(**{**a, "proj": proj2})
    assert np.allclose(out1, out2, rtol=1e-5, atol=1e-6)
    proj3 = a["proj"].copy()
    proj3[:, :] = proj3[np.argsort(np.arange(L * ld) % L, kind="stable")]   # strided regroup
    out3, _ = O.ple_gather_project(**{**a, "proj": proj3})
    assert not np.allclose(out1, out3, rtol=1e-3, atol=1e-4)


# --------------------------------------------------------------------------
# S=64 GEMM tiles
# --------------------------------------------------------------------------
def pin_bf16_rounding(O, seed=41):
    import torch
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(20000) * 10 ** rng.uniform(-6, 4, 20000)).astype(np.float32)
    ties = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -9, 3.0,
                     1.0 + 2 ** -7 + 2 ** -8], np.float32)
    v = np.concatenate([v, ties])
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(O.bf16_rne(v), want)


def pin_gemm_onehot(O, seed=43, N=8, K=64, S=4):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    codes, scales = O.quantize_q4_0(W)
    X = np.zeros((S, K), np.float16)
    ks = [0, 5, 33, 63]
    for t, k in enumerate(ks):
        X[t, k] = 1.0
    Y = O.q4_gemm_chunk(codes, scales, X)
    import torch
    for t, k in enumerate(ks):
        for n in range(N):
            w = np.float32(_scale(scales, n, k) * (_nib(codes, n, k) - 8))
            want = float(torch.tensor(float(w)).to(torch.bfloat16).float())
            assert float(Y[t, n]) == want


def pin_gemm_tile_bound(O, seed=47, N=16, K=256, S=8):
    """Tile rounding error stays within the bf16 bound 2u + u^2 (u = 2^-9) of
    sum |w'| |x| around the exact result, and the tiled result matches exact
    rational arithmetic on the rounded tiles."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    X = rng.standard_normal((S, K)).astype(np.float16)
    codes, scales = O.quantize_q4_0(W)
    Y = O.q4_gemm_chunk(codes, scales, X).astype(np.float64)
    u = 2.0 ** -9
    import torch
    for t in range(S):
        ex = _exact_gemv(codes, scales, X[t])
        for n in range(N):
            absum = sum(abs(_scale(scales, n, k) * (_nib(codes, n, k) - 8) * float(X[t, k]))
                        for k in range(K))
            assert abs(Y[t, n] - float(ex[n])) <= (2 * u + u * u) * absum + 1e-12
        if t == 0:
            for n in range(2):
                acc = Fraction(0)
                for k in range(K):
                    w = float(torch.tensor(_scale(scales, n, k) * (_nib(codes, n, k) - 8)).to(torch.bfloat16).float())
                    x = float(torch.tensor(float(X[t, k])).to(torch.bfloat16).float())
                    acc += Fraction(w) * Fraction(x)
                assert abs(Y[t, n] - float(acc)) <= 1e-6 * max(1.0, abs(float(acc)))


# --------------------------------------------------------------------------
# chain pieces
# --------------------------------------------------------------------------
def pin_rmsnorm(O, seed=53):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(1536) * 3.0
    out = O.rmsnorm(v)
    ms = np.mean(v * v)
    assert abs(np.mean(out * out) - ms / (ms + 1e-6)) < 1e-12       # closed form
    assert np.allclose(O.rmsnorm(v, w=np.full(1536, 2.0)), 2 * out, rtol=1e-15, atol=0)
    assert np.allclose(O.rmsnorm(5.0 * v), out, rtol=1e-6, atol=0)    # scale invariance
    c = np.full(256, -0.75)
    assert np.allclose(O.rmsnorm(c), -0.75 / math.sqrt(0.5625 + 1e-6))


def pin_gelu_tanh(O):
    import torch
    x = np.linspace(-12, 12, 2401)
    g = O.gelu_tanh(x)
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    assert np.allclose(g, ref, rtol=1e-13, atol=1e-15)
    exact = torch.nn.functional.gelu(torch.from_numpy(x)).numpy()      # erf form
    assert np.max(np.abs(g - exact)) < 1e-3
    assert float(O.gelu_tanh(np.array([0.0]))[0]) == 0.0
    assert abs(float(O.gelu_tanh(np.array([12.0]))[0]) - 12.0) < 1e-12


def pin_f16_rounding(O):
    """Rounding to binary16 (nearest, ties to even), on values whose exact answer
    follows from the format: 11 significant bits, subnormal step 2^-24,
    largest finite 65504 (the fp16 casts of the decode chain and the stored
    scales use it)."""
    ldexp = math.ldexp
    cases = [
        (1.0, 1.0), (ldexp(1.0, -24), ldexp(1.0, -24)), (65504.0, 65504.0),
        (1.0 + ldexp(1.0, -11), 1.0),                          # tie: to the even neighbour 1
        (1.0 + 3 * ldexp(1.0, -11), 1.0 + ldexp(1.0, -9)),     # tie: up to the even neighbour
        (1.0 + ldexp(1.0, -11) + ldexp(1.0, -40), 1.0 + ldexp(1.0, -10)),   # just past the tie
        (2049.0, 2048.0), (2051.0, 2052.0),                    # spacing 2 above 2048
        (-(1.0 + ldexp(1.0, -11)), -1.0),
        (ldexp(1.0, -25), 0.0),                                # half the smallest subnormal: to 0
        (3 * ldexp(1.0, -25), ldexp(1.0, -23)),                # subnormal tie: to even (2 steps)
        (ldexp(1.0, -14) - ldexp(1.0, -25), ldexp(1.0, -14)),  # tie at the normal boundary: up (even)
        (65519.0, 65504.0), (65520.0, math.inf), (-1e6, -math.inf),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float64)
    with np.errstate(over="ignore"):                           # the overflow cases are intended
        got = np.asarray(O.to_f16(x)).astype(np.float64)
    want = np.array([c[1] for c in cases], dtype=np.float64)
    assert np.array_equal(got, want), [(c[0], g) for c, g, w in zip(cases, got, want) if g != w]


def pin_e2b_dims(O):
    for r in _read_golden("e2b_layer_shapes.txt"):
        layer, full, q, kv, mlp = (int(v) for v in r)
        d = O.e2b_layer_dims(layer)
        assert (d["q"], d["kv"], d["mlp"]) == (q, kv, mlp), (layer, d)
        assert (layer in O.E2B_FULL_LAYERS) == bool(full)


def pin_e2b_layer_structure(O, seed=59):
    """k/v are produced and not consumed; the layer output is RMS-normalised; and
    the output changes with every consumed matrix."""
    rng = np.random.default_rng(seed)
    H, Q, KV, I = 64, 96, 32, 128

    def mat(r, c):
        return O.quantize_q4_0((rng.standard_normal((r, c)) * 0.1).astype(np.float32))

    lw = {"q": mat(Q, H), "k": mat(KV, H), "v": mat(KV, H), "o": mat(H, Q),
          "g": mat(I, H), "u": mat(I, H), "d": mat(H, I)}
    h = rng.standard_normal(H).astype(np.float16)
    st = O.e2b_layer(h, lw)
    assert st["h"].dtype == np.float16 and st["h"].shape == (H,)
    ms = float(np.mean(st["h"].astype(np.float64) ** 2))
    assert abs(ms - 1.0) < 5e-3
    lw2 = dict(lw, k=mat(KV, H), v=mat(KV, H))
    assert np.array_equal(O.e2b_layer(h, lw2)["h"], st["h"])
    for name in ("q", "o", "g", "u", "d"):
        lw3 = dict(lw)
        lw3[name] = mat(*{"q": (Q, H), "o": (H, Q), "g": (I, H), "u": (I, H), "d": (H, I)}[name])
        assert not np.array_equal(O.e2b_layer(h, lw3)["h"], st["h"]), name


def _pack_row_codes(codes_row):
    """Pack one row of 4-bit codes, column 2j in the low nibble of byte j."""
    out = []
    for j in range(0, len(codes_row), 2):
        out.append((int(codes_row[j]) & 0xF) | ((int(codes_row[j + 1]) & 0xF) << 4))
    return out


def _f16(x):
    """Round an fp64 value to the nearest fp16 (ties to even), back to fp64."""
    return float(np.float64(x).astype(np.float16))


def _f32(x):
    return float(np.float64(x).astype(np.float32))


def pin_e2b_layer_stage_by_stage(O, seed=61):
    """One tiny layer restated stage by stage in plain fp64 loops (reading R8),
    sharing no code with the oracle: the weights are built from integer codes
    and power-of-two scales, packed here bit by bit; each GEMV output is the
    correctly rounded fp64 sum (math.fsum of exact products) rounded to fp32;
    each RMSNorm is v / sqrt(mean(v^2) + 1e-6) with weight 1 ([E2B] Signature
    features: the weight multiplies directly); gelu is the tanh form ([MB]
    Speed: fp32 precise-tanh GELU), and the gate feeds the GELU while the up
    projection multiplies it ([MB] Speed: "gate/up matvecs + gelu + mul").
    Every stage output of O.e2b_layer must match: fp32 stages to 1e-6
    relative, fp16 stages to one fp16 step.  The input's RMS is 3 and the
    projections are scaled so that o's RMS is far from 1, so a dropped norm, a
    gate/up swap or a dropped fp16 cast moves some stage far outside that."""
    rng = np.random.default_rng(seed)
    H, Q, KV, I = 32, 64, 32, 96
    eps = 1e-6

    def build(rows, cols, scale_exp):
        codes = rng.integers(0, 16, size=(rows, cols))
        # one power-of-two scale per 32-column block, exponent scale_exp or one below
        exps = scale_exp - rng.integers(0, 2, size=(rows, cols // 32))
        d = [[math.ldexp(1.0, int(e)) for e in row] for row in exps]
        packed = np.array([_pack_row_codes(codes[n]) for n in range(rows)], dtype=np.uint8)
        bits = np.array([[np.float16(v).view(np.uint16) for v in row] for row in d], dtype=np.uint16)
        W = [[d[n][k // 32] * (int(codes[n, k]) - 8) for k in range(cols)] for n in range(rows)]
        return (packed, bits), W

    def gemv(W, x):
        return [_f32(math.fsum(w * xv for w, xv in zip(row, x))) for row in W]

    def rms(v):
        r = math.sqrt(math.fsum(t * t for t in v) / len(v) + eps)
        return [t / r for t in v]

    def gelu(x):
        return 0.5 * x * (1.0 + math.tanh(math.sqrt(2.0 / math.pi) * (x + 0.044715 * x * x * x)))

    lw, Wm = {}, {}
    for name, (r, c, e) in {"q": (Q, H, -5), "k": (KV, H, -5), "v": (KV, H, -5), "o": (H, Q, -3),
                            "g": (I, H, -5), "u": (I, H, -4), "d": (H, I, -6)}.items():
        lw[name], Wm[name] = build(r, c, e)
    h = [_f16(3.0 * v) for v in rng.standard_normal(H)]
    want = {}
    want["a"] = [_f16(t) for t in rms(h)]
    want["q"] = gemv(Wm["q"], want["a"])
    want["k"] = gemv(Wm["k"], want["a"])
    want["v"] = gemv(Wm["v"], want["a"])
    want["o"] = gemv(Wm["o"], [_f16(t) for t in want["q"]])
    want["b"] = [_f16(t) for t in rms(want["o"])]
    want["g"] = gemv(Wm["g"], want["b"])
    want["u"] = gemv(Wm["u"], want["b"])
    want["m"] = [_f16(gelu(gv) * uv) for gv, uv in zip(want["g"], want["u"])]
    want["y"] = gemv(Wm["d"], want["m"])
    want["h"] = [_f16(t) for t in rms(want["y"])]
    o_rms = math.sqrt(sum(t * t for t in want["o"]) / H)
    assert o_rms > 2.0 or o_rms < 0.5, o_rms       # the mid norm must change b
    assert not np.allclose(want["g"], want["u"], rtol=0.1)
    st = O.e2b_layer(np.array(h, dtype=np.float16), lw, eps=eps)
    for name in ("a", "q", "k", "v", "o", "b", "g", "u", "m", "y", "h"):
        got = np.asarray(st[name], dtype=np.float64)
        w = np.array(want[name], dtype=np.float64)
        assert got.shape == w.shape, (name, got.shape, w.shape)
        if name in ("a", "b", "m", "h"):
            tol = np.abs(w) * 2.0 ** -10 + 2.0 ** -24          # one fp16 step
        else:
            tol = np.abs(w) * 1e-6 + 1e-30
        assert np.all(np.abs(got - w) <= tol), (name, float(np.max(np.abs(got - w) - tol)))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
