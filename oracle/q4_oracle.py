"""CPU oracle for the q4_0 weight-only int4 decode path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
this module; only the test-suite, the package smoke check and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs use it.  It shares no code with the
CUDA library (no common helpers, tables or constants) and imports nothing from
the package.  Every input it sees comes from the caller (the seeded input
generators); it draws no random numbers itself.

Plain and slow on purpose: numpy, fp64 wherever the pages do not fix the
precision, one library primitive (``numpy`` matmul) per contraction, no
blocking, fusion or reordering.  Each function names the passage it follows.

Sources (page title, section):
  [MC]  "visible-cx/gemma-4-E2B-CoreAI" (Hugging Face model card)
        - Provenance table: "Weight format: int4, per-block-32 ... the ggml q4_0 grid";
          export functions main (S=1 decode) and prefill (S=64 chunked prefill).
        - "The PLE gather-table sidecar": file sizes and meta.json (V 262144,
          D 1536, PLD 8960, L 35, ld 256, embed_scale_pl 16.0 = sqrt(256)).
  [E2B] "Gemma 4 E2B (text decoder) - Core AI" (Core AI model zoo)
        - "Signature features": 35 layers, dual head_dim 256/512, KV-sharing,
          double-wide MLP on shared layers, final logit softcap tanh(z/30)*30,
          RMSNorm multiplies by weight directly.
        - "QAT weights": q4_0 = per-block-32 absmax symmetric int4; plain absmax
          (--lin-sym) is the literal q4_0 grid; shared layers carry no k/v proj.
        - "What it took": fused head with two-level in-kernel argmax, no logit
          readback.
  [MB]  "Gemma-4 E2B mobile mixed-bit QAT weights - extraction + Core AI
        transplant" (Core AI model zoo knowledge page)
        - "P6 DONE": packing = UNSIGNED code minus midpoint (int4 -8).
        - "The decode recipe (Section 10)": layer shapes, 1 KV head x 256 on
          L0-L14, FFN 12288 on L15-L34; INT4 packing assumed low nibble first.
        - "P2 progress" / "P2 DONE": full-attention layers L4/9/14/19/24/29/34
          with q [4096,1536] and kv [512,1536]; norms by direct assignment;
          ple_projection_norm is a real (256,) vector; PLE tables concatenated
          layer-major on axis 1 into [262144, 8960].
        - "P3 DONE / Receiving-end design": INT4 dequant as the affine form
          w = d*q_u - 8*d, exact in fp16; fused gate/up with an fp32
          precise-tanh GELU epilogue.

Readings where the pages are silent (each also listed in the design notes):
  R1  rounding in the quantiser is half away from zero (C ``roundf``), applied
      to the IEEE fp32 quotient w / d32 with d32 = m / -8 kept in fp32; the fp16
      scale is stored separately (round to nearest even).
  R2  the signed absmax m is the first element of largest |w| in k order.
  R3  an all-zero block stores d = +0 (fp16 bits 0x0000) and codes 8.
  R4  RMSNorm epsilon is 1e-6; the synthetic decode chain uses weight 1.
  R5  PLE: gathered term is (float(q) * scale) * 16 in fp32; the projection is
      proj [L*ld, D] row-major applied to the fp16 hidden; no further constant
      factors; the result is f32.
  R6  head: ties in the softcapped logit go to the lowest index; top-2 is the
      largest value over the other indices; margin is in softcapped units.
  R7  the S=64 prefill contraction rounds both tiles to bf16 (round to nearest
      even) before an exact fp64 sum; the exact-dequant result is also returned
      so the rounding gap can be reported.
  R8  the synthetic E2B weight pass per layer is
      a = f16(RMSNorm(h)); [q|k|v] = W_qkv a; o = W_o f16(q);
      b = f16(RMSNorm(o)); [g|u] = W_gu b; m = f16(gelu_tanh(g) * u);
      h' = f16(RMSNorm(W_d m)).  k and v are produced and not consumed.
"""
from __future__ import annotations

import math

import numpy as np

QK = 32            # weights per q4_0 block ([MC] Provenance; [E2B] QAT weights)
Q4_MID = 8         # unsigned code minus midpoint ([MB] P6 DONE)

# E2B shape facts ([E2B] Signature features; [MB] decode recipe, P2 progress).
E2B_LAYERS = 35
E2B_HIDDEN = 1536
E2B_FULL_LAYERS = (4, 9, 14, 19, 24, 29, 34)
E2B_KV_LAYERS = tuple(range(15))          # L15-L34 share K/V: no k/v projections
SOFTCAP = 30.0
PLE_EMBED_SCALE = 16.0                    # = sqrt(256), [MC] meta.json


# --------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------
def f16_from_bits(bits) -> np.ndarray:
    """uint16 bit patterns -> float64 values of those fp16 numbers."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def to_f16(v) -> np.ndarray:
    """Round to fp16, nearest-even (numpy's half conversion)."""
    return np.asarray(v, dtype=np.float64).astype(np.float16)


def round_half_away(v) -> np.ndarray:
    """Round to integer, ties away from zero (reading R1), exact in fp64."""
    v = np.asarray(v, dtype=np.float64)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def bf16_rne(v) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returned as float32.

    bf16 keeps the upper 16 bits of an fp32 word; rounding adds 0x7FFF plus
    the lowest kept bit before truncating.  Inputs here are finite.
    """
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    kept_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + kept_lsb) >> np.uint64(16)
    return (r << np.uint64(16)).astype(np.uint32).view(np.float32)


# --------------------------------------------------------------------------
# a1: quantise onto the q4_0 grid
# --------------------------------------------------------------------------
def block_absmax_signed(blocks: np.ndarray) -> np.ndarray:
    """Signed element of largest magnitude per block (reading R2)."""
    idx = np.argmax(np.abs(blocks), axis=-1)          # first occurrence
    return np.take_along_axis(blocks, idx[..., None], axis=-1)[..., 0]


def pack_nibbles(q: np.ndarray) -> np.ndarray:
    """Codes [N, K] (0..15) -> bytes [N, K/2]; even k in the low nibble.

    [MB] decode recipe: packed low-bits-first ("INT4 assumed analogous (low
    nibble first)").
    """
    q = np.asarray(q, dtype=np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Bytes [N, K/2] -> codes [N, K] (0..15); inverse of :func:`pack_nibbles`."""
    codes = np.asarray(codes, dtype=np.uint8)
    N, H = codes.shape
    q = np.empty((N, 2 * H), dtype=np.uint8)
    q[:, 0::2] = codes & 0x0F
    q[:, 1::2] = codes >> 4
    return q


def quantize_q4_0(W) -> tuple[np.ndarray, np.ndarray]:
    """fp32 weights [N, K] -> (codes uint8 [N, K/2], scales fp16 bits uint16 [N, K/32]).

    Per 32-block along K: m = signed absmax, d = m / -8, code =
    clamp(round(w / d) + 8, 0, 15), d stored as fp16 ([MC] Provenance,
    [E2B] QAT weights "per-block-32 absmax symmetric int4", [MB] P6 DONE
    "unsigned code minus midpoint").  Readings R1-R3 apply.
    """
    W = np.asarray(W, dtype=np.float32)
    if W.ndim != 2 or W.shape[1] % QK:
        raise ValueError("W must be [N, K] with K a multiple of 32")
    if not np.all(np.isfinite(W)):
        raise ValueError("non-finite weight")
    N, K = W.shape
    blocks = W.reshape(N, K // QK, QK)
    m = block_absmax_signed(blocks)                    # float32
    d32 = (m / np.float32(-8.0)).astype(np.float32)    # exact
    d32 = np.where(m == 0, np.float32(0.0), d32).astype(np.float32)   # +0, reading R3
    if np.any(np.abs(d32) > 65504.0):
        raise ValueError("block scale overflows fp16")
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (blocks / d32[..., None]).astype(np.float32)   # IEEE fp32 quotient
    q = round_half_away(ratio) + Q4_MID
    q = np.clip(q, 0, 15)
    q = np.where(d32[..., None] == 0, Q4_MID, q).astype(np.uint8)
    codes = pack_nibbles(q.reshape(N, K))
    scales = d32.astype(np.float16).view(np.uint16)
    return codes, scales


# --------------------------------------------------------------------------
# dequantisation (exact)
# --------------------------------------------------------------------------
def dequantize_q4_0(codes, scales) -> np.ndarray:
    """w' = d * (code - 8), exact in fp64 (and in fp32: an 11-bit by 4-bit product).

    [MB] Receiving-end design: the affine form d*q_u - 8*d is exact.
    """
    q = unpack_nibbles(codes).astype(np.int64) - Q4_MID
    d = f16_from_bits(scales)
    N, K = q.shape
    return (q.reshape(N, K // QK, QK) * d[..., None]).reshape(N, K)


# --------------------------------------------------------------------------
# a2: S=1 (and small-batch) dequant-GEMV
# --------------------------------------------------------------------------
def q4_gemv(codes, scales, x_f16) -> np.ndarray:
    """y[b, n] = sum_k w'[n, k] * x[b, k]; fp64 sum, returned as fp32.

    x is fp16 [b, K] (or [K]).  [MC] Provenance (main, S=1 decode).
    """
    Wd = dequantize_q4_0(codes, scales)
    x = np.asarray(x_f16, dtype=np.float16).astype(np.float64)
    y = x @ Wd.T
    return y.astype(np.float32)


# --------------------------------------------------------------------------
# a6: S=64 chunked-prefill dequant-GEMM
# --------------------------------------------------------------------------
def q4_gemm_chunk(codes, scales, X_f16) -> np.ndarray:
    """Y[t, n] = sum_k bf16(w'[n, k]) * bf16(x[t, k]); fp64 sum, fp32 result.

    The tiles are rounded to bf16 before the exact sum (reading R7).
    [MC] Provenance (prefill, static query width 64).
    """
    Wt = bf16_rne(dequantize_q4_0(codes, scales).astype(np.float32))
    Xt = bf16_rne(np.asarray(X_f16, dtype=np.float16).astype(np.float32))
    return (Xt.astype(np.float64) @ Wt.astype(np.float64).T).astype(np.float32)


def q4_gemm_chunk_exact(codes, scales, X_f16) -> np.ndarray:
    """Same contraction without tile rounding (exact dequant, exact fp16 x)."""
    return q4_gemv(codes, scales, X_f16)


# --------------------------------------------------------------------------
# a5: LM head + softcap + argmax
# --------------------------------------------------------------------------
def softcap(z, cap: float = SOFTCAP) -> np.ndarray:
    """s = tanh(z / cap) * cap ([E2B] Signature features)."""
    z = np.asarray(z, dtype=np.float64)
    return np.tanh(z / cap) * cap


def lmhead_softcap_argmax(codes, scales, h_f16, cap: float = SOFTCAP):
    """Per row b of h: z = W' h (fp64), s = softcap(z); argmax, top-1, top-2.

    Returns (idx int32 [b], top1 f32 [b], top2 f32 [b], margin f64 [b],
    logits s f32 [b, V]).  Reading R6 for ties.  [E2B] What it took (fused
    head + in-kernel argmax).
    """
    Wd = dequantize_q4_0(codes, scales)
    h = np.atleast_2d(np.asarray(h_f16, dtype=np.float16)).astype(np.float64)
    z = h @ Wd.T
    s = softcap(z, cap)
    idx = np.argmax(s, axis=1)                         # lowest index on ties
    rows = np.arange(s.shape[0])
    top1 = s[rows, idx]
    rest = s.copy()
    rest[rows, idx] = -np.inf
    top2 = rest.max(axis=1) if s.shape[1] > 1 else np.full(s.shape[0], -np.inf)
    return (idx.astype(np.int32), top1.astype(np.float32), top2.astype(np.float32),
            top1 - top2, s.astype(np.float32))


# --------------------------------------------------------------------------
# a4: PLE gather + projection + per-256 RMSNorm
# --------------------------------------------------------------------------
def rmsnorm(v, w=None, eps: float = 1e-6, axis: int = -1) -> np.ndarray:
    """v * rsqrt(mean(v^2) + eps) * w, weight applied directly (no 1+w shift).

    [E2B] Signature features ("RMSNorm multiplies by weight directly");
    [MB] P2 DONE (norms by direct assignment).  Reading R4 for eps.
    """
    v = np.asarray(v, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(v * v, axis=axis, keepdims=True) + eps)
    out = v * r
    if w is not None:
        out = out * np.asarray(w, dtype=np.float64)
    return out


def ple_gather_project(ids, table, row_scale, proj, hidden_f16, norm_w,
                       L: int = 35, ld: int = 256,
                       embed_scale: float = PLE_EMBED_SCALE, eps: float = 1e-6):
    """Per-Layer-Embedding input for S tokens.

    gathered[t] = table[ids[t], :]                    (int8 bytes, [L*ld])
    g[t]        = (float(gathered[t]) * scale[ids[t]]) * 16.0   in fp32
    p[t]        = proj @ float(hidden[t])             (fp64, [L*ld])
    n[t, c]     = RMSNorm(p[t, c*ld:(c+1)*ld]) * w    per layer chunk c
    out[t]      = n[t] + g[t]                          (f32 [L*ld])

    [MC] PLE gather-table sidecar (table int8 [V, 8960] + per-row f32 scale,
    x16.0, proj.f32 [8960, 1536], proj_norm.f32 [256]); [MB] P2 progress /
    P2 DONE (layer-major concat, real (256,) norm).  Reading R5.
    Returns (out f32 [S, L*ld], gathered int8 [S, L*ld]).
    """
    ids = np.asarray(ids, dtype=np.int64)
    table = np.asarray(table, dtype=np.int8)
    V, PLD = table.shape
    if PLD != L * ld:
        raise ValueError("table width must be L*ld")
    if np.any(ids < 0) or np.any(ids >= V):
        raise ValueError("token id out of range")
    gathered = table[ids]
    sc = np.asarray(row_scale, dtype=np.float32)[ids][:, None]
    g = (gathered.astype(np.float32) * sc).astype(np.float32) * np.float32(embed_scale)
    hid = np.asarray(hidden_f16, dtype=np.float16).astype(np.float64)
    p = hid @ np.asarray(proj, dtype=np.float32).astype(np.float64).T
    S = ids.shape[0]
    n = rmsnorm(p.reshape(S, L, ld), norm_w, eps=eps, axis=-1).reshape(S, L * ld)
    out = n + g.astype(np.float64)
    return out.astype(np.float32), gathered


# --------------------------------------------------------------------------
# a3 / a7: synthetic E2B weight pass (S=1 chain)
# --------------------------------------------------------------------------
def gelu_tanh(x) -> np.ndarray:
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), fp64.

    [MB] Speed (fused gate/up with an fp32 precise-tanh GELU epilogue).
    """
    x = np.asarray(x, dtype=np.float64)
    c = math.sqrt(2.0 / math.pi)
    return 0.5 * x * (1.0 + np.tanh(c * (x + 0.044715 * x * x * x)))


def e2b_layer_dims(layer: int) -> dict:
    """Projection widths of E2B layer ``layer`` (0-based).

    Full-attention layers (every 5th from L4) have 8 heads x 512, others
    8 x 256; one KV head of the same head_dim on L0-L14 only; MLP 6144 on
    L0-L14 and 12288 (double-wide) on L15-L34.  [E2B] Signature features;
    [MB] decode recipe and P2 progress.
    """
    full = layer in E2B_FULL_LAYERS
    head_dim = 512 if full else 256
    kv = head_dim if layer in E2B_KV_LAYERS else 0
    return {"q": 8 * head_dim, "kv": kv, "mlp": 6144 if layer < 15 else 12288}


def e2b_layer(h_f16, lw: dict, eps: float = 1e-6) -> dict:
    """One layer of the synthetic weight pass (reading R8).

    ``lw`` maps 'q','k','v','o','g','u','d' to (codes, scales); 'k' and 'v'
    may be absent.  Returns every stage output: a, q, k, v, o, b, g, u, m, y, h.
    """
    st = {}
    st["a"] = to_f16(rmsnorm(np.asarray(h_f16, np.float16).astype(np.float64), eps=eps))
    st["q"] = q4_gemv(*lw["q"], st["a"])
    if "k" in lw:
        st["k"] = q4_gemv(*lw["k"], st["a"])
        st["v"] = q4_gemv(*lw["v"], st["a"])
    st["o"] = q4_gemv(*lw["o"], to_f16(st["q"]))
    st["b"] = to_f16(rmsnorm(st["o"], eps=eps))
    st["g"] = q4_gemv(*lw["g"], st["b"])
    st["u"] = q4_gemv(*lw["u"], st["b"])
    st["m"] = to_f16(gelu_tanh(st["g"]) * st["u"].astype(np.float64))
    st["y"] = q4_gemv(*lw["d"], st["m"])
    st["h"] = to_f16(rmsnorm(st["y"], eps=eps))
    return st


def e2b_pass(h0_f16, layers: list, eps: float = 1e-6) -> np.ndarray:
    """Run the synthetic chain over ``layers``; returns the final fp16 h."""
    h = np.asarray(h0_f16, dtype=np.float16)
    for lw in layers:
        h = e2b_layer(h, lw, eps=eps)["h"]
    return h
