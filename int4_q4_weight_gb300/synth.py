"""Seeded synthetic inputs for the q4_0 decode path.

This module holds no arithmetic of the method: it only draws seeded random
tensors with the shapes and distributions of the workloads (weights from
N(0, 0.02) in fp32, activations from N(0, 1) rounded to fp16, PLE table bytes
uniform in [-127, 127], row scales U(0.001, 0.02), norm weights U(0.5, 1.5),
token ids uniform in [0, 262144)).  Both the CUDA path and the CPU oracle are
fed from here; whatever is compared is generated once and copied.

Every tensor has its own generator, seeded from a base seed and the tensor's
name, so adding a tensor never shifts another one's values.  Values depend on
the device they are drawn on (torch's CPU and CUDA generators differ); callers
draw once and copy.
"""
from __future__ import annotations

import zlib
from dataclasses import dataclass

import torch

# E2B decoder shape table, restated here as workload data: 35 layers at hidden
# 1536; q/o 8 heads x 256 (sliding) or x 512 (full: every 5th layer from L4);
# one KV head on L0-L14 only; MLP 6144 on L0-L14 and 12288 on L15-L34.
E2B_HIDDEN = 1536
E2B_N_LAYERS = 35
_FULL = frozenset({4, 9, 14, 19, 24, 29, 34})


def e2b_dims(layer: int) -> dict:
    hd = 512 if layer in _FULL else 256
    return {"q": 8 * hd, "kv": hd if layer < 15 else 0,
            "mlp": 6144 if layer < 15 else 12288}


def e2b_matrix_shapes(layer: int) -> dict:
    """Name -> [rows, cols] of every weight matrix of one layer."""
    d = e2b_dims(layer)
    H = E2B_HIDDEN
    shapes = {"q": (d["q"], H)}
    if d["kv"]:
        shapes["k"] = (d["kv"], H)
        shapes["v"] = (d["kv"], H)
    shapes["o"] = (H, d["q"])
    shapes["g"] = (d["mlp"], H)
    shapes["u"] = (d["mlp"], H)
    shapes["d"] = (H, d["mlp"])
    return shapes


# Workload sizes of the five synthetic configurations.
GEMV_N, GEMV_K = 2048, 1536
PLE_V, PLE_L, PLE_LD, PLE_D, PLE_S = 262144, 35, 256, 1536, 64
HEAD_V, HEAD_K = 262144, 1536
CHUNK_S = 64
GEMM_SHAPES = {"up": (6144, 1536), "down": (1536, 6144), "head": (262144, 1536)}


def sub_seed(base: int, *names) -> int:
    key = "/".join([str(base)] + [str(n) for n in names]).encode()
    return (int(base) * 1_000_003 + zlib.crc32(key)) & 0x7FFF_FFFF_FFFF_FFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """fp32 samples of N(0, std^2)."""
    t = torch.randn(tuple(shape), generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    return t.mul_(std)


def normal_f16(shape, seed: int, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in fp32 and rounded to fp16."""
    return normal(shape, 1.0, seed, device).to(torch.float16)


def uniform(shape, lo: float, hi: float, seed: int, device="cpu") -> torch.Tensor:
    t = torch.rand(tuple(shape), generator=_gen(seed, device), device=device,
                   dtype=torch.float32)
    return t.mul_(hi - lo).add_(lo)


def randint(shape, lo: int, hi_inclusive: int, seed: int, device="cpu",
            dtype=torch.int64) -> torch.Tensor:
    return torch.randint(lo, hi_inclusive + 1, tuple(shape), generator=_gen(seed, device),
                         device=device, dtype=dtype)


# --------------------------------------------------------------------------
# configuration recipes
# --------------------------------------------------------------------------
def gemv_inputs(seed: int = 1001, device="cpu", N: int = GEMV_N, K: int = GEMV_K,
                batch: int = 1):
    """W [N, K] ~ N(0, 0.02) fp32 and x [batch, K] ~ N(0, 1) fp16."""
    W = normal((N, K), 0.02, sub_seed(seed, "W", N, K), device)
    x = normal_f16((batch, K), sub_seed(seed, "x", batch, K), device)
    return W, x


# INT2 shapes of the mixed-bit recipe: FFN gate/up and down of L15-L34, the tied head
Q2_SHAPES = {"gate": (12288, 1536), "down": (1536, 12288), "head": (262144, 1536)}


def q2_inputs(seed: int = 1006, device="cpu", N: int = 12288, K: int = 1536, batch: int = 1):
    """INT2 weights drawn directly (the format comes from QAT, no quantiser):
    codes [N, K/4] uint8 with every 2-bit code uniform in 0..3, per-row f32
    scales 0.02 * (0.5 + U[0,1)), and x [batch, K] ~ N(0, 1) fp16."""
    codes = randint((N, K // 4), 0, 255, sub_seed(seed, "codes", N, K), device, dtype=torch.int32).to(torch.uint8)
    scales = uniform((N,), 0.01, 0.03, sub_seed(seed, "scales", N), device)
    x = normal_f16((batch, K), sub_seed(seed, "x", batch, K), device)
    return codes, scales, x


@dataclass
class PleInputs:
    ids: torch.Tensor        # int32 [S]
    table: torch.Tensor      # int8 [V, L*ld]
    row_scale: torch.Tensor  # f32 [V]
    proj: torch.Tensor       # f32 [L*ld, D]
    hidden: torch.Tensor     # f16 [S, D]
    norm_w: torch.Tensor     # f32 [ld]


def ple_inputs(seed: int = 1002, device="cpu", S: int = PLE_S, V: int = PLE_V,
               L: int = PLE_L, ld: int = PLE_LD, D: int = PLE_D) -> PleInputs:
    return PleInputs(
        ids=randint((S,), 0, V - 1, sub_seed(seed, "ids", S, V), device, torch.int32),
        table=randint((V, L * ld), -127, 127, sub_seed(seed, "table", V, L * ld), device,
                      torch.int8),
        row_scale=uniform((V,), 0.001, 0.02, sub_seed(seed, "scale", V), device),
        proj=normal((L * ld, D), 0.02, sub_seed(seed, "proj", L * ld, D), device),
        hidden=normal_f16((S, D), sub_seed(seed, "hidden", S, D), device),
        norm_w=uniform((ld,), 0.5, 1.5, sub_seed(seed, "norm_w", ld), device),
    )


def e2b_weight(seed: int, layer: int, name: str, device="cpu") -> torch.Tensor:
    """fp32 weight matrix ``name`` of layer ``layer`` ~ N(0, 0.02)."""
    rows, cols = e2b_matrix_shapes(layer)[name]
    return normal((rows, cols), 0.02, sub_seed(seed, "e2b", layer, name), device)


def e2b_h0(seed: int = 1003, device="cpu") -> torch.Tensor:
    return normal_f16((E2B_HIDDEN,), sub_seed(seed, "h0"), device)


def head_inputs(seed: int = 1004, device="cpu", batch: int = 1, V: int = HEAD_V,
                K: int = HEAD_K):
    W = normal((V, K), 0.02, sub_seed(seed, "W", V, K), device)
    h = normal_f16((batch, K), sub_seed(seed, "h", batch, K), device)
    return W, h


def gemm_inputs(seed: int = 1005, device="cpu", N: int = 6144, K: int = 1536,
                S: int = CHUNK_S):
    W = normal((N, K), 0.02, sub_seed(seed, "W", N, K), device)
    X = normal_f16((S, K), sub_seed(seed, "X", S, K), device)
    return W, X
