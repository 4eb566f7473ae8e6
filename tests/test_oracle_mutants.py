"""Plant a mistake in the oracle, on the CPU, and check that some pin catches it.

Each mutant rewrites one function of the oracle (a textual edit of its source:
a flipped sign, a dropped term, a swapped index, a wrong constant) inside a
private copy of the module, then runs every pin against that copy.  A mutant
that no pin rejects would mean the pins do not cover that part of the oracle.
"""
import importlib.util
import inspect
import os
import sys
import textwrap

import pytest

import oracle.q4_oracle as O_real
from oracle_pins import ALL_PINS

MUTANTS = [
    # quantiser
    ("round half to even", "round_half_away", "np.sign(v) * np.floor(np.abs(v) + 0.5)", "np.round(v)"),
    ("scale sign flipped", "quantize_q4_0", "m / np.float32(-8.0)", "m / np.float32(8.0)"),
    ("midpoint 7", "quantize_q4_0", "round_half_away(ratio) + Q4_MID", "round_half_away(ratio) + 7"),
    ("no clipping", "quantize_q4_0", "np.clip(q, 0, 15)", "np.clip(q, 0, 16) % 16"),
    ("last absmax on ties", "block_absmax_signed",
     "idx = np.argmax(np.abs(blocks), axis=-1)",
     "idx = blocks.shape[-1] - 1 - np.argmax(np.abs(blocks)[..., ::-1], axis=-1)"),
    ("high nibble first", "pack_nibbles", "(q[:, 0::2] | (q[:, 1::2] << 4))", "(q[:, 1::2] | (q[:, 0::2] << 4))"),
    ("high nibble first (read)", "unpack_nibbles", "q[:, 0::2] = codes & 0x0F", "q[:, 1::2] = codes & 0x0F\n    q[:, 0::2] = codes >> 4\n    return q"),
    ("scale from fp32 truncated", "quantize_q4_0", "scales = d32.astype(np.float16)",
     "scales = (d32.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32).astype(np.float16)"),
    # dequant / gemv
    ("dequant without midpoint", "dequantize_q4_0", "astype(np.int64) - Q4_MID", "astype(np.int64)"),
    ("dequant scale of wrong block", "dequantize_q4_0", "* d[..., None]", "* np.roll(d, 1, axis=1)[..., None]"),
    ("gemv transposed", "q4_gemv", "y = x @ Wd.T", "y = (Wd @ x.T).T if Wd.shape[0] == Wd.shape[1] else x @ Wd.T[:, ::-1]"),
    ("gemv x rounded to bf16", "q4_gemv", "x = np.asarray(x_f16, dtype=np.float16).astype(np.float64)",
     "x = bf16_rne(np.asarray(x_f16, dtype=np.float16).astype(np.float32)).astype(np.float64)"),
    # head
    ("softcap cap 20", "softcap", "np.tanh(z / cap) * cap", "np.tanh(z / cap) * 20.0"),
    ("softcap inside", "softcap", "np.tanh(z / cap) * cap", "np.tanh(z) * cap"),
    ("argmax highest index", "lmhead_softcap_argmax", "idx = np.argmax(s, axis=1)",
     "idx = s.shape[1] - 1 - np.argmax(s[:, ::-1], axis=1)"),
    ("top2 = min", "lmhead_softcap_argmax", "rest[rows, idx] = -np.inf", "rest[rows, idx] = -np.inf\n    rest = np.where(np.isinf(rest), np.inf, -rest)"),
    # PLE / norm
    ("ple without x16", "ple_gather_project", "* np.float32(embed_scale)", "* np.float32(1.0)"),
    ("ple norm over whole row", "ple_gather_project", "rmsnorm(p.reshape(S, L, ld), norm_w, eps=eps, axis=-1).reshape(S, L * ld)",
     "rmsnorm(p, np.tile(norm_w, L), eps=eps, axis=-1)"),
    ("ple strided chunks", "ple_gather_project", "p.reshape(S, L, ld)", "p.reshape(S, ld, L).transpose(0, 2, 1)"),
    ("ple norm weight 1+w", "ple_gather_project", "norm_w, eps=eps", "1.0 + np.asarray(norm_w, np.float64), eps=eps"),
    ("ple proj transposed", "ple_gather_project", "hid @ np.asarray(proj, dtype=np.float32).astype(np.float64).T",
     "hid @ np.asarray(proj, dtype=np.float32).astype(np.float64)[::-1].T"),
    ("rmsnorm eps outside", "rmsnorm", "np.sqrt(np.mean(v * v, axis=axis, keepdims=True) + eps)",
     "(np.sqrt(np.mean(v * v, axis=axis, keepdims=True)) + eps)"),
    ("rmsnorm mean over sum", "rmsnorm", "np.mean(v * v, axis=axis, keepdims=True)", "np.sum(v * v, axis=axis, keepdims=True)"),
    # GEMM tiles
    ("bf16 truncation", "bf16_rne", "(u + np.uint64(0x7FFF) + kept_lsb)", "(u)"),
    ("bf16 ties up", "bf16_rne", "(u + np.uint64(0x7FFF) + kept_lsb)", "(u + np.uint64(0x8000))"),
    ("gemm without tile rounding of w", "q4_gemm_chunk", "Wt = bf16_rne(dequantize_q4_0(codes, scales).astype(np.float32))",
     "Wt = dequantize_q4_0(codes, scales).astype(np.float32)"),
    # chain
    ("gelu erf form", "gelu_tanh", "0.5 * x * (1.0 + np.tanh(c * (x + 0.044715 * x * x * x)))",
     "0.5 * x * (1.0 + np.tanh(c * (x + 0.04 * x * x * x)))"),
    ("full layers from L5", "e2b_layer_dims", "full = layer in E2B_FULL_LAYERS", "full = layer % 5 == 0"),
    ("kv on all layers", "e2b_layer_dims", "kv = head_dim if layer in E2B_KV_LAYERS else 0", "kv = head_dim"),
    ("chain o consumes a", "e2b_layer", 'st["o"] = q4_gemv(*lw["o"], to_f16(st["q"]))',
     'st["o"] = q4_gemv(*lw["o"], to_f16(st["q"])) + q4_gemv(*lw["k"], st["a"]).sum() * 0.01 if "k" in lw else q4_gemv(*lw["o"], to_f16(st["q"]))'),
    ("chain no final norm", "e2b_layer", 'st["h"] = to_f16(rmsnorm(st["y"], eps=eps))', 'st["h"] = to_f16(st["y"])'),
    ("chain gate only", "e2b_layer", 'to_f16(gelu_tanh(st["g"]) * st["u"].astype(np.float64))', 'to_f16(gelu_tanh(st["g"]))'),
    ("chain gate and up swapped", "e2b_layer", 'to_f16(gelu_tanh(st["g"]) * st["u"].astype(np.float64))',
     'to_f16(gelu_tanh(st["u"]) * st["g"].astype(np.float64))'),
    ("chain pre-attention norm dropped", "e2b_layer",
     'st["a"] = to_f16(rmsnorm(np.asarray(h_f16, np.float16).astype(np.float64), eps=eps))',
     'st["a"] = to_f16(np.asarray(h_f16, np.float16).astype(np.float64))'),
    ("chain mid-layer norm dropped", "e2b_layer", 'st["b"] = to_f16(rmsnorm(st["o"], eps=eps))', 'st["b"] = to_f16(st["o"])'),
    ("chain down reads the gate", "e2b_layer", 'st["y"] = q4_gemv(*lw["d"], st["m"])',
     'st["y"] = q4_gemv(*lw["d"], to_f16(st["g"]))'),
]


def _fresh_oracle():
    spec = importlib.util.spec_from_file_location("oracle_mutant_copy", O_real.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mutate(mod, func_name, old, new):
    src = textwrap.dedent(inspect.getsource(getattr(O_real, func_name)))
    assert old in src, f"mutation anchor not found in {func_name}: {old!r}"
    src = src.replace(old, new, 1)
    exec(compile(src, f"<mutant {func_name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_rejects_mutant(mutant):
    _, func, old, new = mutant
    mod = _mutate(_fresh_oracle(), func, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # any failure or crash counts as the pin biting
            caught.append(pin.__name__)
            break
    assert caught, f"no pin rejects mutant {mutant[0]!r}"
