"""Plant a mistake in the C++ oracle, on the CPU, and check that some pin catches it.

Each mutant is a textual edit of a copy of oracle/q4_oracle.cpp (a flipped
sign, a dropped term, a swapped index, a wrong constant, swapped operands),
compiled with the oracle's own flags into a temporary library and loaded
behind the same API; the pins of tests/oracle_pins.py then run against it.
"""
import os

import pytest

from oracle import cpp_oracle
from oracle_pins import ALL_PINS

MUTANTS = [
    ("round half to even", "(double)std::round(ratio)", "(double)std::nearbyint(ratio)"),
    ("scale sign flipped", "float d32 = m / -8.0f;                                 // exact",
     "float d32 = m / 8.0f;"),
    ("midpoint 7", "(double)std::round(ratio) + 8.0;", "(double)std::round(ratio) + 7.0;"),
    ("last absmax on ties", "if (std::fabs(blk[i]) > std::fabs(m)) m = blk[i];   // first of the largest",
     "if (std::fabs(blk[i]) >= std::fabs(m)) m = blk[i];"),
    ("high nibble first", "return (k & 1) ? (b >> 4) : (b & 15);", "return (k & 1) ? (b & 15) : (b >> 4);"),
    ("dequant without midpoint", "(double)(code_at(codes, K, n, k) - 8)", "(double)(code_at(codes, K, n, k))"),
    ("fp16 ties away from zero", "const double r = std::nearbyint(std::ldexp(a, 11 - e));",
     "const double r = std::round(std::ldexp(a, 11 - e));"),
    ("softcap inside", "s[v] = std::tanh(z[(size_t)v + (size_t)b * V] / cap) * cap;",
     "s[v] = std::tanh(z[(size_t)v + (size_t)b * V]) * cap;"),
    ("argmax highest index", "if (s[v] > s[best]) best = v;", "if (s[v] >= s[best]) best = v;"),
    ("ple without x16", "const float g = ((float)q * row_scale[id]) * embed_scale;",
     "const float g = ((float)q * row_scale[id]);"),
    ("ple norm weight 1+w", "(chunk[i] * f) * (double)norm_w[i]", "(chunk[i] * f) * (1.0 + (double)norm_w[i])"),
    ("rmsnorm eps outside", "return 1.0 / std::sqrt(ss / n + eps);", "return 1.0 / (std::sqrt(ss / n) + eps);"),
    ("bf16 truncation", "const uint64_t r = (w + 0x7fffu + ((w >> 16) & 1u)) >> 16;", "const uint64_t r = w >> 16;"),
    ("gemm without tile rounding of w", "wt[k] = (double)bf16_round((float)weight_at(codes, scales, K, n, k));",
     "wt[k] = weight_at(codes, scales, K, n, k);"),
    ("gelu wrong cubic term", "(x + 0.044715 * x * x * x)", "(x + 0.04 * x * x * x)"),
    ("full layers from L5", "const bool full = layer % 5 == 4;", "const bool full = layer % 5 == 0;"),
    ("kv on all layers", "*kv = layer < 15 ? head_dim : 0;", "*kv = head_dim;"),
    ("chain gate and up swapped", "m[i] = f16_bits(gelu_tanh_value((double)g[i]) * (double)u[i]);",
     "m[i] = f16_bits(gelu_tanh_value((double)u[i]) * (double)g[i]);"),
    ("chain mid-layer norm dropped", "  for (int i = 0; i < H; ++i) t[i] = (double)o[i];\n  rms_to_f16(t.data(), H, b);",
     "  for (int i = 0; i < H; ++i) b[i] = f16_bits((double)o[i]);"),
    ("chain pre-attention norm dropped", "  for (int i = 0; i < H; ++i) t[i] = f16_value(h[i]);\n  rms_to_f16(t.data(), H, a);",
     "  for (int i = 0; i < H; ++i) a[i] = h[i];"),
]


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_some_pin_rejects_cpp_mutant(mutant, tmp_path):
    _, old, new = mutant
    src = open(cpp_oracle.SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mut_src = os.path.join(tmp_path, "q4_oracle_mutant.cpp")
    with open(mut_src, "w") as f:
        f.write(src.replace(old, new))
    lib_path = cpp_oracle.build(force=True, src=mut_src, out=os.path.join(tmp_path, "libmutant.so"))
    mod = cpp_oracle.Oracle(cpp_oracle.load(lib_path))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:   # any failure or crash counts as the pin biting
            caught.append(pin.__name__)
            break
    assert caught, f"no pin rejects C++ mutant {mutant[0]!r}"
