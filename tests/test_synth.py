"""The seeded input generators: deterministic, independent per tensor, and with
the shapes and distributions of the workloads."""
import numpy as np
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O


def test_deterministic_and_independent():
    a = synth.normal((64, 32), 0.02, synth.sub_seed(1, "W"))
    b = synth.normal((64, 32), 0.02, synth.sub_seed(1, "W"))
    c = synth.normal((64, 32), 0.02, synth.sub_seed(1, "x"))
    assert torch.equal(a, b) and not torch.equal(a, c)


def test_distributions():
    W, x = synth.gemv_inputs(seed=3, N=512, K=1536)
    assert W.shape == (512, 1536) and W.dtype == torch.float32
    assert abs(W.std().item() - 0.02) < 0.0005 and abs(W.mean().item()) < 1e-3
    assert x.shape == (1, 1536) and x.dtype == torch.float16
    p = synth.ple_inputs(seed=3, S=64, V=1000, L=3, D=64)
    assert p.ids.dtype == torch.int32 and int(p.ids.min()) >= 0 and int(p.ids.max()) < 1000
    assert p.table.dtype == torch.int8 and int(p.table.min()) >= -127 and int(p.table.max()) <= 127
    assert float(p.row_scale.min()) >= 0.001 and float(p.row_scale.max()) <= 0.02
    assert float(p.norm_w.min()) >= 0.5 and float(p.norm_w.max()) <= 1.5


def test_e2b_shapes_agree_with_oracle_and_pages():
    total = 0
    for layer in range(synth.E2B_N_LAYERS):
        d1 = synth.e2b_dims(layer)
        d2 = O.e2b_layer_dims(layer)
        assert d1 == d2, layer
        total += sum(r * c for r, c in synth.e2b_matrix_shapes(layer).values())
    assert total == 1_835_532_288
    assert total * 9 // 16 == 1_032_486_912        # 0.5625 bytes per q4_0 weight
