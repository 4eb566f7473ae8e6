"""The int8 per-block-32 projection: the GPU quantiser bit for bit against the
oracle's, and the PLE on the int8 projection against the oracle.

Each side quantises the same seeded f32 projection with its own quantiser;
the codes and scales must agree bit for bit before the PLE outputs are
compared (the oracle then runs on its own codes)."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q8_oracle as Q8
from parity import assert_close

pytestmark = pytest.mark.gpu


def _quantize_both(q4w, W):
    codes, scales = q4w.q8_quantize(W)
    torch.cuda.synchronize()
    rc, rs = Q8.quantize_q8_0(W.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), rs)
    return codes, scales, rc, rs


def test_q8_quantize_edge_blocks(cuda_lib):
    """Zero blocks, exact ties, one-element blocks, mixed magnitudes, and a
    block whose step underflows fp32 (stored as zero)."""
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((6, 256)) * 0.02).astype(np.float32)
    W[0, :32] = 0.0
    d = 2.0 ** -6
    W[1, :32] = 0.0
    W[1, :6] = np.array([127, 2.5, -3.5, 0.5, -0.5, 126.5]) * d
    W[2, 32:64] = 0.0
    W[2, 40] = -3.0
    W[3, 64:96] = np.linspace(-1e4, 1e4, 32)
    W[4, 96:128] = np.float32(1e-44)          # subnormal: max / 127 is zero in fp32
    W[5, 128:160] = np.float32(3e-39)         # subnormal step
    _quantize_both(cuda_lib, torch.from_numpy(W).cuda())


def test_q8_quantize_projection_shape(cuda_lib):
    p = synth.ple_inputs(seed=1002, device="cuda", S=1, V=16)
    _quantize_both(cuda_lib, p.proj)


def _ple_q8_check(q4w, p, L, proj_zero=False):
    codes, scales, rc, rs = _quantize_both(q4w, p.proj)
    if proj_zero:
        codes.zero_()
        rc = np.zeros_like(rc)
    S = p.ids.numel()
    out, gathered = q4w.ple_gather_project_q8(
        p.ids, p.table, p.row_scale, codes, scales, p.hidden, p.norm_w, L=L,
        gathered=torch.empty((S, L * 256), dtype=torch.int8, device="cuda"))
    torch.cuda.synchronize()
    ro, rg = Q8.ple_gather_project_q8(p.ids.cpu().numpy(), p.table.cpu().numpy(), p.row_scale.cpu().numpy(),
                                      rc, rs, p.hidden.cpu().numpy(), p.norm_w.cpu().numpy(), L=L, ld=256)
    assert np.array_equal(gathered.cpu().numpy(), rg)
    if proj_zero:
        assert np.array_equal(out.cpu().numpy(), ro)
    else:
        assert_close(out.cpu().numpy(), ro, what="ple q8 out")


@pytest.mark.parametrize("S,V,L,D", [(5, 1000, 3, 128), (17, 333, 2, 1536), (64, 4096, 35, 1536),
                                     (1, 50, 1, 128), (9, 77, 2, 384), (33, 120, 1, 2048),
                                     (12, 200, 2, 1920)])   # K halves of 8 and 7 stages
def test_ple_q8_small(cuda_lib, S, V, L, D):
    p = synth.ple_inputs(seed=95, device="cuda", S=S, V=V, L=L, D=D)
    _ple_q8_check(cuda_lib, p, L)


@pytest.mark.parametrize("S,V,L,D", [(130, 900, 2, 128), (65, 300, 3, 1536), (4096, 100, 1, 128),
                                     (2, 50, 256, 128)])
def test_ple_q8_token_groups(cuda_lib, S, V, L, D):
    # several 64-token groups with a ragged last group
    p = synth.ple_inputs(seed=96, device="cuda", S=S, V=V, L=L, D=D)
    _ple_q8_check(cuda_lib, p, L)


def test_ple_q8_projection_term_alone(cuda_lib):
    # zero table bytes: the output is the normalised int8 projection alone
    p = synth.ple_inputs(seed=97, device="cuda", S=64, V=512, L=35, D=1536)
    p.table.zero_()
    _ple_q8_check(cuda_lib, p, 35)


def test_ple_q8_proj_zero_bit_exact(cuda_lib):
    p = synth.ple_inputs(seed=98, device="cuda", S=20, V=700, L=4, D=128)
    _ple_q8_check(cuda_lib, p, 4, proj_zero=True)


def test_ple_q8_bad_id(cuda_lib):
    p = synth.ple_inputs(seed=99, device="cuda", S=18, V=500, L=2, D=256)
    p.ids[3] = 500
    p.ids[17] = -1
    codes, scales, rc, rs = _quantize_both(cuda_lib, p.proj)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = cuda_lib.ple_gather_project_q8(p.ids, p.table, p.row_scale, codes, scales, p.hidden, p.norm_w,
                                            L=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert float(out[3].abs().max()) == 0.0 and float(out[17].abs().max()) == 0.0
    ok = [t for t in range(18) if t not in (3, 17)]
    ro, _ = Q8.ple_gather_project_q8(p.ids[ok].cpu().numpy(), p.table.cpu().numpy(), p.row_scale.cpu().numpy(),
                                     rc, rs, p.hidden[ok].cpu().numpy(), p.norm_w.cpu().numpy(), L=2, ld=256)
    assert_close(out[ok].cpu().numpy(), ro, what="ple q8 ok rows")


@pytest.mark.parametrize("S", [64, 1])
def test_ple_q8_full_config(cuda_lib, S):
    """The sidecar's full shape (V = 262144, L = 35, D = 1536), as timed."""
    p = synth.ple_inputs(seed=1002, device="cuda", S=S)
    _ple_q8_check(cuda_lib, p, 35)


def test_ple_q8_repeatable(cuda_lib):
    p = synth.ple_inputs(seed=100, device="cuda", S=64, V=1000, L=4, D=1536)
    codes, scales = cuda_lib.q8_quantize(p.proj)
    a = cuda_lib.ple_gather_project_q8(p.ids, p.table, p.row_scale, codes, scales, p.hidden, p.norm_w, L=4)[0].clone()
    b = cuda_lib.ple_gather_project_q8(p.ids, p.table, p.row_scale, codes, scales, p.hidden, p.norm_w, L=4)[0]
    torch.cuda.synchronize()
    assert torch.equal(a, b)
