"""GPU INT2 per-row symmetric GEMV (q2_gemv) against the CPU oracle."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q2_oracle as Q
from parity import assert_close

pytestmark = pytest.mark.gpu

# ragged rows, one chunk per row up to the full shapes of the mixed-bit recipe
SHAPES = [(1, 64), (7, 192), (130, 320), (1000, 1536), (333, 4096), (12288, 1536), (1536, 12288), (5, 32768)]


@pytest.mark.parametrize("N,K", SHAPES)
def test_q2_gemv_matches_oracle(cuda_lib, N, K):
    codes, scales, x = synth.q2_inputs(seed=synth.sub_seed(31, N, K), device="cuda", N=N, K=K)
    y = cuda_lib.q2_gemv(codes, scales, x[0])
    torch.cuda.synchronize()
    ref = Q.q2_gemv(codes.cpu().numpy(), scales.cpu().numpy(), x[0].cpu().numpy())
    assert_close(y.cpu().numpy(), ref, what=f"q2_gemv {N}x{K}")


def test_q2_gemv_head_sampled_rows(cuda_lib):
    """The tied-head shape [262144, 1536]: every output, checked on 2048 sampled rows."""
    N, K = synth.Q2_SHAPES["head"]
    codes, scales, x = synth.q2_inputs(seed=1007, device="cuda", N=N, K=K)
    y = cuda_lib.q2_gemv(codes, scales, x[0]).cpu().numpy()
    rows = np.random.default_rng(3).choice(N, 2048, replace=False)
    rows.sort()
    idx = torch.from_numpy(rows).to("cuda")
    ref = Q.q2_gemv(codes[idx].cpu().numpy(), scales[idx].cpu().numpy(), x[0].cpu().numpy())
    assert_close(y[rows], ref, what="q2 head rows")
    assert np.isfinite(y).all()


def test_q2_gemv_constant_codes(cuda_lib):
    """codes all 3 -> scale * sum(x); all 0 -> -2 * scale * sum(x) (special cases)."""
    N, K = 96, 1536
    _, scales, x = synth.q2_inputs(seed=1008, device="cuda", N=N, K=K)
    sx = float(x[0].double().sum())
    for byte, factor in ((0xFF, 1.0), (0x00, -2.0)):
        codes = torch.full((N, K // 4), byte, dtype=torch.uint8, device="cuda")
        y = cuda_lib.q2_gemv(codes, scales, x[0]).cpu().numpy()
        ref = factor * sx * scales.cpu().numpy().astype(np.float64)
        assert_close(y, ref, what=f"constant byte {byte:#x}")


def test_q2_gemv_back_to_back_streams(cuda_lib):
    """Two calls in a row on different weights give each call's own result."""
    N, K = 4096, 1536
    c1, s1, x = synth.q2_inputs(seed=1009, device="cuda", N=N, K=K)
    c2, s2, _ = synth.q2_inputs(seed=1010, device="cuda", N=N, K=K)
    y1 = cuda_lib.q2_gemv(c1, s1, x[0])
    y2 = cuda_lib.q2_gemv(c2, s2, x[0])
    torch.cuda.synchronize()
    assert_close(y1.cpu().numpy(), Q.q2_gemv(c1.cpu().numpy(), s1.cpu().numpy(), x[0].cpu().numpy()))
    assert_close(y2.cpu().numpy(), Q.q2_gemv(c2.cpu().numpy(), s2.cpu().numpy(), x[0].cpu().numpy()))
