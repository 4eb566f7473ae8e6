"""The w4a8 activation quantize/dequantize pair on the GPU against the oracle:
the min-max calibration bit for bit, the integer codes through exact
single-column products (ties, saturation, a tie that only the fp32 quotient
decides), and the GEMV / S=64 GEMM on the dequantised activations
elementwise.

Tolerances: with integer codes every block's dot product is exact in fp32,
so the GEMV's error is the fp32 sum of at most K/32 rounded block terms,
far inside 2e-5 of the rms-scaled result; the GEMM keeps the shared 2e-3
(tensor-core accumulation in its own order)."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import a8_oracle as A8
from oracle import q4_oracle as O
from parity import assert_close

pytestmark = pytest.mark.gpu
GEMV_TOL = 2e-5


def _quant(q4w, N, K, seed):
    W = synth.normal((N, K), 0.02, seed, "cuda")
    c, s = q4w.q4_quantize(W)
    torch.cuda.synchronize()
    return c, s, c.cpu().numpy(), s.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("n", [1, 7, 1001, 128 * 1536])
def test_calibrate_bit_exact(cuda_lib, n):
    x = (synth.normal_f16((n,), synth.sub_seed(40, n), "cuda").float() * 3.0).half()
    s = cuda_lib.q4_act_calibrate_a8(x)
    torch.cuda.synchronize()
    assert s.cpu().numpy()[0] == A8.a8_calibrate(x.cpu().numpy())
    z = cuda_lib.q4_act_calibrate_a8(torch.zeros((2, 8), dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    assert float(z.cpu()[0]) == 1.0


def test_codes_exact_single_column(cuda_lib):
    """x = v e_k: y = s * d (c - 8) q exactly (a 23-bit integer product times
    s, one rounding), so every integer decision is visible: ties to even,
    saturation, and a tie only the fp32 quotient produces."""
    N, K = 40, 96
    c, sc, oc, os_ = _quant(cuda_lib, N, K, synth.sub_seed(41))
    Wd = O.dequantize_q4_0(oc, os_)
    cases = [(0.5, 2.0 ** -4, 5), (1.5 * 2.0 ** -4, 2.0 ** -4, 10), (2.5 * 2.0 ** -4, 2.0 ** -4, 31),
             (-2.5 * 2.0 ** -4, 2.0 ** -4, 32), (60000.0, 1.0, 0), (-60000.0, 1.0, 95),
             (1.001953125, 0.40078124, 63), (-1.001953125, 0.40078124, 64), (0.01, 0.5, 7)]
    for v, s, k in cases:
        x = torch.zeros(K, dtype=torch.float16, device="cuda")
        x[k] = v
        y = cuda_lib.q4_gemv_a8(c, sc, x, s)
        torch.cuda.synchronize()
        q = int(A8.a8_quantize(np.array([v], np.float16), s)[0])
        want = (Wd[:, k] * q).astype(np.float32) * np.float32(s)
        assert np.array_equal(y.cpu().numpy(), want), (v, s, k, q)


@pytest.mark.parametrize("N,K", [(2048, 1536), (1, 32), (513, 160), (300, 2048), (129, 6144), (64, 12288),
                                 (7, 32768), (1536, 6144)])
def test_gemv_a8_parity(cuda_lib, N, K):
    c, sc, oc, os_ = _quant(cuda_lib, N, K, synth.sub_seed(42, N, K))
    x = synth.normal_f16((K,), synth.sub_seed(43, K), "cuda")
    for s in (float(A8.a8_calibrate(x.cpu().numpy())), 0.004):   # calibrated; many codes saturated
        y = cuda_lib.q4_gemv_a8(c, sc, x, s)
        torch.cuda.synchronize()
        assert_close(y.cpu().numpy(), A8.q4_gemv_a8(oc, os_, x.cpu().numpy(), s), tol=GEMV_TOL,
                     what=f"gemv_a8 {N}x{K} s={s}")


def test_gemv_a8_on_grid_is_q4_gemv(cuda_lib):
    """Activations on the grid: the QDQ is the identity, so q4_gemv_a8 agrees
    with q4_gemv (and both with the oracle)."""
    N, K = 2048, 1536
    c, sc, oc, os_ = _quant(cuda_lib, N, K, synth.sub_seed(44))
    s = 2.0 ** -5
    g = torch.Generator().manual_seed(45)
    x = (torch.randint(-128, 128, (K,), generator=g).float() * s).half().cuda()
    ya = cuda_lib.q4_gemv_a8(c, sc, x, s)
    yp = cuda_lib.q4_gemv(c, sc, x)
    torch.cuda.synchronize()
    yr = O.q4_gemv(oc, os_, x.cpu().numpy())
    assert_close(ya.cpu().numpy(), yr, tol=GEMV_TOL, what="on grid, a8")
    assert_close(yp.cpu().numpy(), yr, what="on grid, plain")


@pytest.mark.parametrize("N,K", [(256, 512), (6144, 1536), (1536, 6144), (128, 64)])
def test_gemm_chunk_a8_parity(cuda_lib, N, K):
    c, sc, oc, os_ = _quant(cuda_lib, N, K, synth.sub_seed(46, N, K))
    X = synth.normal_f16((64, K), synth.sub_seed(47, K), "cuda")
    s = float(A8.a8_calibrate(X.cpu().numpy()))
    Y = cuda_lib.q4_gemm_chunk_a8(c, sc, X, s)
    torch.cuda.synchronize()
    assert_close(Y.cpu().numpy(), A8.q4_gemm_chunk_a8(oc, os_, X.cpu().numpy(), s), what=f"gemm_a8 {N}x{K}")


def test_a8_rejects_bad_scales(cuda_lib):
    c, sc, _, _ = _quant(cuda_lib, 128, 64, synth.sub_seed(48))
    x = torch.ones(64, dtype=torch.float16, device="cuda")
    X = torch.ones((64, 64), dtype=torch.float16, device="cuda")
    for s in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(cuda_lib.Q4Error):
            cuda_lib.q4_gemv_a8(c, sc, x, s)
        with pytest.raises(cuda_lib.Q4Error):
            cuda_lib.q4_gemm_chunk_a8(c, sc, X, s)
