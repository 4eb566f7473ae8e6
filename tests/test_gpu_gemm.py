"""S=64 chunked-prefill GEMM on the tensor cores against the oracle's bf16-tile
contraction (both tiles rounded to bf16, then an exact sum)."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import assert_close, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K", [(128, 64), (256, 1536), (384, 320), (6144, 1536), (1536, 6144),
                                 (1280, 12288), (128, 32768)])
def test_gemm_parity(cuda_lib, N, K):
    W, X = synth.gemm_inputs(seed=100, device="cuda", N=N, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    Y = cuda_lib.q4_gemm_chunk(codes, scales, X)
    cuda_lib.q4_device_status()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    Yr = O.q4_gemm_chunk(oc, os_, X.cpu().numpy())
    assert_close(Y.cpu().numpy(), Yr, what=f"gemm {N}x{K}")


def test_gemm_onehot_bit_exact(cuda_lib):
    N, K = 256, 512
    W, _ = synth.gemm_inputs(seed=101, device="cuda", N=N, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    X = torch.zeros((64, K), dtype=torch.float16, device="cuda")
    ks = [(t * 37) % K for t in range(64)]
    for t, k in enumerate(ks):
        X[t, k] = 1.0
    Y = cuda_lib.q4_gemm_chunk(codes, scales, X)
    cuda_lib.q4_device_status()
    Wd = O.dequantize_q4_0(codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)).astype(np.float32)
    Wt = O.bf16_rne(Wd)
    want = np.stack([Wt[:, k] for k in ks])
    assert np.array_equal(Y.cpu().numpy(), want)


def test_gemm_head_shape(cuda_lib):
    W, X = synth.gemm_inputs(seed=1005, device="cuda", N=262144, K=1536)
    codes, scales = cuda_lib.q4_quantize(W)
    del W
    Y = cuda_lib.q4_gemm_chunk(codes, scales, X)
    cuda_lib.q4_device_status()
    rows = np.r_[0:256, 262144 - 256:262144, np.random.default_rng(3).integers(0, 262144, 512)]
    oc = codes[torch.from_numpy(rows).cuda()].cpu().numpy()
    os_ = scales[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint16)
    Yr = O.q4_gemm_chunk(oc, os_, X.cpu().numpy())
    assert_close(Y[:, torch.from_numpy(rows).cuda()].cpu().numpy(), Yr, what="head-shape gemm")


def test_gemm_tile_rounding_gap(cuda_lib):
    """The bf16 tiles stay within their rounding bound of the exact product."""
    W, X = synth.gemm_inputs(seed=102, device="cuda", N=512, K=1536)
    codes, scales = cuda_lib.q4_quantize(W)
    Y = cuda_lib.q4_gemm_chunk(codes, scales, X)
    cuda_lib.q4_device_status()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    Ye = O.q4_gemm_chunk_exact(oc, os_, X.cpu().numpy())
    Wd = np.abs(O.dequantize_q4_0(oc, os_))
    bound = (2 * 2.0 ** -9 + 2.0 ** -18) * (np.abs(X.cpu().numpy().astype(np.float64)) @ Wd.T) + 1e-6
    assert np.all(np.abs(Y.cpu().numpy() - Ye) <= bound * 1.01)
    assert rel_err(Y.cpu().numpy(), Ye) < 2e-2
