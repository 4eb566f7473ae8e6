"""GPU quantiser and S=1 / batched GEMV against the CPU oracle."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import assert_close

pytestmark = pytest.mark.gpu

SHAPES = [(2048, 1536), (1000, 1536), (37, 96), (1, 32), (513, 160), (300, 2048), (129, 6144),
          (64, 12288), (7, 4096), (3, 224), (5, 32768)]


def _quant_both(q4w, W):
    codes, scales = q4w.q4_quantize(W)
    oc, os_ = O.quantize_q4_0(W.cpu().numpy())
    torch.cuda.synchronize()
    return codes, scales, oc, os_


@pytest.mark.parametrize("N,K", SHAPES)
def test_quantize_bit_exact(cuda_lib, N, K):
    W = synth.normal((N, K), 0.02, synth.sub_seed(21, N, K), "cuda")
    codes, scales, oc, os_ = _quant_both(cuda_lib, W)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)


def test_quantize_special_blocks(cuda_lib):
    q4w = cuda_lib
    rng = np.random.default_rng(5)
    W = (rng.standard_normal((8, 256)) * 0.02).astype(np.float32)
    W[0, :32] = 0.0                                    # zero block -> +0 and codes 8
    W[1, :32] = 0.0
    W[1, 3], W[1, 9] = 0.5, -0.5                       # equal magnitudes: first wins
    W[2, 32:64] = np.array([-2.0, 0.375, -0.375, 2.0, 0.125, -0.125, 1.75, 0.5, -1.0, 0.2] + [0] * 22,
                           np.float32)                 # the hand-worked block
    c = rng.integers(1, 16, 32)
    c[7] = 0
    W[3, 64:96] = (np.float32(np.float16(0.0123)) * (c - 8)).astype(np.float32)   # on the grid
    W[4, :32] = np.float32(1e-30)                      # fp16 scale underflows to 0
    W[5, 100] = np.float32(-3.0e-5)                    # subnormal fp16 scale
    W[5, 96:100] = 0
    W[5, 101:128] = 0
    Wt = torch.from_numpy(W).cuda()
    codes, scales, oc, os_ = _quant_both(q4w, Wt)
    assert np.array_equal(codes.cpu().numpy(), oc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint16), os_)
    assert int(os_[0, 0]) == 0 and int(os_[2, 1]) == 0x3400


def test_quantize_overflow_flag(cuda_lib):
    W = torch.zeros((2, 64), device="cuda")
    W[1, 40] = 1.0e6                                   # |d| = 125000 > fp16 max
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    codes, scales = cuda_lib.q4_quantize(W, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert float(scales[1, 1]) == 0.0 and int(codes[1, 16:].max()) == 0x88


def test_quantize_head_rows_sampled(cuda_lib):
    W, _ = synth.head_inputs(device="cuda", batch=1)
    codes, scales = cuda_lib.q4_quantize(W)
    torch.cuda.synchronize()
    rows = torch.tensor(np.r_[0:64, 262144 - 64:262144,
                              np.random.default_rng(1).integers(0, 262144, 384)], device="cuda")
    oc, os_ = O.quantize_q4_0(W[rows].cpu().numpy())
    assert np.array_equal(codes[rows].cpu().numpy(), oc)
    assert np.array_equal(scales[rows].cpu().numpy().view(np.uint16), os_)


GEMV_CASES = SHAPES + [(2048, 1536, 2), (300, 1536, 8), (37, 96, 3), (100, 6144, 8), (5, 32, 5),
                       (70, 12288, 4), (33, 160, 7), (9, 32768, 3)]


@pytest.mark.parametrize("case", GEMV_CASES)
def test_gemv_parity(cuda_lib, case):
    N, K = case[:2]
    batch = case[2] if len(case) > 2 else 1
    W, x = synth.gemv_inputs(seed=22, device="cuda", N=N, K=K, batch=batch)
    codes, scales, oc, os_ = _quant_both(cuda_lib, W)
    assert np.array_equal(codes.cpu().numpy(), oc)
    y = cuda_lib.q4_gemv(codes, scales, x if batch > 1 else x[0])
    torch.cuda.synchronize()
    yr = O.q4_gemv(oc, os_, x.cpu().numpy() if batch > 1 else x[0].cpu().numpy())
    assert_close(y.cpu().numpy(), yr, what=f"gemv {case}")


@pytest.mark.parametrize("N,K", [(40, 96), (17, 2048), (9, 160)])
def test_gemv_onehot_bit_exact(cuda_lib, N, K):
    """x = e_k selects column k of the dequantised matrix exactly."""
    W = synth.normal((N, K), 0.02, synth.sub_seed(23, N, K), "cuda")
    codes, scales = cuda_lib.q4_quantize(W)
    Wd = O.dequantize_q4_0(codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16))
    for k in (0, 1, 2, 31, 32, K - 2, K - 1):
        x = torch.zeros(K, dtype=torch.float16, device="cuda")
        x[k] = 1.0
        y = cuda_lib.q4_gemv(codes, scales, x)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), Wd[:, k].astype(np.float32)), k
    X = torch.zeros((3, K), dtype=torch.float16, device="cuda")
    X[0, 5], X[1, K - 1], X[2, 33] = 1.0, 1.0, 1.0
    Y = cuda_lib.q4_gemv(codes, scales, X)
    torch.cuda.synchronize()
    for b, k in enumerate((5, K - 1, 33)):
        assert np.array_equal(Y[b].cpu().numpy(), Wd[:, k].astype(np.float32))


def test_gemv_deterministic(cuda_lib):
    W, x = synth.gemv_inputs(seed=24, device="cuda")
    codes, scales = cuda_lib.q4_quantize(W)
    a = cuda_lib.q4_gemv(codes, scales, x[0]).clone()
    b = cuda_lib.q4_gemv(codes, scales, x[0])
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_gemv_weights_ro_same_bits_and_waits_for_x(cuda_lib):
    """The read-only-weights form computes q4_gemv's bits; back to back, and
    when its x comes from the kernel just before it (x must still be read only
    after that kernel's results are visible)."""
    W, x = synth.gemv_inputs(seed=27, device="cuda", N=2048, K=1536)
    codes, scales = cuda_lib.q4_quantize(W)
    W2 = synth.normal((1536, 2048), 0.02, synth.sub_seed(28), "cuda")
    c2, s2 = cuda_lib.q4_quantize(W2)
    torch.cuda.synchronize()                       # the weights exist before the promise starts
    ref = cuda_lib.q4_gemv(codes, scales, x[0]).clone()
    outs = [cuda_lib.q4_gemv_weights_ro(codes, scales, x[0]) for _ in range(6)]
    # a chain: y1 -> fp16 -> the next GEMV's x, each step on the read-only form
    y1 = cuda_lib.q4_gemv_weights_ro(codes, scales, x[0])
    x2 = y1.to(torch.float16)
    y2 = cuda_lib.q4_gemv_weights_ro(c2, s2, x2)
    y2_ref = cuda_lib.q4_gemv(c2, s2, x2.clone())
    torch.cuda.synchronize()
    for y in outs:
        assert torch.equal(y, ref)
    assert torch.equal(y1, ref) and torch.equal(y2, y2_ref)
    yr = O.q4_gemv(c2.cpu().numpy(), s2.cpu().numpy().view(np.uint16), x2.cpu().numpy())
    assert_close(y2.cpu().numpy(), yr, what="weights_ro chain")


def test_gemv_large_activations(cuda_lib):
    """fp16 x near the top of its range and many tiny ones (bias trick headroom)."""
    N, K = 256, 4096
    W = synth.normal((N, K), 0.02, synth.sub_seed(25), "cuda")
    x = (synth.normal((K,), 1.0, synth.sub_seed(26), "cuda") * 3000).to(torch.float16)
    x[::7] = 1e-4
    codes, scales = cuda_lib.q4_quantize(W)
    y = cuda_lib.q4_gemv(codes, scales, x)
    torch.cuda.synchronize()
    yr = O.q4_gemv(codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16), x.cpu().numpy())
    assert_close(y.cpu().numpy(), yr, what="large x")
