"""The LM head entry point that allocates nothing, called through the C ABI.

Callers that cannot allocate device memory (start-up-planned engines, plain C
hosts owning only their own buffers) use lmhead_softcap_argmax_noalloc, whose
scratch is a static device array inside the library.  Two calls in a row must
give what the workspace entry point gives, and what the CPU oracle gives.  This file is collected last so a
run that stops at the first failure has already run every other test; it also
passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import MARGIN_EXEMPT, assert_close

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, codes, scales, h, cap=30.0):
    V, K = codes.shape[0], codes.shape[1] * 2
    b = h.shape[0]
    idx = torch.full((b,), -1, dtype=torch.int32, device="cuda")
    t1 = torch.zeros(b, dtype=torch.float32, device="cuda")
    t2 = torch.zeros(b, dtype=torch.float32, device="cuda")
    st = lib.lmhead_softcap_argmax_noalloc(_p(codes), _p(scales), _p(h), b, V, K, cap, _p(idx), _p(t1),
                                           _p(t2), None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.q4_last_error().decode()
    return idx, t1, t2


def test_noalloc_head_matches_workspace_head(cuda_lib):
    q4w = cuda_lib
    lib = q4w.load()
    W, _ = synth.head_inputs(seed=120, device="cuda", batch=1, V=20000, K=1536)
    codes, scales = q4w.q4_quantize(W)
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    for call, b in enumerate((1, 8)):          # two calls in a row
        _, h = synth.head_inputs(seed=121 + call, device="cuda", batch=b, V=1, K=1536)
        gi, g1, g2 = _noalloc(lib, codes, scales, h)
        ri, r1, r2, _ = q4w.lmhead_softcap_argmax(codes, scales, h)
        torch.cuda.synchronize()
        margin = (r1 - r2).cpu().numpy()
        same = (gi == ri).cpu().numpy()
        assert np.all(same | (margin < MARGIN_EXEMPT)), (gi, ri)
        assert_close(g1.cpu().numpy(), r1.cpu().numpy(), what=f"top1 call {call}")
        assert_close(g2.cpu().numpy(), r2.cpu().numpy(), what=f"top2 call {call}")
        # and against the oracle (fp64 logits of the same codes)
        oi, o1, o2, om, _ = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())
        assert np.all((gi.cpu().numpy() == oi) | (om < MARGIN_EXEMPT)), (gi, oi)
        assert_close(g1.cpu().numpy(), o1, what=f"top1 vs oracle call {call}")
        assert_close(g2.cpu().numpy(), o2, what=f"top2 vs oracle call {call}")


def test_noalloc_head_batch_on_a_tensor_core_sized_vocabulary(cuda_lib):
    # a vocabulary that sends batch rows of the workspace entry point to the
    # tensor cores: the no-alloc entry keeps them on the CUDA cores (its static
    # scratch cannot hold the logits) and agrees within the parity tolerance
    q4w = cuda_lib
    lib = q4w.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    V = 128 * (sms + 3)
    W, h = synth.head_inputs(seed=124, device="cuda", batch=8, V=V, K=1536)
    codes, scales = q4w.q4_quantize(W)
    gi, g1, g2 = _noalloc(lib, codes, scales, h)
    ri, r1, r2, _ = q4w.lmhead_softcap_argmax(codes, scales, h)
    torch.cuda.synchronize()
    margin = (r1 - r2).cpu().numpy()
    same = (gi == ri).cpu().numpy()
    assert np.all(same | (margin < MARGIN_EXEMPT)), (gi, ri)
    assert_close(g1.cpu().numpy(), r1.cpu().numpy(), what="top1")
    assert_close(g2.cpu().numpy(), r2.cpu().numpy(), what="top2")
