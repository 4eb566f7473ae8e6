"""Bounded device-side waits: with a zero cycle budget every kernel that waits
on an mbarrier or on other CTAs gives up at once, returns, and the library
reports Q4_ERR_TIMEOUT; the context stays usable and a normal budget gives
correct results again.  No fault, trap or hang is involved."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import assert_close

pytestmark = pytest.mark.gpu


def _expect_timeout(q4w):
    with pytest.raises(q4w.Q4Error, match="Q4_ERR_TIMEOUT"):
        q4w.q4_device_status()


def test_zero_budget_times_out_then_recovers(cuda_lib):
    q4w = cuda_lib
    q4w.q4_device_status()                 # clean start
    W, X = synth.gemm_inputs(seed=110, device="cuda", N=512, K=1536)
    codes, scales = q4w.q4_quantize(W)
    x1 = X[0].contiguous()
    Wg = synth.normal((65536, 1536), 0.02, synth.sub_seed(113), "cuda")   # many tiles per CTA:
    gc, gs = q4w.q4_quantize(Wg)                                         # the ring must wrap
    del Wg
    layers = []
    for i in range(2):
        g = {}
        for name, shp in (("q", (512, 256)), ("o", (256, 512)), ("g", (768, 256)), ("u", (768, 256)),
                          ("d", (256, 768))):
            g[name] = q4w.q4_quantize(synth.normal(shp, 0.02, synth.sub_seed(111, i, name), "cuda"))
        layers.append(g)
    h0 = synth.normal_f16((256,), 112, "cuda")
    ws = torch.empty(q4w.decode_pass_ws_bytes(layers, 256), dtype=torch.uint8, device="cuda")
    h = torch.empty(256, dtype=torch.float16, device="cuda")
    pp = synth.ple_inputs(seed=114, device="cuda", S=70, V=300, L=2, D=1536)
    old = q4w.q4_set_wait_limit(0)
    try:
        # several tiles per CTA, so that some wait outlasts the hardware's own
        # suspend window of mbarrier.try_wait and the zero budget is seen
        q4w.q4_gemm_chunk(gc, gs, X)
        _expect_timeout(q4w)
        q4w.q4_gemv(gc, gs, x1)                  # streaming GEMV (K = 1536)
        _expect_timeout(q4w)
        q4w.q4_decode_pass(layers, h0, h, ws)    # persistent pass
        _expect_timeout(q4w)
        q4w.ple_gather_project(pp.ids, pp.table, pp.row_scale, pp.proj, pp.hidden, pp.norm_w, L=2)
        _expect_timeout(q4w)                     # PLE: clusters of four still meet at every barrier
    finally:
        q4w.q4_set_wait_limit(old)
    Y = q4w.q4_gemm_chunk(codes, scales, X)
    y = q4w.q4_gemv(codes, scales, x1)
    q4w.q4_device_status()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    assert_close(Y.cpu().numpy(), O.q4_gemm_chunk(oc, os_, X.cpu().numpy()), what="gemm after")
    assert_close(y.cpu().numpy(), O.q4_gemv(oc, os_, x1.cpu().numpy()), what="gemv after")
    out, _ = q4w.ple_gather_project(pp.ids, pp.table, pp.row_scale, pp.proj, pp.hidden, pp.norm_w, L=2)
    q4w.q4_device_status()
    ro, _ = O.ple_gather_project(pp.ids.cpu().numpy(), pp.table.cpu().numpy(), pp.row_scale.cpu().numpy(),
                                 pp.proj.cpu().numpy(), pp.hidden.cpu().numpy(), pp.norm_w.cpu().numpy(), L=2, ld=256)
    assert_close(out.cpu().numpy(), ro, what="ple after")


def test_zero_budget_int8_ple_times_out_then_recovers(cuda_lib):
    """The int8 PLE form shares the clusters' bounded waits and abort path."""
    from oracle import q8_oracle as Q8
    q4w = cuda_lib
    q4w.q4_device_status()
    pp = synth.ple_inputs(seed=115, device="cuda", S=70, V=300, L=2, D=1536)
    codes, scales = q4w.q8_quantize(pp.proj)
    old = q4w.q4_set_wait_limit(0)
    try:
        q4w.ple_gather_project_q8(pp.ids, pp.table, pp.row_scale, codes, scales, pp.hidden, pp.norm_w, L=2)
        _expect_timeout(q4w)
    finally:
        q4w.q4_set_wait_limit(old)
    out, _ = q4w.ple_gather_project_q8(pp.ids, pp.table, pp.row_scale, codes, scales, pp.hidden, pp.norm_w, L=2)
    q4w.q4_device_status()
    rc, rs = Q8.quantize_q8_0(pp.proj.cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), rc)
    ro, _ = Q8.ple_gather_project_q8(pp.ids.cpu().numpy(), pp.table.cpu().numpy(), pp.row_scale.cpu().numpy(),
                                     rc, rs, pp.hidden.cpu().numpy(), pp.norm_w.cpu().numpy(), L=2, ld=256)
    assert_close(out.cpu().numpy(), ro, what="ple q8 after")
