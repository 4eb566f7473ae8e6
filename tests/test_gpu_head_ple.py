"""LM head + softcap + argmax and the PLE gather + projection against the oracle."""
import numpy as np
import pytest
import torch

from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import MARGIN_EXEMPT, assert_close

pytestmark = pytest.mark.gpu


def _head_check(q4w, codes, scales, h, oc, os_, want_logits=True):
    V = codes.shape[0]
    b = h.shape[0]
    logits = torch.empty((b, V), dtype=torch.float32, device="cuda") if want_logits else None
    idx, t1, t2, _ = q4w.lmhead_softcap_argmax(codes, scales, h, logits=logits)
    torch.cuda.synchronize()
    ri, r1, r2, margin, rs = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())
    gi = idx.cpu().numpy()
    for i in range(b):
        if margin[i] >= MARGIN_EXEMPT:
            assert gi[i] == ri[i], (i, gi[i], ri[i], margin[i])
        else:      # near tie: the GPU's pick must be one of the tied maxima
            assert rs[i, gi[i]] >= r1[i] - MARGIN_EXEMPT
    assert_close(t1.cpu().numpy(), r1, what="top1")
    assert_close(t2.cpu().numpy(), r2, what="top2")
    assert np.all(np.abs(t1.cpu().numpy()) < 30.0)
    if want_logits:
        assert_close(logits.cpu().numpy(), rs, what="logits")
    return gi, margin


@pytest.mark.parametrize("V,K,b", [(1000, 1536, 1), (4099, 256, 1), (77, 96, 1), (3000, 1536, 8),
                                   (513, 160, 3), (2, 32, 1), (5000, 2048, 2), (300, 32768, 1),
                                   (40, 25024, 4), (33, 12864, 8)])
def test_head_small(cuda_lib, V, K, b):
    W, h = synth.head_inputs(seed=80, device="cuda", batch=b, V=V, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    oc, os_ = O.quantize_q4_0(W.cpu().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), oc)
    _head_check(cuda_lib, codes, scales, h, oc, os_)


@pytest.mark.parametrize("K,b", [(25056, 2), (12896, 5)])
def test_head_batch_beyond_shared_memory_is_refused(cuda_lib, K, b):
    """b >= 2 off the tensor-core path stages every batch row's x in shared
    memory: one block more than fits (K 25024 for b <= 4, 12864 for b <= 8)
    is a shape error, not a launch."""
    W, h = synth.head_inputs(seed=82, device="cuda", batch=b, V=64, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    with pytest.raises(cuda_lib.Q4Error, match="does not fit"):
        cuda_lib.lmhead_softcap_argmax(codes, scales, h)


def test_head_ties_lowest_index(cuda_lib):
    V, K = 2000, 256
    W, h = synth.head_inputs(seed=81, device="cuda", batch=4, V=V, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    torch.cuda.synchronize()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    ri = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())[0]
    for b in range(4):        # copy each winner to a lower and a higher row
        w = int(ri[b])
        for dst in (max(0, w - 37 - b), min(V - 1, w + 11 + b)):
            codes[dst] = codes[w]
            scales[dst] = scales[w]
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    gi, margin = _head_check(cuda_lib, codes, scales, h, oc, os_, want_logits=False)
    ri2 = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())[0]
    assert np.array_equal(gi, ri2)


@pytest.mark.parametrize("b", [1, 8])
def test_head_full_vocab(cuda_lib, b):
    W, h = synth.head_inputs(seed=1004, device="cuda", batch=b)
    codes, scales = cuda_lib.q4_quantize(W)
    torch.cuda.synchronize()
    oc = codes.cpu().numpy()
    os_ = scales.cpu().numpy().view(np.uint16)
    rows = np.random.default_rng(2).integers(0, W.shape[0], 256)
    qc, qs = O.quantize_q4_0(W[torch.from_numpy(rows).cuda()].cpu().numpy())
    assert np.array_equal(oc[rows], qc) and np.array_equal(os_[rows], qs)
    del W
    _head_check(cuda_lib, codes, scales, h, oc, os_, want_logits=(b == 1))


@pytest.mark.parametrize("b", [2, 3, 8])
def test_head_batch_tensor_core_path(cuda_lib, b):
    # V a multiple of 128 with at least one 128-row tile per SM: batch rows go
    # through the tensor-core kernel (fp16 weight tiles) whose epilogue
    # softcaps and selects, including its softcapped logits output and a
    # repeat with the same bits
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    V, K = 128 * (sms + 9), 1536
    W, h = synth.head_inputs(seed=83 + b, device="cuda", batch=b, V=V, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    torch.cuda.synchronize()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    _head_check(cuda_lib, codes, scales, h, oc, os_, want_logits=True)
    a = [t.clone() for t in cuda_lib.lmhead_softcap_argmax(codes, scales, h)[:3]]
    c = cuda_lib.lmhead_softcap_argmax(codes, scales, h)[:3]
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, c))


def test_head_tensor_core_ties_lowest_index(cuda_lib):
    # each winner copied to rows in other 128-row tiles (other CTAs) below and
    # above it: the merged pick is the lowest tied row, the runner-up the tie
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    V, K, b = 128 * (sms + 9), 1536, 4
    W, h = synth.head_inputs(seed=90, device="cuda", batch=b, V=V, K=K)
    codes, scales = cuda_lib.q4_quantize(W)
    torch.cuda.synchronize()
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    ri = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())[0]
    for i in range(b):
        w = int(ri[i])
        for dst in ((w - 128 * (37 + i) - 5) % V, (w + 128 * (5 + i) + 3) % V):
            codes[dst] = codes[w]
            scales[dst] = scales[w]
    oc, os_ = codes.cpu().numpy(), scales.cpu().numpy().view(np.uint16)
    gi, _ = _head_check(cuda_lib, codes, scales, h, oc, os_, want_logits=False)
    ri2, r1, r2 = O.lmhead_softcap_argmax(oc, os_, h.cpu().numpy())[:3]
    assert np.array_equal(gi, ri2)
    _, t1, t2, _ = cuda_lib.lmhead_softcap_argmax(codes, scales, h)
    torch.cuda.synchronize()
    tie = r1 == r2            # the copied winner is the runner-up
    assert tie.any()
    assert np.array_equal(t1.cpu().numpy()[tie], t2.cpu().numpy()[tie])


def test_head_repeatable(cuda_lib):
    W, h = synth.head_inputs(seed=82, device="cuda", batch=2, V=3000, K=512)
    codes, scales = cuda_lib.q4_quantize(W)
    ws = cuda_lib.lmhead_ws(3000, 512, 2, "cuda")
    a = [t.clone() for t in cuda_lib.lmhead_softcap_argmax(codes, scales, h, ws=ws)[:3]]
    b = cuda_lib.lmhead_softcap_argmax(codes, scales, h, ws=ws)[:3]
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


# ----------------------------------------------------------------- PLE ---
def _ple_check(q4w, p, L, proj_zero=False, tol=None):
    out, gathered = q4w.ple_gather_project(
        p.ids, p.table, p.row_scale, p.proj, p.hidden, p.norm_w, L=L,
        gathered=torch.empty((p.ids.numel(), L * 256), dtype=torch.int8, device="cuda"))
    torch.cuda.synchronize()
    ro, rg = O.ple_gather_project(p.ids.cpu().numpy(), p.table.cpu().numpy(),
                                  p.row_scale.cpu().numpy(), p.proj.cpu().numpy(),
                                  p.hidden.cpu().numpy(), p.norm_w.cpu().numpy(), L=L, ld=256)
    assert np.array_equal(gathered.cpu().numpy(), rg)
    if proj_zero:
        assert np.array_equal(out.cpu().numpy(), ro)
    else:
        assert_close(out.cpu().numpy(), ro, what="ple out", **({} if tol is None else {"tol": tol}))


@pytest.mark.parametrize("S,V,L,D", [(5, 1000, 3, 64), (17, 333, 2, 1536), (64, 4096, 35, 1536),
                                     (1, 50, 1, 32), (3, 50, 1, 32768)])
def test_ple_small(cuda_lib, S, V, L, D):
    p = synth.ple_inputs(seed=90, device="cuda", S=S, V=V, L=L, D=D)
    _ple_check(cuda_lib, p, L)


@pytest.mark.parametrize("S,V,L,D", [(130, 900, 2, 96), (65, 300, 3, 1536), (4096, 100, 1, 64),
                                     (2, 50, 256, 64)])
def test_ple_token_groups(cuda_lib, S, V, L, D):
    # several 64-token groups with a ragged last group
    p = synth.ple_inputs(seed=94, device="cuda", S=S, V=V, L=L, D=D)
    _ple_check(cuda_lib, p, L)


def test_ple_projection_term_alone(cuda_lib):
    # zero table bytes: out is the normalised projection alone, so the
    # projection's own error is not hidden behind the larger gathered term;
    # the f32 projection is multiplied as two fp16 pieces (22 bits of each
    # weight) with fp32 accumulation, so it is held to 1e-4, well inside the
    # 2e-3 parity rule
    p = synth.ple_inputs(seed=93, device="cuda", S=64, V=512, L=35, D=1536)
    p.table.zero_()
    _ple_check(cuda_lib, p, 35, tol=1e-4)


def test_ple_proj_zero_bit_exact(cuda_lib):
    p = synth.ple_inputs(seed=91, device="cuda", S=20, V=700, L=4, D=96)
    p.proj.zero_()
    _ple_check(cuda_lib, p, 4, proj_zero=True)


def test_ple_bad_id(cuda_lib):
    p = synth.ple_inputs(seed=92, device="cuda", S=18, V=500, L=2, D=64)
    p.ids[3] = 500
    p.ids[17] = -1
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, _ = cuda_lib.ple_gather_project(p.ids, p.table, p.row_scale, p.proj, p.hidden, p.norm_w,
                                         L=2, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert float(out[3].abs().max()) == 0.0 and float(out[17].abs().max()) == 0.0
    ok = [t for t in range(18) if t not in (3, 17)]
    ro, _ = O.ple_gather_project(p.ids[ok].cpu().numpy(), p.table.cpu().numpy(),
                                 p.row_scale.cpu().numpy(), p.proj.cpu().numpy(),
                                 p.hidden[ok].cpu().numpy(), p.norm_w.cpu().numpy(), L=2, ld=256)
    assert_close(out[ok].cpu().numpy(), ro, what="ple ok rows")


@pytest.mark.parametrize("S", [64, 1])
def test_ple_full_config(cuda_lib, S):
    p = synth.ple_inputs(seed=1002, device="cuda", S=S)
    _ple_check(cuda_lib, p, 35)
