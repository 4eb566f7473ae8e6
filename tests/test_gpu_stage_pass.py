"""Fused decode-pass stages and the whole weight pass against the CPU oracle.

The synthetic 35-layer chain is chaotic: an fp32 implementation and the fp64
oracle drift apart by about 1.4x per layer (fp16 rounding forks amplified by
the random projections), so two correct implementations decorrelate after
~17 layers.  Parity is therefore established per stage, on seeded generator
inputs at every distinct E2B stage shape, plus one free-running layer; the
full pass is then shown to be exactly the composition of those stages
(bitwise), deterministic, finite and RMS-normalised.
"""
import numpy as np
import pytest
import torch

import int4_q4_weight_gb300 as q4w_mod
from int4_q4_weight_gb300 import synth
from oracle import q4_oracle as O
from parity import assert_close

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _mat(q4w, rows, cols, seed):
    W = synth.normal((rows, cols), 0.02, seed, "cuda")
    c, s = q4w.q4_quantize(W)
    oc, os_ = O.quantize_q4_0(W.cpu().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy(), oc)
    return (c, s), (oc, os_)


def _oracle_prologue(v, mode):
    v = np.asarray(v)
    if mode == q4w_mod.Q4_IN_F16:
        return v.astype(np.float16)
    if mode in (q4w_mod.Q4_IN_RMS_F16, q4w_mod.Q4_IN_RMS_F32):
        return O.to_f16(O.rmsnorm(v.astype(np.float64), eps=EPS))
    return O.to_f16(O.rmsnorm(O.to_f16(O.rmsnorm(v.astype(np.float64), eps=EPS)).astype(np.float64), eps=EPS))


def _input(mode, K, seed, scale=1.0):
    if mode in (q4w_mod.Q4_IN_F16, q4w_mod.Q4_IN_RMS_F16):
        return synth.normal_f16((K,), seed, "cuda")
    return synth.normal((K,), scale, seed, "cuda")


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("rows,K", [(96, 256), (1000, 1536), (33, 160), (513, 2048)])
def test_stage_prologues(cuda_lib, mode, rows, K):
    q4w = cuda_lib
    (c, s), (oc, os_) = _mat(q4w, rows, K, synth.sub_seed(31, rows, K))
    inp = _input(mode, K, synth.sub_seed(32, mode, K), scale=7.5)
    y = torch.empty(rows, dtype=torch.float32, device="cuda")
    y16 = torch.empty(rows, dtype=torch.float16, device="cuda")
    q4w.q4_gemv_stage([(c, s)], inp, mode, EPS, out32=[y], out16=[y16])
    torch.cuda.synchronize()
    yr = O.q4_gemv(oc, os_, _oracle_prologue(inp.cpu().numpy(), mode))
    assert_close(y.cpu().numpy(), yr, what=f"stage mode {mode}")
    assert np.array_equal(y16.cpu().numpy(), y.cpu().numpy().astype(np.float16))


def _qkv(q4w, Q, KV, H, seed, mode):
    mats, omats = [], []
    for i, r in enumerate([Q, KV, KV] if KV else [Q]):
        m, o = _mat(q4w, r, H, synth.sub_seed(seed, i))
        mats.append(m)
        omats.append(o)
    inp = _input(mode, H, synth.sub_seed(seed, "in"), scale=3.0)
    n = len(mats)
    o32 = [None] + [torch.empty(KV, dtype=torch.float32, device="cuda") for _ in range(n - 1)]
    o16 = [torch.empty(Q, dtype=torch.float16, device="cuda")] + [None] * (n - 1)
    q4w.q4_gemv_stage(mats, inp, mode, EPS, out32=o32, out16=o16)
    torch.cuda.synchronize()
    x = _oracle_prologue(inp.cpu().numpy(), mode)
    assert_close(o16[0].cpu().numpy(), O.to_f16(O.q4_gemv(*omats[0], x)), what="q16")
    for i in range(1, n):
        assert_close(o32[i].cpu().numpy(), O.q4_gemv(*omats[i], x), what=f"kv{i}")


def _gateup(q4w, I, H, seed, mode):
    (gc, gs), og = _mat(q4w, I, H, synth.sub_seed(seed, "g"))
    (uc, us), ou = _mat(q4w, I, H, synth.sub_seed(seed, "u"))
    inp = _input(mode, H, synth.sub_seed(seed, "in"), scale=2.0)
    m16 = torch.empty(I, dtype=torch.float16, device="cuda")
    g32 = torch.empty(I, dtype=torch.float32, device="cuda")
    u32 = torch.empty(I, dtype=torch.float32, device="cuda")
    q4w.q4_gemv_stage([(gc, gs), (uc, us)], inp, mode, EPS, pair=True, out32=[g32, u32],
                      out16=[m16, None])
    torch.cuda.synchronize()
    x = _oracle_prologue(inp.cpu().numpy(), mode)
    gr, ur = O.q4_gemv(*og, x), O.q4_gemv(*ou, x)
    assert_close(g32.cpu().numpy(), gr, what="gate")
    assert_close(u32.cpu().numpy(), ur, what="up")
    mr = O.to_f16(O.gelu_tanh(gr) * ur.astype(np.float64))
    assert_close(m16.cpu().numpy(), mr, what="m")


def _down(q4w, H, I, seed):
    (c, s), o = _mat(q4w, H, I, synth.sub_seed(seed, "d"))
    inp = _input(q4w_mod.Q4_IN_F16, I, synth.sub_seed(seed, "in"))
    y = torch.empty(H, dtype=torch.float32, device="cuda")
    q4w.q4_gemv_stage([(c, s)], inp, q4w_mod.Q4_IN_F16, EPS, out32=[y])
    torch.cuda.synchronize()
    assert_close(y.cpu().numpy(), O.q4_gemv(*o, inp.cpu().numpy()), what="down")


@pytest.mark.parametrize("layer", [0, 4, 15, 19])
def test_e2b_stage_shapes(cuda_lib, layer):
    """Every distinct stage shape of the E2B pass at full size."""
    d = synth.e2b_dims(layer)
    H = synth.E2B_HIDDEN
    seed = synth.sub_seed(40, layer)
    _qkv(cuda_lib, d["q"], d["kv"], H, seed, q4w_mod.Q4_IN_RMS2_F32)
    (oc_, os_), oo = _mat(cuda_lib, H, d["q"], synth.sub_seed(seed, "o"))
    q16 = synth.normal_f16((d["q"],), synth.sub_seed(seed, "q16"), "cuda")
    o32 = torch.empty(H, dtype=torch.float32, device="cuda")
    cuda_lib.q4_gemv_stage([(oc_, os_)], q16, q4w_mod.Q4_IN_F16, EPS, out32=[o32])
    torch.cuda.synchronize()
    assert_close(o32.cpu().numpy(), O.q4_gemv(*oo, q16.cpu().numpy()), what="o")
    _gateup(cuda_lib, d["mlp"], H, seed, q4w_mod.Q4_IN_RMS_F32)
    _down(cuda_lib, H, d["mlp"], seed)


def test_qkv_and_pair_small(cuda_lib):
    _qkv(cuda_lib, 96, 32, 128, 50, q4w_mod.Q4_IN_RMS_F16)
    _qkv(cuda_lib, 64, 0, 160, 51, q4w_mod.Q4_IN_RMS_F32)
    _gateup(cuda_lib, 77, 96, 52, q4w_mod.Q4_IN_RMS_F32)
    _gateup(cuda_lib, 1000, 1536, 53, q4w_mod.Q4_IN_F16)


def test_rmsnorm_f16(cuda_lib):
    y = synth.normal((1536,), 4.0, 54, "cuda")
    h = cuda_lib.q4_rmsnorm_f16(y, EPS)
    torch.cuda.synchronize()
    assert_close(h.cpu().numpy(), O.to_f16(O.rmsnorm(y.cpu().numpy().astype(np.float64), eps=EPS)),
                 what="rmsnorm")


# ---------------------------------------------------------------- pass ---
def _layers(q4w, dims_list, H, seed):
    gl, ol = [], []
    for li, d in enumerate(dims_list):
        shapes = {"q": (d["q"], H), "o": (H, d["q"]), "g": (d["mlp"], H), "u": (d["mlp"], H),
                  "d": (H, d["mlp"])}
        if d["kv"]:
            shapes["k"] = (d["kv"], H)
            shapes["v"] = (d["kv"], H)
        g, o = {}, {}
        for name, shp in shapes.items():
            W = synth.normal(shp, 0.02, synth.sub_seed(seed, li, name), "cuda")
            g[name] = q4w.q4_quantize(W)
            if ol is not None:
                o[name] = O.quantize_q4_0(W.cpu().numpy())
        gl.append(g)
        ol.append(o)
    torch.cuda.synchronize()
    return gl, ol


def _pass(q4w, gl, h0, H):
    ws = torch.empty(q4w.decode_pass_ws_bytes(gl, H), dtype=torch.uint8, device="cuda")
    h = torch.empty(H, dtype=torch.float16, device="cuda")
    q4w.q4_decode_pass(gl, h0, h, ws, EPS)
    torch.cuda.synchronize()
    return h


def _composed(q4w, gl, h0, H):
    """The same pass as separate stage calls (no programmatic dependent launch)."""
    y = None
    for li, g in enumerate(gl):
        Q = g["q"][0].shape[0]
        mats = [g["q"]] + ([g["k"], g["v"]] if "k" in g else [])
        q16 = torch.empty(Q, dtype=torch.float16, device="cuda")
        o32s = [None] + [torch.empty(m[0].shape[0], dtype=torch.float32, device="cuda") for m in mats[1:]]
        mode = q4w_mod.Q4_IN_RMS_F16 if li == 0 else q4w_mod.Q4_IN_RMS2_F32
        q4w.q4_gemv_stage(mats, h0 if li == 0 else y, mode, EPS, out32=o32s,
                          out16=[q16] + [None] * (len(mats) - 1))
        o = torch.empty(H, dtype=torch.float32, device="cuda")
        q4w.q4_gemv_stage([g["o"]], q16, q4w_mod.Q4_IN_F16, EPS, out32=[o])
        I = g["g"][0].shape[0]
        m = torch.empty(I, dtype=torch.float16, device="cuda")
        q4w.q4_gemv_stage([g["g"], g["u"]], o, q4w_mod.Q4_IN_RMS_F32, EPS, pair=True,
                          out16=[m, None])
        y = torch.empty(H, dtype=torch.float32, device="cuda")
        q4w.q4_gemv_stage([g["d"]], m, q4w_mod.Q4_IN_F16, EPS, out32=[y])
    h = q4w.q4_rmsnorm_f16(y, EPS)
    torch.cuda.synchronize()
    return h


def test_one_layer_free_running_small(cuda_lib):
    H = 256
    gl, ol = _layers(cuda_lib, [{"q": 512, "kv": 64, "mlp": 1024}], H, 60)
    h0 = synth.normal_f16((H,), 61, "cuda")
    h = _pass(cuda_lib, gl, h0, H)
    assert_close(h.cpu().numpy(), O.e2b_layer(h0.cpu().numpy(), ol[0], eps=EPS)["h"], what="layer")


@pytest.mark.parametrize("layer", [0, 19])
def test_one_e2b_layer_free_running(cuda_lib, layer):
    H = synth.E2B_HIDDEN
    gl, ol = _layers(cuda_lib, [synth.e2b_dims(layer)], H, 62 + layer)
    h0 = synth.e2b_h0(device="cuda")
    h = _pass(cuda_lib, gl, h0, H)
    assert_close(h.cpu().numpy(), O.e2b_layer(h0.cpu().numpy(), ol[0], eps=EPS)["h"],
                 what=f"E2B layer {layer}")


def test_pass_is_stage_composition_small(cuda_lib):
    H = 128
    dims = [{"q": 256, "kv": 32, "mlp": 384}, {"q": 192, "kv": 0, "mlp": 512},
            {"q": 256, "kv": 64, "mlp": 256}]
    gl, _ = _layers(cuda_lib, dims, H, 70)
    h0 = synth.normal_f16((H,), 71, "cuda")
    assert torch.equal(_pass(cuda_lib, gl, h0, H), _composed(cuda_lib, gl, h0, H))


@pytest.mark.parametrize("n", [48, 49])
def test_layer_count_across_the_persistent_limit(cuda_lib, n):
    """48 layers still run as one persistent launch, 49 as one launch per
    stage (4 n + 1 kernels); both equal the stage-by-stage composition bit
    for bit."""
    H = 256
    dims = [{"q": 256, "kv": 0 if i % 2 else 256, "mlp": 512} for i in range(n)]
    gl, _ = _layers(cuda_lib, dims, H, 74)
    assert cuda_lib.q4_decode_pass_launches(cuda_lib.make_layers(gl, H), H) == (1 if n <= 48 else 4 * n + 1)
    h0 = synth.normal_f16((H,), 75, "cuda")
    assert torch.equal(_pass(cuda_lib, gl, h0, H), _composed(cuda_lib, gl, h0, H))


def test_full_e2b_pass(cuda_lib):
    """35 E2B layers: deterministic, finite, RMS-normalised, and bitwise equal to
    the stage-by-stage composition whose stages are oracle-checked above."""
    q4w = cuda_lib
    H = synth.E2B_HIDDEN
    gl = []
    for layer in range(synth.E2B_N_LAYERS):
        g = {}
        for name in synth.e2b_matrix_shapes(layer):
            W = synth.e2b_weight(1003, layer, name, "cuda")
            g[name] = q4w.q4_quantize(W)
            del W
        gl.append(g)
    h0 = synth.e2b_h0(device="cuda")
    h1 = _pass(q4w, gl, h0, H)
    h2 = _pass(q4w, gl, h0, H)
    assert torch.equal(h1, h2)
    hv = h1.float()
    assert torch.isfinite(hv).all()
    assert abs(float((hv * hv).mean()) - 1.0) < 5e-3
    assert torch.equal(h1, _composed(q4w, gl, h0, H))


def test_persistent_pass_is_stage_composition(cuda_lib):
    """Shapes the persistent kernel takes (all K multiples of 256): its output
    equals the stage-by-stage launches bit for bit."""
    H = 512
    dims = [{"q": 768, "kv": 128, "mlp": 1280}, {"q": 1024, "kv": 0, "mlp": 2048},
            {"q": 512, "kv": 256, "mlp": 768}, {"q": 768, "kv": 0, "mlp": 1536}]
    gl, ol = _layers(cuda_lib, dims, H, 72)
    h0 = synth.normal_f16((H,), 73, "cuda")
    hp = _pass(cuda_lib, gl, h0, H)
    cuda_lib.q4_device_status()
    assert torch.equal(hp, _composed(cuda_lib, gl, h0, H))
    h1 = _pass(cuda_lib, gl[:1], h0, H)
    assert_close(h1.cpu().numpy(), O.e2b_layer(h0.cpu().numpy(), ol[0], eps=EPS)["h"], what="layer 0")
