"""The Python binding's size checks, on CPU with a stand-in for the library.

The kernels trust the sizes they are given (N, K, S, L, D ...), so the binding
checks, before any call, that every array holds exactly the elements those
sizes imply; a short output or a table narrower than L*ld would otherwise be
overrun on the device.  Correctly sized calls must reach the library
unchanged, mis-sized ones must raise without reaching it."""
import pytest
import torch

import int4_q4_weight_gb300 as q4w


class _Lib:
    """Records which entry points were called; every call succeeds."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append(name)
            return 0
        return call


@pytest.fixture
def lib(monkeypatch):
    fake = _Lib()
    monkeypatch.setattr(q4w, "load", lambda: fake)
    monkeypatch.setattr(q4w, "_dev", lambda t, dtype, name: None)   # CPU tensors stand in
    monkeypatch.setattr(q4w, "_stream", lambda: None)
    return fake


def _z(shape, dtype):
    return torch.zeros(shape, dtype=dtype)


def _ple_args(S=5, V=7, L=2, D=128, q8=False):
    args = dict(ids=_z(S, torch.int32), table=_z((V, L * 256), torch.int8), row_scale=_z(V, torch.float32),
                hidden=_z((S, D), torch.float16), norm_w=_z(256, torch.float32))
    if q8:
        args.update(proj_codes=_z((L * 256, D), torch.int8), proj_scales=_z((L * 256, D // 32), torch.float16))
    else:
        args["proj"] = _z((L * 256, D), torch.float32)
    return args


def test_correct_sizes_reach_the_library(lib):
    N, K = 256, 128
    codes, scales = _z((N, K // 2), torch.uint8), _z((N, K // 32), torch.float16)
    q4w.q4_quantize(_z((N, K), torch.float32))
    q4w.q8_quantize(_z((N, K), torch.float32))
    q4w.q4_gemv(codes, scales, _z(K, torch.float16))                      # batch 1, x as a vector
    q4w.q4_gemv(codes, scales, _z((4, K), torch.float16), _z((4, N), torch.float32))
    q4w.lmhead_softcap_argmax(codes, scales, _z((2, K), torch.float16), logits=_z((2, N), torch.float32))
    q4w.q4_gemm_chunk(codes, scales, _z((64, K), torch.float16))
    q4w.q4_gemv_a8(codes, scales, _z(K, torch.float16), 0.01)
    q4w.q4_gemm_chunk_a8(codes, scales, _z((64, K), torch.float16), 0.01)
    q4w.q4_act_calibrate_a8(_z((128, K), torch.float16))
    q4w.q2_gemv(_z((N, K // 4), torch.uint8), _z(N, torch.float32), _z(K, torch.float16))
    a = _ple_args()
    q4w.ple_gather_project(a["ids"], a["table"], a["row_scale"], a["proj"], a["hidden"], a["norm_w"], L=2,
                           gathered=_z((5, 512), torch.int8))
    b = _ple_args(q8=True)
    q4w.ple_gather_project_q8(b["ids"], b["table"], b["row_scale"], b["proj_codes"], b["proj_scales"],
                              b["hidden"], b["norm_w"], L=2)
    assert lib.calls.count("q4_gemv") == 2
    for name in ("q4_quantize", "q8_quantize", "lmhead_softcap_argmax", "q4_gemm_chunk", "q2_gemv",
                 "ple_gather_project", "ple_gather_project_q8", "q4_gemv_a8", "q4_gemm_chunk_a8",
                 "q4_act_calibrate_a8"):
        assert name in lib.calls, name


def _rejects(lib, fn, what):
    with pytest.raises(q4w.Q4Error, match=what):
        fn()
    assert not [c for c in lib.calls if c != "q4_workspace_bytes"], lib.calls


def test_mis_sized_arrays_are_refused(lib):
    N, K = 256, 128
    codes, scales = _z((N, K // 2), torch.uint8), _z((N, K // 32), torch.float16)
    _rejects(lib, lambda: q4w.q4_gemv(codes, scales[:-1], _z(K, torch.float16)), "scales")
    _rejects(lib, lambda: q4w.q4_gemv(codes, scales, _z(K, torch.float16), _z(N - 1, torch.float32)), "y")
    _rejects(lib, lambda: q4w.q4_gemv(codes, scales, _z((2, K), torch.float16), _z(N, torch.float32)), "y")
    _rejects(lib, lambda: q4w.lmhead_softcap_argmax(codes, scales, _z((2, K), torch.float16),
                                                     logits=_z((1, N), torch.float32)), "logits")
    _rejects(lib, lambda: q4w.q4_gemm_chunk(codes, scales, _z((64, K), torch.float16),
                                            _z((64, N // 2), torch.float32)), "Y")
    _rejects(lib, lambda: q4w.q4_gemv_a8(codes, scales, _z(K - 32, torch.float16), 0.01), "x")
    _rejects(lib, lambda: q4w.q4_gemv_a8(codes, scales, _z(K, torch.float16), 0.01, _z(N + 1, torch.float32)), "y")
    _rejects(lib, lambda: q4w.q4_gemm_chunk_a8(codes, scales[:-1], _z((64, K), torch.float16), 0.01), "scales")
    _rejects(lib, lambda: q4w.q4_act_calibrate_a8(_z(8, torch.float16), out=_z(2, torch.float32)), "out")
    _rejects(lib, lambda: q4w.q2_gemv(_z((N, K // 4), torch.uint8), _z(N, torch.float32),
                                      _z(K // 2, torch.float16)), "x")
    _rejects(lib, lambda: q4w.q4_quantize(_z((N, K), torch.float32), codes=_z((N, K // 4), torch.uint8)), "codes")
    a = _ple_args()
    # a table narrower than L*ld (here L = 3 against a table built for L = 2)
    _rejects(lib, lambda: q4w.ple_gather_project(a["ids"], a["table"], a["row_scale"], a["proj"], a["hidden"],
                                                 a["norm_w"], L=3), "table")
    _rejects(lib, lambda: q4w.ple_gather_project(a["ids"], a["table"], a["row_scale"], a["proj"], a["hidden"],
                                                 a["norm_w"], L=2, out=_z((4, 512), torch.float32)), "out")
    _rejects(lib, lambda: q4w.ple_gather_project(a["ids"], a["table"], a["row_scale"], a["proj"],
                                                 a["hidden"][:4], a["norm_w"], L=2), "hidden")
    b = _ple_args(q8=True)
    _rejects(lib, lambda: q4w.ple_gather_project_q8(b["ids"], b["table"], b["row_scale"], b["proj_codes"],
                                                    b["proj_scales"][:-1], b["hidden"], b["norm_w"], L=2),
             "proj_scales")
    _rejects(lib, lambda: q4w.ple_gather_project_q8(b["ids"], b["table"], b["row_scale"], b["proj_codes"],
                                                    b["proj_scales"], b["hidden"], b["norm_w"], L=2,
                                                    gathered=_z((5, 256), torch.int8)), "gathered")


def _layer(H=64, Q=96, KV=32, I=128, kv=True):
    def m(r, c):
        return _z((r, c // 2), torch.uint8), _z((r, c // 32), torch.float16)
    lw = {"q": m(Q, H), "o": m(H, Q), "g": m(I, H), "u": m(I, H), "d": m(H, I)}
    if kv:
        lw.update(k=m(KV, H), v=m(KV, H))
    return lw


def test_stage_and_pass_shapes_reach_the_library(lib):
    K = 128
    g, u = (_z((64, K // 2), torch.uint8), _z((64, K // 32), torch.float16)), \
           (_z((64, K // 2), torch.uint8), _z((64, K // 32), torch.float16))
    q4w.q4_gemv_stage([g, u], _z(K, torch.float32), q4w.Q4_IN_RMS_F32, pair=True,
                      out32=[_z(64, torch.float32), None], out16=[_z(64, torch.float16), None])
    q4w.q4_rmsnorm_f16(_z(64, torch.float32))
    layers = [_layer(), _layer(kv=False)]
    q4w.q4_decode_pass(layers, _z(64, torch.float16), _z(64, torch.float16), _z(1, torch.uint8))
    descs = q4w.make_layers(layers, 64)
    q4w.q4_decode_pass(layers, _z(64, torch.float16), _z(64, torch.float16), _z(1, torch.uint8), descs=descs)
    assert lib.calls.count("q4_decode_pass") == 2
    assert "q4_gemv_stage" in lib.calls and "q4_rmsnorm_f16" in lib.calls


def test_mis_shaped_stage_and_pass_are_refused(lib):
    K = 128
    a = (_z((64, K // 2), torch.uint8), _z((64, K // 32), torch.float16))
    narrow = (_z((64, K // 4), torch.uint8), _z((64, K // 64), torch.float16))   # fewer columns than K
    x = _z(K, torch.float16)
    _rejects(lib, lambda: q4w.q4_gemv_stage([a, narrow], x, q4w.Q4_IN_F16), r"mats\[1\].codes")
    _rejects(lib, lambda: q4w.q4_gemv_stage([(a[0], a[1][:-1])], x, q4w.Q4_IN_F16), r"mats\[0\].scales")
    _rejects(lib, lambda: q4w.q4_gemv_stage([a], x[:-8], q4w.Q4_IN_F16), "in has")
    _rejects(lib, lambda: q4w.q4_gemv_stage([a], x, q4w.Q4_IN_F16, out32=[_z(63, torch.float32)]), r"out32\[0\]")
    _rejects(lib, lambda: q4w.q4_gemv_stage([a], x, q4w.Q4_IN_F16, out16=[_z(65, torch.float16)]), r"out16\[0\]")
    _rejects(lib, lambda: q4w.q4_gemv_stage([a, a, a, a], x, q4w.Q4_IN_F16), "1 to 3")
    _rejects(lib, lambda: q4w.q4_rmsnorm_f16(_z(64, torch.float32), out=_z(32, torch.float16)), "out")
    bad = _layer()
    bad["d"] = (_z((64, 32), torch.uint8), _z((64, 2), torch.float16))        # down narrower than the MLP
    h = _z(64, torch.float16)
    _rejects(lib, lambda: q4w.q4_decode_pass([_layer(), bad], h, h, _z(1, torch.uint8)), r"layers\[1\].d")
    _rejects(lib, lambda: q4w.q4_decode_pass([_layer()], _z(32, torch.float16), _z(32, torch.float16),
                                             _z(1, torch.uint8)), r"layers\[0\].q")    # h0 of another H
    _rejects(lib, lambda: q4w.q4_decode_pass([_layer()], h, _z(63, torch.float16), _z(1, torch.uint8)), "h_out")
    nov = _layer()
    del nov["v"]
    _rejects(lib, lambda: q4w.make_layers([nov], 64), "k and v")
    good = q4w.make_layers([_layer()], 64)
    _rejects(lib, lambda: q4w.q4_decode_pass([_layer(), _layer()], h, h, _z(1, torch.uint8), descs=good),
             "descs holds")


class _FakeCuda:
    """Stands in for a CUDA tensor on a given device (the check reads nothing else first)."""

    def __init__(self, index):
        self.is_cuda = True
        self.device = torch.device("cuda", index)
        self.dtype = torch.float16

    def is_contiguous(self):
        return True


def test_tensor_on_another_device_is_refused(monkeypatch):
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 0)
    q4w._dev(_FakeCuda(0), torch.float16, "x")                 # the current device passes
    with pytest.raises(q4w.Q4Error, match="cuda:1"):
        q4w._dev(_FakeCuda(1), torch.float16, "x")
