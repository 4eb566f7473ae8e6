"""The C-ABI library on a machine without a GPU: it builds, loads, exports every
symbol the header declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

import int4_q4_weight_gb300 as q4w

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4w.h")


@pytest.fixture(scope="module")
def lib():
    q4w.build()
    return q4w.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


def test_header_lists_the_entry_points():
    names = _declared_functions()
    for n in ("q4_gemv", "q4_gemm_chunk", "ple_gather_project", "lmhead_softcap_argmax",
              "q4_quantize", "q4_decode_pass", "q4_workspace_bytes", "q4_status_string",
              "q4_last_error"):
        assert n in names, n


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), f"libq4w.so does not export {n}"


def test_status_strings(lib):
    names = [lib.q4_status_string(i).decode() for i in range(9)]
    assert names == ["Q4_OK", "Q4_ERR_NULL", "Q4_ERR_SHAPE", "Q4_ERR_ALIGN", "Q4_ERR_WORKSPACE",
                     "Q4_ERR_ARCH", "Q4_ERR_CUDA", "Q4_ERR_TIMEOUT", "Q4_ERR_DEVICE"]
    assert lib.q4_status_string(99) == b"Q4_ERR_UNKNOWN"
    assert lib.q4_version() == 100


def test_decode_workspace_formula(lib):
    up = lambda n: (n + 255) // 256 * 256
    H, QKV, I = 1536, 4096 + 1024, 12288
    # k/v f32, then q, o, m, y in their tagged form (half|tag: 4 B, float|tag: 8 B),
    # then a 256-byte control block
    want = up(QKV * 4) + up(QKV * 4) + up(H * 8) + up(I * 4) + up(H * 8) + 256
    assert lib.q4_workspace_bytes(q4w.Q4_OP_DECODE_PASS, H, QKV, I) == want
    assert lib.q4_workspace_bytes(q4w.Q4_OP_GEMV, 10, 64, 1) == 0


A = 1 << 20  # an aligned, never-dereferenced stand-in address


def test_null_and_shape_rejections(lib):
    assert lib.q4_gemv(None, A, A, A, 16, 64, 1, None, 0, None) == 1
    assert b"codes" in lib.q4_last_error()
    assert lib.q4_gemv(A, A, A, A, 16, 48, 1, None, 0, None) == 2       # K % 32
    assert b"K=48" in lib.q4_last_error()
    assert lib.q4_gemv(A, A, A, A, 16, 64, 9, None, 0, None) == 2       # batch > 8
    assert lib.q4_gemv(A, A, A, A, 0, 64, 1, None, 0, None) == 2        # N < 1
    assert lib.q4_gemv(A, A, A, A, 16, 65536, 1, None, 0, None) == 2    # K too large
    assert lib.q4_gemv_weights_ro(None, A, A, A, 16, 64, 1, None, 0, None) == 1
    assert lib.q4_gemv_weights_ro(A, A, A, A, 16, 48, 1, None, 0, None) == 2
    assert lib.q4_gemm_chunk(A, A, A, A, 32, 128, 64, None, 0, None) == 2   # M != 64
    assert lib.q4_gemm_chunk(A, A, A, A, 64, 100, 64, None, 0, None) == 2   # N % 128
    assert lib.q4_gemm_chunk(A, A, A, A, 64, 128, 64, None, 0, None) == 4   # no workspace
    assert lib.q4_gemm_chunk(A, A, A, A, 64, 128, 1536, A, 1000, None) == 4  # workspace too small
    assert lib.q4_workspace_bytes(q4w.Q4_OP_GEMM_CHUNK, 128, 1536, 64) == 64 * 1536 * 2
    assert lib.ple_gather_project(A, 4, A, A, 10, 35, 128, 16.0, A, A, 64, A, 1e-6, A, None, None,
                                  None) == 2                                # ld != 256
    assert lib.lmhead_softcap_argmax(A, A, A, 9, 100, 64, 30.0, A, A, A, None, A, 1 << 20,
                                     None) == 2                             # b > 8
    assert lib.lmhead_softcap_argmax(A, A, A, 1, 100, 64, 0.0, A, A, A, None, A, 1 << 20,
                                     None) == 2                             # cap <= 0
    assert lib.q4_quantize(A, 4, 40, A, A, None, None) == 2


def test_alignment_rejection(lib):
    assert lib.q4_gemv(A + 4, A, A, A, 16, 64, 1, None, 0, None) == 3
    assert b"16-byte" in lib.q4_last_error()
    assert lib.q4_quantize(A, 4, 64, A, A + 2, None, None) == 3


def test_decode_pass_rejections(lib):
    layer = q4w.q4_layer()
    layer.q_rows, layer.kv_rows, layer.mlp_rows = 64, 0, 64
    assert lib.q4_decode_pass(ctypes.byref(layer), 1, 64, A, A, 1e-6, A, 1 << 20, None) == 1
    assert b"layers[0].q" in lib.q4_last_error()
    for f in ("q", "o", "gate", "up", "down"):
        setattr(layer, f, q4w.q4_matrix(A, A))
    layer.mlp_rows = 40
    assert lib.q4_decode_pass(ctypes.byref(layer), 1, 64, A, A, 1e-6, A, 1 << 20, None) == 2
    layer.mlp_rows = 64
    assert lib.q4_decode_pass(ctypes.byref(layer), 1, 64, A, A, 1e-6, A, 16, None) == 4   # ws small


def test_q2_gemv_rejections(lib):
    assert lib.q2_gemv(None, A, A, A, 4, 64, None) == 1                 # NULL
    assert lib.q2_gemv(A + 4, A, A, A, 4, 64, None) == 3                # alignment
    assert lib.q2_gemv(A, A, A, A, 4, 96, None) == 2                    # K % 64
    assert b"K=96" in lib.q4_last_error()
    assert lib.q2_gemv(A, A, A, A, 0, 64, None) == 2                    # N


def test_q8_entry_rejections(lib):
    F = ctypes.c_float
    assert lib.q8_quantize(None, 4, 64, A, A, None, None) == 1              # NULL
    assert lib.q8_quantize(A, 4, 48, A, A, None, None) == 2                 # K % 32
    assert lib.q8_quantize(A, 4, 64, A + 8, A, None, None) == 3             # alignment

    def ple(**kw):
        a = dict(ids=A, S=8, table=A, rs=A, V=10, L=2, ld=256, codes=A, scales=A, hid=A, D=128,
                 nw=A, out=A)
        a.update(kw)
        return lib.ple_gather_project_q8(a["ids"], a["S"], a["table"], a["rs"], a["V"], a["L"], a["ld"],
                                         F(16.0), a["codes"], a["scales"], a["hid"], a["D"], a["nw"],
                                         F(1e-6), a["out"], None, None, None)
    assert ple(scales=None) == 1
    assert b"proj_scales" in lib.q4_last_error()
    assert ple(codes=A + 4) == 3
    assert ple(D=192) == 2                                                  # D % 128
    assert b"D=192" in lib.q4_last_error()
    assert ple(D=2176) == 2                                                 # D > 2048
    assert ple(ld=128) == 2
    assert ple(S=0) == 2


def test_decode_pass_launch_count(lib):
    """One persistent launch when H <= 4096, every K a multiple of 256 up to
    12288 and at most 48 layers; otherwise one launch per stage plus the
    closing RMSNorm."""
    L = (q4w.q4_layer * 3)()
    for l in L:
        l.q_rows, l.kv_rows, l.mlp_rows = 2048, 256, 6144
    assert lib.q4_decode_pass_launches(L, 3, 1536) == 1
    assert lib.q4_decode_pass_launches(L, 3, 4352) == 13      # H above the staging limit
    assert lib.q4_decode_pass_launches(L, 3, 1568) == 13      # H not a multiple of 256
    L[1].mlp_rows = 16384                                      # K above 12288
    assert lib.q4_decode_pass_launches(L, 3, 1536) == 13
    assert lib.q4_decode_pass_launches(None, 3, 1536) == -1
    assert lib.q4_decode_pass_launches(L, 0, 1536) == -2


def test_valid_call_without_gpu_fails_loudly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.q4_gemv(A, A, A, A, 16, 64, 1, None, 0, None)
    assert st in (5, 6)            # no device: CUDA error (never a silent success)
    assert lib.q4_last_error() != b""


def test_binding_refuses_cpu_tensors(lib):
    import torch
    W = torch.zeros(4, 64)
    with pytest.raises(q4w.Q4Error):
        q4w.q4_quantize(W)
