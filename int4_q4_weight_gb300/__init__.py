"""Python binding of libq4w.so, the q4_0 weight-only int4 decode kernels for GB300.

Argument marshalling only: every function here checks tensor placement and
dtypes, passes raw device pointers and the current CUDA stream to the C ABI
of the same name (declared in ``include/q4w.h``) and raises on a non-zero
status.  PyTorch provides device memory and streams; all computation runs in
the library's CUDA kernels.  There is no fallback: if the library cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "load", "build", "Q4Error", "q4_quantize", "q4_gemv", "q4_gemv_weights_ro", "q4_gemv_stage", "q4_rmsnorm_f16",
    "q4_decode_pass", "q4_decode_pass_launches", "q2_gemv", "lmhead_softcap_argmax", "ple_gather_project", "q4_gemm_chunk",
    "q8_quantize", "ple_gather_project_q8", "q4_gemv_a8", "q4_gemm_chunk_a8", "q4_act_calibrate_a8",
    "q4_workspace_bytes", "q4_version", "Q4_IN_F16", "Q4_IN_RMS_F16", "Q4_IN_RMS_F32",
    "Q4_IN_RMS2_F32", "Q4_OP_GEMV", "Q4_OP_GEMM_CHUNK", "Q4_OP_PLE", "Q4_OP_LMHEAD",
    "Q4_OP_DECODE_PASS", "q4_layer", "q4_matrix",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libq4w.so")

Q4_IN_F16, Q4_IN_RMS_F16, Q4_IN_RMS_F32, Q4_IN_RMS2_F32 = 0, 1, 2, 3
Q4_OP_GEMV, Q4_OP_GEMM_CHUNK, Q4_OP_PLE, Q4_OP_LMHEAD, Q4_OP_DECODE_PASS = 0, 1, 2, 3, 4

_lib = None

vp = ctypes.c_void_p
ci = ctypes.c_int
cf = ctypes.c_float
csz = ctypes.c_size_t


class q4_matrix(ctypes.Structure):
    _fields_ = [("codes", vp), ("scales", vp)]


class q4_layer(ctypes.Structure):
    _fields_ = [("q_rows", ci), ("kv_rows", ci), ("mlp_rows", ci),
                ("q", q4_matrix), ("k", q4_matrix), ("v", q4_matrix), ("o", q4_matrix),
                ("gate", q4_matrix), ("up", q4_matrix), ("down", q4_matrix)]


_SIGS = {
    "q4_quantize": (ci, [vp, ci, ci, vp, vp, vp, vp]),
    "q4_gemv": (ci, [vp, vp, vp, vp, ci, ci, ci, vp, csz, vp]),
    "q4_gemv_weights_ro": (ci, [vp, vp, vp, vp, ci, ci, ci, vp, csz, vp]),
    "q4_gemm_chunk": (ci, [vp, vp, vp, vp, ci, ci, ci, vp, csz, vp]),
    "q4_gemv_a8": (ci, [vp, vp, vp, cf, vp, ci, ci, vp]),
    "q4_gemm_chunk_a8": (ci, [vp, vp, vp, cf, vp, ci, ci, ci, vp, csz, vp]),
    "q4_act_calibrate_a8": (ci, [vp, ctypes.c_longlong, vp, vp]),
    "ple_gather_project": (ci, [vp, ci, vp, vp, ci, ci, ci, cf, vp, vp, ci, vp, cf, vp, vp, vp, vp]),
    "q8_quantize": (ci, [vp, ci, ci, vp, vp, vp, vp]),
    "ple_gather_project_q8": (ci, [vp, ci, vp, vp, ci, ci, ci, cf, vp, vp, vp, ci, vp, cf, vp, vp, vp, vp]),
    "lmhead_softcap_argmax": (ci, [vp, vp, vp, ci, ci, ci, cf, vp, vp, vp, vp, vp, csz, vp]),
    "lmhead_softcap_argmax_noalloc": (ci, [vp, vp, vp, ci, ci, ci, cf, vp, vp, vp, vp, vp]),
    "q4_decode_pass": (ci, [ctypes.POINTER(q4_layer), ci, ci, vp, vp, cf, vp, csz, vp]),
    "q4_decode_pass_launches": (ci, [ctypes.POINTER(q4_layer), ci, ci]),
    "q2_gemv": (ci, [vp, vp, vp, vp, ci, ci, vp]),
    "q4_gemv_stage": (ci, [ctypes.POINTER(q4_matrix), ctypes.POINTER(ci), ci, ci, vp, ci, cf, ci,
                           ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
    "q4_rmsnorm_f16": (ci, [vp, ci, cf, vp, vp]),
    "q4_workspace_bytes": (csz, [ci, ci, ci, ci]),
    "q4_status_string": (ctypes.c_char_p, [ci]),
    "q4_last_error": (ctypes.c_char_p, []),
    "q4_version": (ci, []),
    "q4_device_status": (ci, [vp]),
    "q4_set_wait_limit": (ctypes.c_longlong, [ctypes.c_longlong]),
    "q4_set_trace": (ci, [vp, csz]),
}


class Q4Error(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile libq4w.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def load():
    """Load libq4w.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise Q4Error(f"{LIB_PATH} not found: build it first (int4_q4_weight_gb300.build())")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status: int, name: str):
    if status != 0:
        lib = load()
        raise Q4Error(f"{name}: {lib.q4_status_string(status).decode()}: "
                      f"{lib.q4_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _numel(t, n, name):
    """An array a kernel reads or writes holds exactly the elements its sizes imply
    (the kernels trust the sizes, so a short buffer would be overrun)."""
    if t is not None and t.numel() != n:
        raise Q4Error(f"{name} has {t.numel()} elements; the sizes imply {n}")


def _dev(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda:
        raise Q4Error(f"{name} must be a CUDA tensor")
    # every call launches on the current device's stream: a tensor on another
    # GPU would reach its kernels as a foreign pointer
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise Q4Error(f"{name} is on cuda:{t.device.index}, the current device is cuda:{cur}")
    if t.dtype != dtype:
        raise Q4Error(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise Q4Error(f"{name} must be contiguous")


def q4_device_status():
    """Synchronise the current stream; raise if a kernel's bounded wait ran out."""
    _check(load().q4_device_status(_stream()), "q4_device_status")


def q4_set_wait_limit(cycles: int) -> int:
    return int(load().q4_set_wait_limit(cycles))


def q4_set_trace(buf=None):
    """Diagnostic stamps of the persistent decode pass into ``buf`` (uint64 CUDA tensor), or off."""
    if buf is None:
        _check(load().q4_set_trace(None, 0), "q4_set_trace")
    else:
        _dev(buf, torch.int64, "trace")
        _check(load().q4_set_trace(_ptr(buf), buf.numel() * 8), "q4_set_trace")


def q4_version() -> int:
    return load().q4_version()


def q4_workspace_bytes(op: int, a: int, b: int, c: int) -> int:
    return int(load().q4_workspace_bytes(op, a, b, c))


def q4_quantize(W, codes=None, scales=None, err=None):
    """fp32 W [N, K] -> (codes uint8 [N, K/2], scales fp16 [N, K/32])."""
    lib = load()
    _dev(W, torch.float32, "W")
    N, K = W.shape
    if codes is None:
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // 32), dtype=torch.float16, device=W.device)
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(err, torch.int32, "err")
    _numel(codes, N * K // 2, "codes")
    _numel(scales, N * K // 32, "scales")
    _check(lib.q4_quantize(_ptr(W), N, K, _ptr(codes), _ptr(scales), _ptr(err), _stream()),
           "q4_quantize")
    return codes, scales


def q8_quantize(W, codes=None, scales=None, err=None):
    """fp32 W [N, K] -> (codes int8 [N, K], scales fp16 [N, K/32]), int8 per block of 32."""
    lib = load()
    _dev(W, torch.float32, "W")
    N, K = W.shape
    if codes is None:
        codes = torch.empty((N, K), dtype=torch.int8, device=W.device)
    if scales is None:
        scales = torch.empty((N, K // 32), dtype=torch.float16, device=W.device)
    _dev(codes, torch.int8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(err, torch.int32, "err")
    _numel(codes, N * K, "codes")
    _numel(scales, N * K // 32, "scales")
    _check(lib.q8_quantize(_ptr(W), N, K, _ptr(codes), _ptr(scales), _ptr(err), _stream()),
           "q8_quantize")
    return codes, scales


def q4_gemv(codes, scales, x, y=None):
    """y [b, N] f32 = dequant(codes, scales) @ x[b]  (x fp16 [b, K] or [K])."""
    return _gemv("q4_gemv", codes, scales, x, y)


def q4_gemv_weights_ro(codes, scales, x, y=None):
    """q4_gemv, promising that no earlier kernel still running on the stream
    writes codes or scales: the weight tiles stream before that kernel ends."""
    return _gemv("q4_gemv_weights_ro", codes, scales, x, y)


def _gemv(name, codes, scales, x, y):
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(x, torch.float16, "x")
    N, K = codes.shape[0], codes.shape[1] * 2
    batch = 1 if x.dim() == 1 else x.shape[0]
    if y is None:
        y = torch.empty((batch, N) if x.dim() == 2 else (N,), dtype=torch.float32, device=x.device)
    _dev(y, torch.float32, "y")
    _numel(scales, N * K // 32, "scales")
    _numel(x, batch * K, "x")
    _numel(y, batch * N, "y")
    _check(getattr(lib, name)(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), N, K, batch, None, 0, _stream()), name)
    return y


def _matrix_shape(codes, scales, rows, cols, name):
    """codes uint8 [rows, cols/2] and rows * cols/32 scales, as the sizes imply."""
    if codes.dim() != 2 or tuple(codes.shape) != (rows, cols // 2):
        raise Q4Error(f"{name}.codes has shape {tuple(codes.shape)}; the sizes imply ({rows}, {cols // 2})")
    _numel(scales, rows * cols // 32, f"{name}.scales")


def q4_gemv_stage(mats, inp, in_mode, eps=1e-6, pair=False, out32=None, out16=None):
    """One fused decode-pass stage; ``mats`` is a list of (codes, scales)."""
    lib = load()
    n = len(mats)
    if not 1 <= n <= 3 or (pair and n != 2):
        raise Q4Error(f"q4_gemv_stage takes 1 to 3 matrices (exactly 2 with pair), got {n}")
    K = mats[0][0].shape[1] * 2
    for i, (c, s) in enumerate(mats):
        _matrix_shape(c, s, c.shape[0], K, f"mats[{i}]")
    if pair and mats[0][0].shape[0] != mats[1][0].shape[0]:
        raise Q4Error("pair: gate and up must have the same rows")
    _numel(inp, K, "in")
    arr = (q4_matrix * n)()
    rows = (ci * n)()
    o32 = (vp * n)()
    o16 = (vp * n)()
    out32 = list(out32) if out32 is not None else [None] * n
    out16 = list(out16) if out16 is not None else [None] * n
    for i, (c, s) in enumerate(mats):
        _dev(c, torch.uint8, f"mats[{i}].codes")
        _dev(s, torch.float16, f"mats[{i}].scales")
        arr[i] = q4_matrix(c.data_ptr(), s.data_ptr())
        rows[i] = c.shape[0]
        _dev(out32[i], torch.float32, f"out32[{i}]")
        _dev(out16[i], torch.float16, f"out16[{i}]")
        _numel(out32[i], c.shape[0], f"out32[{i}]")
        _numel(out16[i], c.shape[0], f"out16[{i}]")
        o32[i] = out32[i].data_ptr() if out32[i] is not None else None
        o16[i] = out16[i].data_ptr() if out16[i] is not None else None
    _dev(inp, torch.float16 if in_mode in (Q4_IN_F16, Q4_IN_RMS_F16) else torch.float32, "in")
    _check(lib.q4_gemv_stage(arr, rows, n, K, _ptr(inp), in_mode, eps, int(pair), o32, o16,
                             _stream()), "q4_gemv_stage")
    return out32, out16


def q4_rmsnorm_f16(inp, eps=1e-6, out=None):
    lib = load()
    _dev(inp, torch.float32, "in")
    if out is None:
        out = torch.empty(inp.shape, dtype=torch.float16, device=inp.device)
    _dev(out, torch.float16, "out")
    _numel(out, inp.numel(), "out")
    _check(lib.q4_rmsnorm_f16(_ptr(inp), inp.numel(), eps, _ptr(out), _stream()), "q4_rmsnorm_f16")
    return out


def _check_layers(layers, H):
    """Every matrix of every layer has the shape the pass reads for hidden H:
    q [Q, H], k and v [KV, H] (together or both absent), o [H, Q],
    gate and up [I, H], down [H, I]."""
    for i, lw in enumerate(layers):
        if ("k" in lw) != ("v" in lw):
            raise Q4Error(f"layers[{i}]: k and v must be given together")
        Q, I = lw["q"][0].shape[0], lw["g"][0].shape[0]
        KV = lw["k"][0].shape[0] if "k" in lw else 0
        want = {"q": (Q, H), "k": (KV, H), "v": (KV, H), "o": (H, Q), "g": (I, H), "u": (I, H), "d": (H, I)}
        for key, (r, c) in want.items():
            if key in lw:
                _matrix_shape(*lw[key], r, c, f"layers[{i}].{key}")
            elif key not in ("k", "v"):
                raise Q4Error(f"layers[{i}] has no '{key}' matrix")


def make_layers(layers, H=None):
    """Host descriptor array from a list of dicts name -> (codes, scales); every
    shape is checked against hidden size H (taken from layer 0's q when None)."""
    if H is None:
        H = layers[0]["q"][0].shape[1] * 2
    _check_layers(layers, H)
    arr = (q4_layer * len(layers))()
    for i, lw in enumerate(layers):
        d = q4_layer()
        d.q_rows = lw["q"][0].shape[0]
        d.kv_rows = lw["k"][0].shape[0] if "k" in lw else 0
        d.mlp_rows = lw["g"][0].shape[0]
        for fld, key in (("q", "q"), ("k", "k"), ("v", "v"), ("o", "o"), ("gate", "g"),
                         ("up", "u"), ("down", "d")):
            if key in lw:
                c, s = lw[key]
                _dev(c, torch.uint8, f"layers[{i}].{key}.codes")
                _dev(s, torch.float16, f"layers[{i}].{key}.scales")
                setattr(d, fld, q4_matrix(c.data_ptr(), s.data_ptr()))
        arr[i] = d
    return arr


def decode_pass_ws_bytes(layers, H):
    qkv = max(lw["q"][0].shape[0] + 2 * (lw["k"][0].shape[0] if "k" in lw else 0) for lw in layers)
    mlp = max(lw["g"][0].shape[0] for lw in layers)
    return q4_workspace_bytes(Q4_OP_DECODE_PASS, H, qkv, mlp)


def q4_decode_pass(layers, h0, h_out, ws, eps=1e-6, descs=None):
    """Run the weight pass over ``layers`` (list of dicts) from fp16 h0 [H] into
    fp16 h_out [H].  ``descs``: the descriptor array make_layers(layers, H) built
    for the same layers (the layers' shapes are checked either way)."""
    lib = load()
    _dev(h0, torch.float16, "h0")
    _dev(h_out, torch.float16, "h_out")
    _dev(ws, torch.uint8, "ws")
    H = h0.numel()
    _numel(h_out, H, "h_out")
    if descs is None:
        descs = make_layers(layers, H)
    else:
        if len(descs) != len(layers):
            raise Q4Error(f"descs holds {len(descs)} layers, layers {len(layers)}")
        _check_layers(layers, H)
    _check(lib.q4_decode_pass(descs, len(descs), h0.numel(), _ptr(h0), _ptr(h_out), eps, _ptr(ws),
                              ws.numel(), _stream()), "q4_decode_pass")
    return h_out


def lmhead_ws(V, K, b, device):
    return torch.empty(q4_workspace_bytes(Q4_OP_LMHEAD, V, K, b), dtype=torch.uint8, device=device)


def lmhead_softcap_argmax(codes, scales, h, cap=30.0, ws=None, idx=None, top1=None, top2=None,
                          logits=None):
    """Returns (idx int32 [b], top1 f32 [b], top2 f32 [b], logits or None)."""
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(h, torch.float16, "h")
    V, K = codes.shape[0], codes.shape[1] * 2
    b = 1 if h.dim() == 1 else h.shape[0]
    dev = h.device
    if ws is None:
        ws = lmhead_ws(V, K, b, dev)
    idx = torch.empty(b, dtype=torch.int32, device=dev) if idx is None else idx
    top1 = torch.empty(b, dtype=torch.float32, device=dev) if top1 is None else top1
    top2 = torch.empty(b, dtype=torch.float32, device=dev) if top2 is None else top2
    for t, dt, nm in ((idx, torch.int32, "idx"), (top1, torch.float32, "top1"),
                      (top2, torch.float32, "top2"), (logits, torch.float32, "logits"),
                      (ws, torch.uint8, "ws")):
        _dev(t, dt, nm)
    _numel(scales, V * K // 32, "scales")
    _numel(h, b * K, "h")
    for t, nm in ((idx, "idx"), (top1, "top1"), (top2, "top2")):
        _numel(t, b, nm)
    _numel(logits, b * V, "logits")
    _check(lib.lmhead_softcap_argmax(_ptr(codes), _ptr(scales), _ptr(h), b, V, K, cap, _ptr(idx),
                                     _ptr(top1), _ptr(top2), _ptr(logits), _ptr(ws), ws.numel(),
                                     _stream()), "lmhead_softcap_argmax")
    return idx, top1, top2, logits


def _ple_sizes(S, V, L, ld, D, table, row_scale, hidden, norm_w, out, gathered):
    _numel(table, V * L * ld, "table (V rows of L*ld bytes)")
    _numel(row_scale, V, "row_scale")
    _numel(hidden, S * D, "hidden")
    _numel(norm_w, ld, "norm_w")
    _numel(out, S * L * ld, "out")
    _numel(gathered, S * L * ld, "gathered")


def ple_gather_project(ids, table, row_scale, proj, hidden, norm_w, L=35, ld=256,
                       embed_scale=16.0, eps=1e-6, out=None, gathered=None, err=None):
    """Returns (out f32 [S, L*ld], gathered int8 [S, L*ld] or None)."""
    lib = load()
    _dev(ids, torch.int32, "ids")
    _dev(table, torch.int8, "table")
    _dev(row_scale, torch.float32, "row_scale")
    _dev(proj, torch.float32, "proj")
    _dev(hidden, torch.float16, "hidden")
    _dev(norm_w, torch.float32, "norm_w")
    S = ids.numel()
    V = table.shape[0]
    D = proj.shape[1]
    if out is None:
        out = torch.empty((S, L * ld), dtype=torch.float32, device=ids.device)
    _dev(out, torch.float32, "out")
    _dev(gathered, torch.int8, "gathered")
    _dev(err, torch.int32, "err")
    _ple_sizes(S, V, L, ld, D, table, row_scale, hidden, norm_w, out, gathered)
    _numel(proj, L * ld * D, "proj")
    _check(lib.ple_gather_project(_ptr(ids), S, _ptr(table), _ptr(row_scale), V, L, ld, embed_scale,
                                  _ptr(proj), _ptr(hidden), D, _ptr(norm_w), eps, _ptr(out),
                                  _ptr(gathered), _ptr(err), _stream()), "ple_gather_project")
    return out, gathered


def ple_gather_project_q8(ids, table, row_scale, proj_codes, proj_scales, hidden, norm_w, L=35, ld=256,
                          embed_scale=16.0, eps=1e-6, out=None, gathered=None, err=None):
    """ple_gather_project with the projection as int8 codes [L*ld, D] and fp16
    scales [L*ld, D/32]; returns (out f32 [S, L*ld], gathered int8 or None)."""
    lib = load()
    _dev(ids, torch.int32, "ids")
    _dev(table, torch.int8, "table")
    _dev(row_scale, torch.float32, "row_scale")
    _dev(proj_codes, torch.int8, "proj_codes")
    _dev(proj_scales, torch.float16, "proj_scales")
    _dev(hidden, torch.float16, "hidden")
    _dev(norm_w, torch.float32, "norm_w")
    S = ids.numel()
    V = table.shape[0]
    D = proj_codes.shape[1]
    if out is None:
        out = torch.empty((S, L * ld), dtype=torch.float32, device=ids.device)
    _dev(out, torch.float32, "out")
    _dev(gathered, torch.int8, "gathered")
    _dev(err, torch.int32, "err")
    _ple_sizes(S, V, L, ld, D, table, row_scale, hidden, norm_w, out, gathered)
    _numel(proj_codes, L * ld * D, "proj_codes")
    _numel(proj_scales, L * ld * D // 32, "proj_scales")
    _check(lib.ple_gather_project_q8(_ptr(ids), S, _ptr(table), _ptr(row_scale), V, L, ld, embed_scale,
                                     _ptr(proj_codes), _ptr(proj_scales), _ptr(hidden), D, _ptr(norm_w), eps,
                                     _ptr(out), _ptr(gathered), _ptr(err), _stream()), "ple_gather_project_q8")
    return out, gathered


def q4_gemm_chunk(codes, scales, X, Y=None):
    """Y [64, N] f32 = bf16 tiles of dequant(codes, scales) times bf16(X [64, K])."""
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(X, torch.float16, "X")
    N, K = codes.shape[0], codes.shape[1] * 2
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _dev(Y, torch.float32, "Y")
    _numel(scales, N * K // 32, "scales")
    _numel(X, M * K, "X")
    _numel(Y, M * N, "Y")
    nws = lib.q4_workspace_bytes(Q4_OP_GEMM_CHUNK, N, K, M)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=X.device)
    _check(lib.q4_gemm_chunk(_ptr(codes), _ptr(scales), _ptr(X), _ptr(Y), M, N, K, _ptr(ws), nws,
                             _stream()), "q4_gemm_chunk")
    return Y


def q4_gemv_a8(codes, scales, x, act_scale, y=None):
    """w4a8 GEMV: y [N] f32 = act_scale * dequant(codes, scales) @ q, q the int8
    codes clamp(rint(x / act_scale), -128, 127) of x (fp16 [K])."""
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(x, torch.float16, "x")
    N, K = codes.shape[0], codes.shape[1] * 2
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    _dev(y, torch.float32, "y")
    _numel(scales, N * K // 32, "scales")
    _numel(x, K, "x")
    _numel(y, N, "y")
    _check(lib.q4_gemv_a8(_ptr(codes), _ptr(scales), _ptr(x), float(act_scale), _ptr(y), N, K, _stream()),
           "q4_gemv_a8")
    return y


def q4_gemm_chunk_a8(codes, scales, X, act_scale, Y=None):
    """w4a8 S=64 chunk: Y [64, N] f32 = act_scale * (bf16 tiles of dequant(codes, scales)) @ Q.T,
    Q the int8 codes of X [64, K] under act_scale."""
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float16, "scales")
    _dev(X, torch.float16, "X")
    N, K = codes.shape[0], codes.shape[1] * 2
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    _dev(Y, torch.float32, "Y")
    _numel(scales, N * K // 32, "scales")
    _numel(X, M * K, "X")
    _numel(Y, M * N, "Y")
    nws = lib.q4_workspace_bytes(Q4_OP_GEMM_CHUNK, N, K, M)
    ws = torch.empty(max(nws, 1), dtype=torch.uint8, device=X.device)
    _check(lib.q4_gemm_chunk_a8(_ptr(codes), _ptr(scales), _ptr(X), float(act_scale), _ptr(Y), M, N, K,
                                _ptr(ws), nws, _stream()), "q4_gemm_chunk_a8")
    return Y


def q4_act_calibrate_a8(samples, out=None):
    """Min-max calibration of a w4a8 activation scale: a one-element f32 CUDA
    tensor holding max |x| / 127 over every value of ``samples`` (fp16, any
    shape, e.g. [128, K]), or 1 when all are zero."""
    lib = load()
    _dev(samples, torch.float16, "samples")
    if out is None:
        out = torch.empty(1, dtype=torch.float32, device=samples.device)
    _dev(out, torch.float32, "out")
    _numel(out, 1, "out")
    if samples.numel() < 1:
        raise Q4Error("samples must hold at least one value")
    _check(lib.q4_act_calibrate_a8(_ptr(samples), samples.numel(), _ptr(out), _stream()),
           "q4_act_calibrate_a8")
    return out


def q2_gemv(codes, scales, x, y=None):
    """INT2 per-row symmetric GEMV: y [N] f32 = scale[n] * sum_k (code - 2) x[k] (x fp16 [K])."""
    lib = load()
    _dev(codes, torch.uint8, "codes")
    _dev(scales, torch.float32, "scales")
    _dev(x, torch.float16, "x")
    N, K = codes.shape[0], codes.shape[1] * 4
    if y is None:
        y = torch.empty(N, dtype=torch.float32, device=x.device)
    _dev(y, torch.float32, "y")
    _numel(scales, N, "scales")
    _numel(x, K, "x")
    _numel(y, N, "y")
    _check(lib.q2_gemv(_ptr(codes), _ptr(scales), _ptr(x), _ptr(y), N, K, _stream()), "q2_gemv")
    return y


def q4_decode_pass_launches(descs, H):
    """Kernels one q4_decode_pass call over ``descs`` (make_layers output) launches."""
    n = load().q4_decode_pass_launches(descs, len(descs), H)
    if n < 0:
        _check(-n, "q4_decode_pass_launches")
    return n


class Q4DecodePlan:
    """A decode weight pass bound to fixed device buffers and captured once into
    a CUDA graph, so that a step is one graph launch.

    ``layers``: list of dicts name -> (codes, scales) as for q4_decode_pass.
    ``step_device()`` replays the graph on the current stream (h_in -> h_out,
    both device buffers).  ``step_host(h_pinned, out_pinned)`` copies one fp16
    hidden vector host->device, replays, and copies the result back.
    """

    def __init__(self, layers, H, eps=1e-6, device="cuda"):
        self.layers = layers
        self.H = H
        self.eps = eps
        self.descs = make_layers(layers, H)
        self.ws = torch.empty(decode_pass_ws_bytes(layers, H), dtype=torch.uint8, device=device)
        self.h_in = torch.zeros(H, dtype=torch.float16, device=device)
        self.h_out = torch.zeros(H, dtype=torch.float16, device=device)
        self.stream = torch.cuda.Stream(device=device)
        self.graph = None

    def run_eager(self):
        q4_decode_pass(self.layers, self.h_in, self.h_out, self.ws, self.eps, descs=self.descs)

    def capture(self):
        with torch.cuda.stream(self.stream):
            self.run_eager()                       # warm-up outside the capture
        torch.cuda.current_stream().wait_stream(self.stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            self.run_eager()
        torch.cuda.synchronize()
        return self

    def step_device(self):
        self.graph.replay()

    def step_host(self, h_pinned, out_pinned):
        self.h_in.copy_(h_pinned, non_blocking=True)
        self.graph.replay()
        out_pinned.copy_(self.h_out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return out_pinned

    @property
    def launches_per_step(self):
        """Kernels one replay launches (the library's own count)."""
        return q4_decode_pass_launches(self.descs, self.H)
