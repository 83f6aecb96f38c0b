"""Thin ctypes binding of ``libw8lin.so`` (the C ABI in ``include/w8lin.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and the current stream.  When the
library is missing the calls raise instead of falling back to anything else.
"""

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libw8lin.so")

W8_OK = 0
STATUS_NAMES = {
    0: "W8_OK", 1: "W8_ERR_NULL", 2: "W8_ERR_SHAPE", 3: "W8_ERR_ALIGN", 4: "W8_ERR_STRIDE",
    5: "W8_ERR_DTYPE", 6: "W8_ERR_ARCH", 7: "W8_ERR_POLICY", 8: "W8_ERR_TIMEOUT",
    9: "W8_ERR_CUDA", 10: "W8_ERR_SCALE", 11: "W8_ERR_PARAM",
}
DTYPE_BF16, DTYPE_E4M3, DTYPE_F16 = 0, 1, 2
MODE_A8, MODE_A16 = 0, 1

# Every symbol the header declares, with its ctypes signature.
_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


class StepPolicy(ctypes.Structure):
    """Mirror of ``w8_step_policy``."""
    _fields_ = [("schema_version", _i32), ("enabled", _i32),
                ("first_steps", _i32), ("last_steps", _i32)]


class SwigluParams(ctypes.Structure):
    """Mirror of ``w8_swiglu_params``."""
    _fields_ = [("has_limit", _i32), ("limit", ctypes.c_float), ("alpha", ctypes.c_float),
                ("beta", ctypes.c_float)]


SIGNATURES = {
    "w8_abi_version": (ctypes.c_int, []),
    "w8_last_error": (ctypes.c_char_p, []),
    "w8_device_check": (ctypes.c_int, []),
    "w8_poll_device_error": (ctypes.c_int, [_c_void_p]),
    "w8_selftest_timeout": (ctypes.c_int, [_c_void_p]),
    "fp8_quant_static": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "fp8_linear_w8a8": (ctypes.c_int, [_c_void_p, _i32, _i64, _i64, _c_void_p, _i64, _c_void_p,
                                       _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "fp8_linear_w8a16": (ctypes.c_int, [_c_void_p, _i32, _i64, _i64, _c_void_p, _i64, _c_void_p,
                                        _c_void_p, _c_void_p, _c_void_p]),
    "qkv_shared_quant_gemm": (ctypes.c_int, [_i32, _c_void_p, _i64, _i64, _c_void_p, _i32,
                                             ctypes.POINTER(_c_void_p), ctypes.POINTER(_i64),
                                             ctypes.POINTER(_c_void_p), ctypes.POINTER(_c_void_p),
                                             _c_void_p, _c_void_p]),
    "fp8_dequant_weight": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "fp8_e4m3_from_f32": (ctypes.c_int, [_c_void_p, _i64, _c_void_p, _c_void_p]),
    "bf16_gate_up_swiglu": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i64, _c_void_p,
                                           _c_void_p]),
    "bf16_linear_group": (ctypes.c_int, [_c_void_p, _i64, _i64, _i32, ctypes.POINTER(_c_void_p),
                                         ctypes.POINTER(_i64), ctypes.POINTER(_c_void_p), _c_void_p]),
    "fp8_linear_w8a8_group": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _i32,
                                             ctypes.POINTER(_c_void_p), ctypes.POINTER(_i64),
                                             ctypes.POINTER(_c_void_p), ctypes.POINTER(_c_void_p),
                                             _c_void_p]),
    "gate_up_swiglu_fp8": (ctypes.c_int, [_c_void_p, _i32, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                          _i64, _c_void_p, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                          _c_void_p]),
    "fp8_linear_w8a8_noalloc": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _i64, _c_void_p,
                                               _c_void_p, _c_void_p, _c_void_p]),
    "swiglu_2in_fp8": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p,
                                      _c_void_p]),
    "swiglu_2in_bf16": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _i64, _c_void_p, _c_void_p]),
    "swiglu_2in_ex_fp8": (ctypes.c_int, [_c_void_p, _c_void_p, _i32, _i64, _i64, ctypes.POINTER(SwigluParams),
                                         _c_void_p, _c_void_p, _c_void_p]),
    "swiglu_2in_ex_16": (ctypes.c_int, [_c_void_p, _c_void_p, _i32, _i64, _i64, ctypes.POINTER(SwigluParams),
                                        _c_void_p, _c_void_p]),
    "gate_up_swiglu_ex_fp8": (ctypes.c_int, [_c_void_p, _i32, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                             _i64, _c_void_p, _c_void_p, ctypes.POINTER(SwigluParams),
                                             _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "bf16_gate_up_swiglu_ex": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i64,
                                              ctypes.POINTER(SwigluParams), _c_void_p, _c_void_p]),
    "ln_modulate_quant": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i64, ctypes.c_float,
                                         _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "step_policy_dispatch": (ctypes.c_int, [_c_void_p, _i32, _i32, ctypes.POINTER(_i32)]),
    "w8_check_group_scales": (ctypes.c_int, [ctypes.POINTER(_c_void_p), _i32]),
    "w8_step_policy_parse": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(StepPolicy),
                                            ctypes.POINTER(_i32)]),
}


class W8Error(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def _check(status):
    if status != W8_OK:
        raise W8Error(status, lib().w8_last_error().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dense(t, name):
    if not t.is_contiguous():
        raise W8Error(4, f"{name}: non-contiguous tensors are rejected")
    if not t.is_cuda:
        raise W8Error(1, f"{name}: must be a CUDA tensor")
    return t


def _as_u8(t, name):
    _dense(t, name)
    if t.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", None)):
        return t.view(torch.uint8)
    raise W8Error(5, f"{name}: expected E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")


def _as_bf16(t, name):
    _dense(t, name)
    if t.dtype != torch.bfloat16:
        raise W8Error(5, f"{name}: expected bfloat16, got {t.dtype}")
    return t


def _flat2(t):
    return t.reshape(-1, t.shape[-1])


def _scalar(t, name):
    _dense(t, name)
    if t.dtype != torch.float32 or t.numel() != 1:
        raise W8Error(5, f"{name}: expected a one-element float32 device tensor")
    return t


# ---------------------------------------------------------------- entry points

def abi_version():
    return lib().w8_abi_version()


def device_check():
    _check(lib().w8_device_check())


def poll_device_error(stream=None):
    _check(lib().w8_poll_device_error(_stream(stream)))


def selftest_timeout(stream=None):
    """Enqueue the bounded-wait self-test (its timeout shows up in the next
    poll_device_error)."""
    _check(lib().w8_selftest_timeout(_stream(stream)))


def fp8_quant_static(x, s_in, out=None, stream=None):
    """E4M3 codes (uint8) of ``x / s_in``; same shape as ``x``.  Row pitches
    are passed as they are: a tensor whose rows are not dense is refused by
    the library (W8_ERR_STRIDE)."""
    if x.dtype != torch.bfloat16:
        raise W8Error(5, f"x: expected bfloat16, got {x.dtype}")
    if not x.is_cuda:
        raise W8Error(1, "x: must be a CUDA tensor")
    if x.dim() < 2:
        raise W8Error(2, "x: expected at least 2 dimensions")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    if out.dtype not in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) or out.shape != x.shape:
        raise W8Error(5, "out: expected E4M3 codes of x's shape")
    K = x.shape[-1]
    M = x.numel() // K if K else 0
    ldx = _row_pitch(x)
    ldq = _row_pitch(out)
    _check(lib().fp8_quant_static(_ptr(x), M, K, ldx, _ptr(_scalar(s_in, "s_in")), _ptr(out), ldq,
                                  _stream(stream)))
    return out


def _row_pitch(t):
    """Elements between consecutive row starts when the last dimension is
    contiguous and every leading dimension is packed row after row; -1 for
    any other layout (refused by the library as non-dense)."""
    if t.dim() < 2 or t.stride(-1) != 1:
        return -1
    pitch = t.stride(-2)
    expect = pitch * t.shape[-2]
    for d in range(t.dim() - 3, -1, -1):
        if t.shape[d] != 1 and t.stride(d) != expect:
            return -1
        expect *= t.shape[d]
    return pitch


def _ln_call(x, shift, scale, eps, s_in, q, h, stream):
    x = _as_bf16(x, "x")
    x2 = _flat2(x)
    M, K = x2.shape
    sh = _flat2(_as_bf16(shift, "shift"))
    sc = _flat2(_as_bf16(scale, "scale"))
    S = sh.shape[0]
    if sc.shape != sh.shape or sh.shape[1] != K or S < 1:
        raise W8Error(2, f"shift/scale: expected [S, {K}], got {tuple(sh.shape)} and {tuple(sc.shape)}")
    if M % S:
        raise W8Error(2, f"{M} rows do not split into {S} samples")
    rps = max(M // S, 1)
    _check(lib().ln_modulate_quant(_ptr(x2), M, K, _ptr(sh), _ptr(sc), rps, float(eps),
                                   _ptr(s_in), _ptr(q), _ptr(h), _stream(stream)))


def ln_modulate_quant(x, shift, scale, s_in, eps=1e-6, out=None, h_out=None, stream=None):
    """E4M3 codes of the modulated LayerNorm of ``x`` (rows split evenly into
    ``shift.shape[0]`` samples), quantized with ``s_in``; also writes the
    bf16 h into ``h_out`` when given.  Returns the codes."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    q = _as_u8(out, "out")
    h = _as_bf16(h_out, "h_out") if h_out is not None else None
    _ln_call(x, shift, scale, eps, _scalar(s_in, "s_in"), q, h, stream)
    return out


def ln_modulate_bf16(x, shift, scale, eps=1e-6, out=None, stream=None):
    """The bf16 modulated LayerNorm alone (the unfused producer)."""
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _ln_call(x, shift, scale, eps, None, None, _as_bf16(out, "out"), stream)
    return out


def fp8_linear_w8a8(x, w, s_in, s_w, out=None, ws=None, stream=None):
    """W8A8 linear.  ``x`` bf16 (quantized into ``ws``) or E4M3 codes."""
    if x.dtype == torch.bfloat16:
        xd, dt = _as_bf16(x, "x"), DTYPE_BF16
    else:
        xd, dt = _as_u8(x, "x"), DTYPE_E4M3
    x2 = _flat2(xd)
    M, K = x2.shape
    wq = _as_u8(w, "w")
    N = wq.shape[0]
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    _as_bf16(out, "out")
    if dt == DTYPE_BF16 and ws is None:
        ws = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    _check(lib().fp8_linear_w8a8(_ptr(x2), dt, M, K, _ptr(wq), N, _ptr(_scalar(s_in, "s_in")),
                                 _ptr(_scalar(s_w, "s_w")), _ptr(out),
                                 _ptr(_as_u8(ws, "ws") if ws is not None else None), _stream(stream)))
    return out


def fp8_linear_w8a16(x, w, s_w, out=None, ws=None, stream=None):
    """W8A16 linear.  ``x`` must be bf16.  With ``ws`` (bf16, at least N*K
    values) the weight is dequantized into it and a bf16 GEMM runs on it;
    without, the dequantization happens inside the GEMM."""
    dt = DTYPE_BF16 if x.dtype == torch.bfloat16 else DTYPE_E4M3
    xd = _dense(x, "x")
    x2 = _flat2(xd)
    M, K = x2.shape
    wq = _as_u8(w, "w")
    N = wq.shape[0]
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    _as_bf16(out, "out")
    if ws is not None:
        _as_bf16(ws, "ws")
        if ws.numel() < N * K:
            raise W8Error(2, f"ws: {ws.numel()} bf16 values, the weight needs {N * K}")
    _check(lib().fp8_linear_w8a16(_ptr(x2), dt, M, K, _ptr(wq), N, _ptr(_scalar(s_w, "s_w")),
                                  _ptr(out), _ptr(ws), _stream(stream)))
    return out


def qkv_shared_quant_gemm(mode, x, s_in, weights, weight_scales, outs=None, ws=None, stream=None):
    """A projection group sharing one activation (mode MODE_A8 or MODE_A16)."""
    x = _as_bf16(x, "x")
    x2 = _flat2(x)
    M, K = x2.shape
    G = len(weights)
    ws_q = [_as_u8(w, f"w[{i}]") for i, w in enumerate(weights)]
    if outs is None:
        outs = [torch.empty(*x.shape[:-1], w.shape[0], dtype=torch.bfloat16, device=x.device) for w in ws_q]
    for i, o in enumerate(outs):
        _as_bf16(o, f"y[{i}]")
    if mode == MODE_A8 and ws is None:
        ws = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if mode == MODE_A8 or ws is None:
        ws_p = _ptr(_as_u8(ws, "ws") if ws is not None else None)
    else:   # A16 with a workspace: room for the group's dequantized bf16 weights
        _as_bf16(ws, "ws")
        need = sum(int(w.shape[0]) * K for w in ws_q)
        if ws.numel() < need:
            raise W8Error(2, f"ws: {ws.numel()} bf16 values, the group needs {need}")
        ws_p = _ptr(ws)
    arr_w = (ctypes.c_void_p * G)(*[w.data_ptr() for w in ws_q])
    arr_n = (ctypes.c_int64 * G)(*[w.shape[0] for w in ws_q])
    arr_s = (ctypes.c_void_p * G)(*[_scalar(s, f"s_w[{i}]").data_ptr() for i, s in enumerate(weight_scales)])
    arr_y = (ctypes.c_void_p * G)(*[o.data_ptr() for o in outs])
    s_in_p = _ptr(_scalar(s_in, "s_in")) if s_in is not None else ctypes.c_void_p(0)
    _check(lib().qkv_shared_quant_gemm(mode, _ptr(x2), M, K, s_in_p, G, arr_w, arr_n, arr_s, arr_y,
                                       ws_p, _stream(stream)))
    return outs


def fp8_e4m3_from_f32(x, out=None, stream=None):
    """E4M3 codes (uint8, same shape) of the float32 values of ``x``:
    round to nearest even, saturating at +-448."""
    if x.dtype != torch.float32:
        raise W8Error(5, f"x: expected float32, got {x.dtype}")
    _dense(x, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    q = _as_u8(out, "out")
    if q.shape != x.shape:
        raise W8Error(2, f"out: shape {tuple(q.shape)} differs from x {tuple(x.shape)}")
    _check(lib().fp8_e4m3_from_f32(_ptr(x), x.numel(), _ptr(q), _stream(stream)))
    return out


def fp8_dequant_weight(w, s_w, out=None, stream=None):
    """bf16 [N, K] = bf16(fl32(dec(w) * s_w)): the W8A16 step's transient weight."""
    wq = _as_u8(w, "w")
    N, K = wq.shape
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=wq.device)
    _check(lib().fp8_dequant_weight(_ptr(wq), N, K, _ptr(_scalar(s_w, "s_w")), _ptr(_as_bf16(out, "out")),
                                    _stream(stream)))
    return out


def bf16_linear_group(x, wds, outs=None, stream=None):
    """y_g = bf16(x . Wd_g^T) for dequantized bf16 weights Wd_g (one launch)."""
    x = _as_bf16(x, "x")
    x2 = _flat2(x)
    M, K = x2.shape
    G = len(wds)
    wq = [_as_bf16(w, f"wd[{i}]") for i, w in enumerate(wds)]
    if outs is None:
        outs = [torch.empty(*x.shape[:-1], w.shape[0], dtype=torch.bfloat16, device=x.device) for w in wq]
    for i, o in enumerate(outs):
        _as_bf16(o, f"y[{i}]")
    arr_w = (ctypes.c_void_p * G)(*[w.data_ptr() for w in wq])
    arr_n = (ctypes.c_int64 * G)(*[w.shape[0] for w in wq])
    arr_y = (ctypes.c_void_p * G)(*[o.data_ptr() for o in outs])
    _check(lib().bf16_linear_group(_ptr(x2), M, K, G, arr_w, arr_n, arr_y, _stream(stream)))
    return outs


def bf16_gate_up_swiglu(x, wd_gate, wd_up, out=None, stream=None, limit=None, alpha=None, beta=None):
    """bf16 SwiGLU of the gate/up pair on dequantized bf16 weights, one launch.
    With any of ``limit``, ``alpha``, ``beta`` given, the SwiGLU takes those
    options (``bf16_gate_up_swiglu_ex``)."""
    x = _as_bf16(x, "x")
    x2 = _flat2(x)
    M, K = x2.shape
    wg, wu = _as_bf16(wd_gate, "wd_gate"), _as_bf16(wd_up, "wd_up")
    if wg.shape != wu.shape:
        raise W8Error(2, "gate and up weights differ in shape")
    I = wg.shape[0]
    if out is None:
        out = torch.empty(*x.shape[:-1], I, dtype=torch.bfloat16, device=x.device)
    if limit is None and alpha is None and beta is None:
        _check(lib().bf16_gate_up_swiglu(_ptr(x2), M, K, _ptr(wg), _ptr(wu), I, _ptr(_as_bf16(out, "out")),
                                         _stream(stream)))
    else:
        prm = _swiglu_params(limit, 1.0 if alpha is None else alpha, 0.0 if beta is None else beta)
        _check(lib().bf16_gate_up_swiglu_ex(_ptr(x2), M, K, _ptr(wg), _ptr(wu), I, ctypes.byref(prm),
                                            _ptr(_as_bf16(out, "out")), _stream(stream)))
    return out


def w8a16_workspace(weights):
    """bf16 scratch for qkv_shared_quant_gemm(MODE_A16, ..., ws=...): room for
    the group's dequantized weights (caller-side allocation)."""
    n = sum(int(w.shape[0]) * int(w.shape[1]) for w in weights)
    return torch.empty((n,), dtype=torch.bfloat16, device=weights[0].device)


def fp8_linear_w8a8_group(qx, s_in, weights, weight_scales, outs=None, stream=None):
    """G W8A8 projections over an activation already quantized to E4M3."""
    q = _as_u8(qx, "qx")
    q2 = _flat2(q)
    M, K = q2.shape
    G = len(weights)
    ws_q = [_as_u8(w, f"w[{i}]") for i, w in enumerate(weights)]
    if outs is None:
        outs = [torch.empty(*qx.shape[:-1], w.shape[0], dtype=torch.bfloat16, device=qx.device) for w in ws_q]
    for i, o in enumerate(outs):
        _as_bf16(o, f"y[{i}]")
    arr_w = (ctypes.c_void_p * G)(*[w.data_ptr() for w in ws_q])
    arr_n = (ctypes.c_int64 * G)(*[w.shape[0] for w in ws_q])
    arr_s = (ctypes.c_void_p * G)(*[_scalar(s, f"s_w[{i}]").data_ptr() for i, s in enumerate(weight_scales)])
    arr_y = (ctypes.c_void_p * G)(*[o.data_ptr() for o in outs])
    _check(lib().fp8_linear_w8a8_group(_ptr(q2), M, K, _ptr(_scalar(s_in, "s_in")), G, arr_w, arr_n,
                                       arr_s, arr_y, _stream(stream)))
    return outs


def gate_up_swiglu_fp8(x, s_in, w_gate, w_up, s_w_gate, s_w_up, s_out, out=None, ws=None, stream=None,
                       limit=None, alpha=None, beta=None):
    """Fused gate/up W8A8 GEMMs + SwiGLU -> E4M3 [M, I] for the down projection.
    With any of ``limit``, ``alpha``, ``beta`` given, the SwiGLU takes those
    options (``gate_up_swiglu_ex_fp8``; alpha defaults to 1, beta to 0)."""
    if x.dtype == torch.bfloat16:
        xd, dt = _as_bf16(x, "x"), DTYPE_BF16
    else:
        xd, dt = _as_u8(x, "x"), DTYPE_E4M3
    x2 = _flat2(xd)
    M, K = x2.shape
    wg, wu = _as_u8(w_gate, "w_gate"), _as_u8(w_up, "w_up")
    if wg.shape != wu.shape:
        raise W8Error(2, "gate and up weights differ in shape")
    I = wg.shape[0]
    if out is None:
        out = torch.empty(*x.shape[:-1], I, dtype=torch.uint8, device=x.device)
    o = _as_u8(out, "out")
    if dt == DTYPE_BF16 and ws is None:
        ws = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    wsp = _ptr(_as_u8(ws, "ws") if ws is not None else None)
    if limit is None and alpha is None and beta is None:
        _check(lib().gate_up_swiglu_fp8(_ptr(x2), dt, M, K, _ptr(_scalar(s_in, "s_in")), _ptr(wg), _ptr(wu), I,
                                        _ptr(_scalar(s_w_gate, "s_w_gate")), _ptr(_scalar(s_w_up, "s_w_up")),
                                        _ptr(_scalar(s_out, "s_out")), _ptr(o), wsp, _stream(stream)))
    else:
        prm = _swiglu_params(limit, 1.0 if alpha is None else alpha, 0.0 if beta is None else beta)
        _check(lib().gate_up_swiglu_ex_fp8(_ptr(x2), dt, M, K, _ptr(_scalar(s_in, "s_in")), _ptr(wg), _ptr(wu),
                                           I, _ptr(_scalar(s_w_gate, "s_w_gate")),
                                           _ptr(_scalar(s_w_up, "s_w_up")), ctypes.byref(prm),
                                           _ptr(_scalar(s_out, "s_out")), _ptr(o), wsp, _stream(stream)))
    return out


def fp8_linear_w8a8_noalloc(x, w, s_in, s_w, out=None, stream=None):
    """W8A8 linear on a bf16 activation using the library's fixed scratch
    array instead of a workspace (for callers that cannot allocate).  ``out``
    must be given by such callers; M*K is limited to 32 MiB."""
    xd = _as_bf16(x, "x")
    x2 = _flat2(xd)
    M, K = x2.shape
    wq = _as_u8(w, "w")
    N = wq.shape[0]
    if out is None:
        out = torch.empty(*x.shape[:-1], N, dtype=torch.bfloat16, device=x.device)
    _as_bf16(out, "out")
    _check(lib().fp8_linear_w8a8_noalloc(_ptr(x2), M, K, _ptr(wq), N, _ptr(_scalar(s_in, "s_in")),
                                         _ptr(_scalar(s_w, "s_w")), _ptr(out), _stream(stream)))
    return out


def swiglu_2in_fp8(gate, up, s_out, out=None, stream=None):
    g = _flat2(_as_bf16(gate, "gate"))
    u = _flat2(_as_bf16(up, "up"))
    if g.shape != u.shape:
        raise W8Error(2, "gate and up shapes differ")
    M, I = g.shape
    if out is None:
        out = torch.empty(gate.shape, dtype=torch.uint8, device=gate.device)
    _check(lib().swiglu_2in_fp8(_ptr(g), _ptr(u), M, I, _ptr(_scalar(s_out, "s_out")),
                                _ptr(_as_u8(out, "out")), _stream(stream)))
    return out


def swiglu_2in_bf16(gate, up, out=None, stream=None):
    g = _flat2(_as_bf16(gate, "gate"))
    u = _flat2(_as_bf16(up, "up"))
    if g.shape != u.shape:
        raise W8Error(2, "gate and up shapes differ")
    M, I = g.shape
    if out is None:
        out = torch.empty(gate.shape, dtype=torch.bfloat16, device=gate.device)
    _check(lib().swiglu_2in_bf16(_ptr(g), _ptr(u), M, I, _ptr(_as_bf16(out, "out")), _stream(stream)))
    return out


def _as_16(t, name):
    _dense(t, name)
    if t.dtype == torch.bfloat16:
        return t, DTYPE_BF16
    if t.dtype == torch.float16:
        return t, DTYPE_F16
    raise W8Error(5, f"{name}: expected bfloat16 or float16, got {t.dtype}")


def _swiglu_params(limit, alpha, beta):
    return SwigluParams(1 if limit is not None else 0, float(limit) if limit is not None else 0.0,
                        float(alpha), float(beta))


def _swiglu_ex_inputs(gate, up):
    (g, dt), (u, du) = _as_16(gate, "gate"), _as_16(up, "up")
    if dt != du:
        raise W8Error(5, "gate and up dtypes differ")
    g, u = _flat2(g), _flat2(u)
    if g.shape != u.shape:
        raise W8Error(2, "gate and up shapes differ")
    return g, u, dt


def swiglu_2in_ex_fp8(gate, up, s_out, limit=None, alpha=1.0, beta=0.0, out=None, stream=None):
    """SwiGLU with options (``limit``: clamp, ``alpha``: sigmoid slope,
    ``beta``: shift of up), bf16 or float16 inputs, E4M3 output."""
    g, u, dt = _swiglu_ex_inputs(gate, up)
    M, I = g.shape
    if out is None:
        out = torch.empty(gate.shape, dtype=torch.uint8, device=gate.device)
    prm = _swiglu_params(limit, alpha, beta)
    _check(lib().swiglu_2in_ex_fp8(_ptr(g), _ptr(u), dt, M, I, ctypes.byref(prm), _ptr(_scalar(s_out, "s_out")),
                                   _ptr(_as_u8(out, "out")), _stream(stream)))
    return out


def swiglu_2in_ex_16(gate, up, limit=None, alpha=1.0, beta=0.0, out=None, stream=None):
    """SwiGLU with options; output in the inputs' 16-bit format."""
    g, u, dt = _swiglu_ex_inputs(gate, up)
    M, I = g.shape
    if out is None:
        out = torch.empty(gate.shape, dtype=gate.dtype, device=gate.device)
    o, do = _as_16(out, "out")
    if do != dt:
        raise W8Error(5, "out must have the inputs' dtype")
    prm = _swiglu_params(limit, alpha, beta)
    _check(lib().swiglu_2in_ex_16(_ptr(g), _ptr(u), dt, M, I, ctypes.byref(prm), _ptr(o), _stream(stream)))
    return out


def step_policy_dispatch(policy, step, num_steps):
    """MODE_A8 or MODE_A16 for a scheduler step; ``policy`` None = no policy."""
    mode = ctypes.c_int32(-1)
    p = ctypes.byref(policy) if policy is not None else None
    _check(lib().step_policy_dispatch(p, step, num_steps, ctypes.byref(mode)))
    return mode.value


def step_policy_parse(text):
    """Parse a diffusion_step_policy JSON text: returns (StepPolicy, reasoner
    mode or None).  Raises W8Error (W8_ERR_POLICY) on any refused shape."""
    pol = StepPolicy()
    reasoner = ctypes.c_int32(-2)
    _check(lib().w8_step_policy_parse(text.encode() if isinstance(text, str) else text,
                                      ctypes.byref(pol), ctypes.byref(reasoner)))
    return pol, (None if reasoner.value < 0 else reasoner.value)


def check_group_scales(scales):
    """Load-time check that a sharing group's input scales are identical."""
    arr = (ctypes.c_void_p * len(scales))(*[_scalar(s, "s_in").data_ptr() for s in scales])
    _check(lib().w8_check_group_scales(arr, len(scales)))
