"""int8_quantized_gb300: Python binding of libi8q.so (include/i8q.h).

Argument marshalling only: every function passes device pointers of torch
CUDA tensors, sizes and the current CUDA stream to the C ABI, and raises
I8QError on a nonzero status.  No computation happens here, and there is no
fallback: without the built library every call raises.

Names follow the C entry points without their ``i8q_`` prefix.
"""
import ctypes

import torch

from . import _lib
from ._lib import (ACT_GELU, ACT_IDENTITY, ACT_RELU, BF16, F32, LSTM_BIDIRECTIONAL, LSTM_FORWARD, LSTM_REVERSE,
                   NO_AXIS, S8, S32, U8, I8QError, check, last_error)

__all__ = ["QGemmDyn", "quantize_linear", "dequantize_linear", "qlinearconv", "qlinearconv_workspace_size",
           "dq_lstm_forward", "dq_lstm_forward_ex", "dq_lstm_state_codes", "dq_lstm_workspace_size", "sync_status",
           "version", "I8QError", "last_error",
           "F32", "BF16", "S8", "U8", "S32", "ACT_IDENTITY", "ACT_RELU", "ACT_GELU", "NO_AXIS",
           "LSTM_FORWARD", "LSTM_REVERSE", "LSTM_BIDIRECTIONAL"]

_TORCH_TYPE = {torch.float32: F32, torch.bfloat16: BF16, torch.int8: S8, torch.uint8: U8, torch.int32: S32}


def _L():
    return _lib.load()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None):
    """Device pointer of a contiguous CUDA tensor (None passes NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _i64_array(vals):
    vals = list(int(v) for v in vals)
    return (ctypes.c_int64 * max(1, len(vals)))(*vals)


def version():
    return _L().i8q_version().decode()


def sync_status(stream=None):
    """Synchronize the stream and raise if a device-side bounded wait gave up."""
    check(_L().i8q_sync_status(_stream(stream)), "sync_status")


def profile_enable(on=True):
    """Start (dropping earlier records) or stop kernel timing."""
    check(_L().i8q_profile_enable(int(bool(on))), "profile_enable")


def profile_collect():
    """{kernel name: (launches, total ms)} of the launches timed so far."""
    n = _L().i8q_profile_collect()
    if n < 0:
        raise I8QError(n, "profile_collect")
    out = {}
    for i in range(n):
        name, launches, ms = ctypes.c_char_p(), ctypes.c_longlong(), ctypes.c_double()
        check(_L().i8q_profile_entry(i, ctypes.byref(name), ctypes.byref(launches), ctypes.byref(ms)),
              "profile_entry")
        out[name.value.decode()] = (int(launches.value), float(ms.value))
    return out


def measure_int8_mma_peak(iters=20000, stream=None):
    """Measured TOPS of back-to-back int8 mma.sync on every SM."""
    tops = ctypes.c_double()
    check(_L().i8q_measure_int8_mma_peak(int(iters), _stream(stream), ctypes.byref(tops)), "measure_int8_mma_peak")
    return float(tops.value)


# ---------------------------------------------------------------------------
class QGemmDyn:
    """Dynamic quantized inner product context (Simd
    SynetDynamicQuantizedInnerProduct16b: Init / Enable / InternalBufferSize /
    ExternalBufferSize / Info / SetParams / Forward / Clear)."""

    def __init__(self, M, N, K, typeA=F32, typeB=F32, typeC=F32, constB=True, bias=True, activation=ACT_IDENTITY,
                 avoidOverflow=False):
        self._ctx = ctypes.c_void_p(None)
        self.init(M, N, K, typeA, typeB, typeC, constB, bias, activation, avoidOverflow)

    def init(self, M, N, K, typeA=F32, typeB=F32, typeC=F32, constB=True, bias=True, activation=ACT_IDENTITY,
             avoidOverflow=False):
        check(_L().i8q_qgemm_dyn_init(ctypes.byref(self._ctx), M, N, K, typeA, typeB, typeC, int(bool(constB)),
                                      int(bool(bias)), activation, int(bool(avoidOverflow))), "qgemm_dyn_init")
        self.M, self.N, self.K = M, N, K
        self.typeA, self.typeB, self.typeC = typeA, typeB, typeC
        self.constB = bool(constB)

    def enabled(self):
        return bool(_L().i8q_qgemm_dyn_enabled(self._ctx))

    def internal_buffer_size(self):
        return int(_L().i8q_qgemm_dyn_internal_buffer_size(self._ctx))

    def external_buffer_size(self):
        return int(_L().i8q_qgemm_dyn_external_buffer_size(self._ctx))

    def info(self):
        r = _L().i8q_qgemm_dyn_info(self._ctx)
        return None if r is None else r.decode()

    def set_params(self, weight=None, scale=None, bias=None, params=None, stream=None):
        """weight K x N (fp32 or int8), scale N fp32, bias N fp32: CUDA tensors."""
        check(_L().i8q_qgemm_dyn_set_params(self._ctx, _dev(weight, "weight"), _dev(scale, "scale", torch.float32),
                                            _dev(bias, "bias", torch.float32), _dev(params, "params", torch.float32),
                                            _stream(stream)), "qgemm_dyn_set_params")

    def forward(self, A, C, B=None, buf=None, stream=None):
        check(_L().i8q_qgemm_dyn_forward(self._ctx, _dev(A, "A"), _dev(B, "B"), _dev(buf, "buf"), _dev(C, "C"),
                                         _stream(stream)), "qgemm_dyn_forward")
        return C

    def forward_s32(self, A, acc, B=None, buf=None, stream=None):
        check(_L().i8q_qgemm_dyn_forward_s32(self._ctx, _dev(A, "A"), _dev(B, "B"), _dev(buf, "buf"),
                                             _dev(acc, "acc", torch.int32), _stream(stream)), "qgemm_dyn_forward_s32")
        return acc

    def forward_host(self, A_host, C_host, stream=None):
        """A_host, C_host: CPU tensors (pinned for asynchronous copies)."""
        for t, n in ((A_host, "A_host"), (C_host, "C_host")):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError(f"{n} must be a contiguous CPU tensor")
        check(_L().i8q_qgemm_dyn_forward_host(self._ctx, ctypes.c_void_p(A_host.data_ptr()),
                                              ctypes.c_void_p(C_host.data_ptr()), _stream(stream)),
              "qgemm_dyn_forward_host")
        return C_host

    def buf_views(self, buf=None):
        """(uA M x lda uint8, scaleA M fp32, zeroA M int32) written by the last
        forward, as torch views of the device buffer."""
        uA, lda, sA, zA = ctypes.c_void_p(), ctypes.c_size_t(), ctypes.c_void_p(), ctypes.c_void_p()
        check(_L().i8q_qgemm_dyn_buf_views(self._ctx, _dev(buf, "buf"), ctypes.byref(uA), ctypes.byref(lda),
                                           ctypes.byref(sA), ctypes.byref(zA)), "qgemm_dyn_buf_views")
        return (_wrap(uA.value, (self.M, lda.value), torch.uint8), _wrap(sA.value, (self.M,), torch.float32),
                _wrap(zA.value, (self.M,), torch.int32), lda.value)

    def weight_views(self, buf=None):
        """(iBt N x ldb int32 codes, scaleB N fp32, colsum N int32, ldb) of
        the stored constant B, or of the B the last forward quantized into
        buf; the codes are read from whichever copy (int8 or bf16) is kept."""
        q8, qb, ldb = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_size_t()
        s, cs = ctypes.c_void_p(), ctypes.c_void_p()
        check(_L().i8q_qgemm_dyn_weight_views(self._ctx, _dev(buf, "buf"), ctypes.byref(q8), ctypes.byref(qb),
                                              ctypes.byref(ldb), ctypes.byref(s), ctypes.byref(cs)),
              "qgemm_dyn_weight_views")
        if q8.value:
            codes = _wrap(q8.value, (self.N, ldb.value), torch.int8).to(torch.int32)
        else:
            raw = _wrap(qb.value, (self.N, ldb.value), torch.int16)
            codes = raw.view(torch.bfloat16).float().to(torch.int32)
        return (codes, _wrap(s.value, (self.N,), torch.float32), _wrap(cs.value, (self.N,), torch.int32),
                ldb.value)

    def clear(self):
        if getattr(self, "_ctx", None) is not None and self._ctx.value:
            _L().i8q_qgemm_dyn_clear(ctypes.byref(self._ctx))

    def __del__(self):
        try:
            self.clear()
        except Exception:
            pass


_TYPESTR = {torch.uint8: "|u1", torch.int8: "|i1", torch.float32: "<f4", torch.int32: "<i4", torch.int16: "<i2"}


class _DeviceArray:
    """Describes library-owned device memory to torch (CUDA array interface)."""

    def __init__(self, ptr, shape, dtype):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": _TYPESTR[dtype], "data": (ptr, False),
                                         "version": 2, "strides": None}


def _wrap(ptr, shape, dtype):
    """Copy of device memory owned by the library, as a torch tensor (the
    copy does not alias library storage)."""
    torch.cuda.current_stream().synchronize()
    return torch.as_tensor(_DeviceArray(ptr, shape, dtype), device="cuda").clone()


# ---------------------------------------------------------------------------
def quantize_linear(x, y_scale, y_zero_point, y, axis=None, stream=None):
    """QuantizeLinear: y (uint8/int8 CUDA tensor, shape of x) from fp32 x;
    y_scale / y_zero_point CUDA tensors (1 entry, or dim[axis] entries)."""
    yt = _TORCH_TYPE[y.dtype]
    if y_zero_point.dtype != y.dtype:
        raise TypeError("y_zero_point must have y's dtype")
    shape = _i64_array(x.shape)
    check(_L().i8q_quantize_linear(_dev(x, "x", torch.float32), shape, x.dim(), NO_AXIS if axis is None else axis,
                                   _dev(y_scale, "y_scale", torch.float32), _dev(y_zero_point, "y_zero_point"),
                                   y_scale.numel(), yt, _dev(y, "y"), _stream(stream)), "quantize_linear")
    return y


def dequantize_linear(x, x_scale, x_zero_point, y, axis=None, stream=None):
    """DequantizeLinear: fp32 y from uint8/int8 x."""
    xt = _TORCH_TYPE[x.dtype]
    shape = _i64_array(x.shape)
    check(_L().i8q_dequantize_linear(_dev(x, "x"), xt, shape, x.dim(), NO_AXIS if axis is None else axis,
                                     _dev(x_scale, "x_scale", torch.float32), _dev(x_zero_point, "x_zero_point"),
                                     x_scale.numel(), _dev(y, "y", torch.float32), _stream(stream)),
          "dequantize_linear")
    return y


def _conv_arrays(x_shape, w_shape, pads, strides, dilations):
    return (_i64_array(x_shape), _i64_array(w_shape), _i64_array(pads), _i64_array(strides), _i64_array(dilations))


def qlinearconv_workspace_size(x_shape, w_shape, pads=(0, 0, 0, 0), strides=(1, 1), dilations=(1, 1), group=1):
    xs, ws, p, s, d = _conv_arrays(x_shape, w_shape, pads, strides, dilations)
    return int(_L().i8q_qlinearconv_workspace_size(xs, ws, p, s, d, group))


def qlinearconv(x, x_scale, x_zero_point, w, w_scale, w_zero_point, y_scale, y_zero_point, y, B=None,
                pads=(0, 0, 0, 0), strides=(1, 1), dilations=(1, 1), group=1, workspace=None, stream=None):
    """QLinearConv, NCHW.  x_scale, y_scale: floats; x_zero_point,
    y_zero_point: ints; w_scale (fp32) / w_zero_point (w's dtype): CUDA
    tensors of 1 or M entries; B: int32 CUDA tensor [M] or None.
    workspace: uint8 CUDA tensor of qlinearconv_workspace_size bytes; when
    None and the shape needs one, it is allocated here for this call."""
    xs, ws, p, s, d = _conv_arrays(x.shape, w.shape, pads, strides, dilations)
    if w_zero_point.dtype != w.dtype:
        raise TypeError("w_zero_point must have w's dtype")
    if workspace is None:
        need = int(_L().i8q_qlinearconv_workspace_size(xs, ws, p, s, d, int(group)))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=y.device)
    check(_L().i8q_qlinearconv(_dev(x, "x"), _TORCH_TYPE[x.dtype], xs, float(x_scale), int(x_zero_point),
                               _dev(w, "w"), _TORCH_TYPE[w.dtype], ws, _dev(w_scale, "w_scale", torch.float32),
                               _dev(w_zero_point, "w_zero_point"), w_scale.numel(), float(y_scale),
                               int(y_zero_point), _dev(B, "B", torch.int32), p, s, d, int(group), _dev(y, "y"),
                               _TORCH_TYPE[y.dtype], _dev(workspace, "workspace"),
                               0 if workspace is None else workspace.numel() * workspace.element_size(),
                               _stream(stream)), "qlinearconv")
    return y


def qgemm_workspace_size(M, N, K):
    return int(_L().i8q_qgemm_workspace_size(M, N, K))


def qgemm(A, a_scale, a_zero_point, B, b_scale, Y, b_zero_point=None, C=None, alpha=1.0, y_scale=None,
          y_zero_point=0, transA=False, transB=False, workspace=None, stream=None):
    """QGemm.  A: uint8/int8 CUDA (M, K), or (K, M) with transA; B: uint8/int8
    CUDA (K, N), or (N, K) with transB; a_scale, a_zero_point: Python
    scalars; b_scale: fp32 CUDA tensor of 1 or N entries; b_zero_point: B's
    dtype, same count, or None; C: int32 CUDA tensor broadcastable to (M, N)
    as (1|M, 1|N) or (N,), or None.  Y: fp32 (M, N), or uint8/int8 (M, N)
    with y_scale given.  workspace: uint8 CUDA tensor of
    qgemm_workspace_size(M, N, K) bytes; allocated here when None."""
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    N = B.shape[0] if transB else B.shape[1]
    if b_zero_point is not None and b_zero_point.dtype != B.dtype:
        raise TypeError("b_zero_point must have B's dtype")
    cr = cc = 0
    if C is not None:
        if C.dim() == 0:
            cr, cc = 1, 1
        elif C.dim() == 1:
            cr, cc = 1, C.shape[0]
        else:
            cr, cc = C.shape
    quant = y_scale is not None
    if quant and Y.dtype not in (torch.uint8, torch.int8):
        raise TypeError("quantized Y must be uint8 or int8")
    if not quant and Y.dtype != torch.float32:
        raise TypeError("Y must be float32 when y_scale is None")
    if workspace is None:
        workspace = torch.empty(qgemm_workspace_size(M, N, K), dtype=torch.uint8, device=Y.device)
    check(_L().i8q_qgemm(_dev(A, "A"), _TORCH_TYPE[A.dtype], int(bool(transA)), M, K, float(a_scale),
                         int(a_zero_point), _dev(B, "B"), _TORCH_TYPE[B.dtype], int(bool(transB)), N,
                         _dev(b_scale, "b_scale", torch.float32), _dev(b_zero_point, "b_zero_point"),
                         b_scale.numel(), _dev(C, "C", torch.int32), cr, cc, float(alpha), int(quant),
                         float(y_scale) if quant else 1.0, int(y_zero_point), _TORCH_TYPE[Y.dtype], _dev(Y, "Y"),
                         _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)),
          "qgemm")
    return Y


def matmul_integer_workspace_size(M, N, K):
    return int(_L().i8q_matmul_integer_workspace_size(M, N, K))


def matmul_integer_to_float(A, B, a_scale, b_scale, Y, a_zero_point=None, b_zero_point=None, bias=None,
                            workspace=None, stream=None):
    """MatMulIntegerToFloat.  A: uint8/int8 CUDA (..., K) (leading dims are
    rows); B: uint8/int8 CUDA (K, N); a_scale: fp32 CUDA, 1 entry or one per
    row of A; a_zero_point: A's dtype, same count, or None; b_scale /
    b_zero_point: 1 or N entries; bias: fp32 CUDA [N] or None; Y: fp32 CUDA
    (..., N)."""
    K = A.shape[-1]
    M = A.numel() // K
    N = B.shape[1]
    for z, t, n in ((a_zero_point, A, "a_zero_point"), (b_zero_point, B, "b_zero_point")):
        if z is not None and z.dtype != t.dtype:
            raise TypeError(f"{n} must have the dtype of its operand")
    if workspace is None:
        workspace = torch.empty(matmul_integer_workspace_size(M, N, K), dtype=torch.uint8, device=Y.device)
    check(_L().i8q_matmul_integer_to_float(
        _dev(A, "A"), _TORCH_TYPE[A.dtype], M, K, _dev(B, "B"), _TORCH_TYPE[B.dtype], N,
        _dev(a_scale, "a_scale", torch.float32), _dev(a_zero_point, "a_zero_point"), a_scale.numel(),
        _dev(b_scale, "b_scale", torch.float32), _dev(b_zero_point, "b_zero_point"), b_scale.numel(),
        _dev(bias, "bias", torch.float32), _dev(Y, "Y", torch.float32), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "matmul_integer_to_float")
    return Y


def dynamic_quantize_matmul(A, B, b_scale, Y, b_zero_point=None, bias=None, a_scale_out=None, a_zero_point_out=None,
                            workspace=None, stream=None):
    """DynamicQuantizeMatMul.  A: fp32 CUDA (..., K), quantized to uint8 per
    tensor; B: uint8/int8 CUDA (K, N); b_scale / b_zero_point: 1 or N
    entries; bias: fp32 [N] or None; Y: fp32 (..., N).  a_scale_out (fp32,
    1) and a_zero_point_out (uint8, 1) receive A's parameters when given."""
    K = A.shape[-1]
    M = A.numel() // K
    N = B.shape[1]
    if b_zero_point is not None and b_zero_point.dtype != B.dtype:
        raise TypeError("b_zero_point must have B's dtype")
    if workspace is None:
        workspace = torch.empty(matmul_integer_workspace_size(M, N, K), dtype=torch.uint8, device=Y.device)
    check(_L().i8q_dynamic_quantize_matmul(
        _dev(A, "A", torch.float32), M, K, _dev(B, "B"), _TORCH_TYPE[B.dtype], N, _dev(b_scale, "b_scale", torch.float32),
        _dev(b_zero_point, "b_zero_point"), b_scale.numel(), _dev(bias, "bias", torch.float32),
        _dev(Y, "Y", torch.float32), _dev(a_scale_out, "a_scale_out", torch.float32),
        _dev(a_zero_point_out, "a_zero_point_out", torch.uint8), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream)), "dynamic_quantize_matmul")
    return Y


QLINEAR_ADD, QLINEAR_MUL = 0, 1
QLINEAR_LEAKY_RELU, QLINEAR_SIGMOID = 0, 1


def _shape_array(t):
    return _i64_array(t.shape) if t.dim() > 0 else None


def qlinear_binary(op, A, a_scale, a_zero_point, B, b_scale, b_zero_point, c_scale, c_zero_point, C, stream=None):
    """QLinearAdd (op "add") / QLinearMul (op "mul"): A, B, C uint8 or int8
    CUDA tensors of one dtype; C has the broadcast shape of A and B."""
    if not (A.dtype == B.dtype == C.dtype):
        raise TypeError("A, B and C must have one dtype")
    check(_L().i8q_qlinear_binary({"add": QLINEAR_ADD, "mul": QLINEAR_MUL}[op], _dev(A, "A"), _shape_array(A), A.dim(),
                                  float(a_scale), int(a_zero_point), _dev(B, "B"), _shape_array(B), B.dim(),
                                  float(b_scale), int(b_zero_point), float(c_scale), int(c_zero_point),
                                  _TORCH_TYPE[A.dtype], _dev(C, "C"), _stream(stream)), "qlinear_binary")
    return C


def mul_integer(A, a_zero_point, B, b_zero_point, C, stream=None):
    """MulInteger: C int32 with the broadcast shape of A and B."""
    check(_L().i8q_mul_integer(_dev(A, "A"), _TORCH_TYPE[A.dtype], _shape_array(A), A.dim(), int(a_zero_point),
                               _dev(B, "B"), _TORCH_TYPE[B.dtype], _shape_array(B), B.dim(), int(b_zero_point),
                               _dev(C, "C", torch.int32), _stream(stream)), "mul_integer")
    return C


def qlinear_unary(op, X, x_scale, x_zero_point, y_scale, y_zero_point, Y, alpha=0.01, stream=None):
    """QLinearLeakyRelu (op "leaky_relu") / QLinearSigmoid (op "sigmoid")."""
    if X.dtype != Y.dtype or X.numel() != Y.numel():
        raise TypeError("X and Y must have one dtype and size")
    check(_L().i8q_qlinear_unary({"leaky_relu": QLINEAR_LEAKY_RELU, "sigmoid": QLINEAR_SIGMOID}[op], _dev(X, "X"),
                                 X.numel(), _TORCH_TYPE[X.dtype], float(x_scale), int(x_zero_point), float(y_scale),
                                 int(y_zero_point), float(alpha), _dev(Y, "Y"), _stream(stream)), "qlinear_unary")
    return Y


def dq_lstm_workspace_size(T, batch, input_size, hidden, direction):
    return int(_L().i8q_dq_lstm_workspace_size(T, batch, input_size, hidden, direction))


def dq_lstm_forward(X, W, R, W_scale, R_scale, workspace, direction=LSTM_FORWARD, B=None, h0=None, c0=None,
                    Y=None, Y_h=None, Y_c=None, W_zero_point=None, R_zero_point=None, stream=None):
    """DynamicQuantizeLSTM.  X [T, batch, I] fp32; W [D, I, 4H], R [D, H, 4H]
    int8; scales [D] or [D, 4H]; B [D, 8H]; h0, c0 [D, batch, H];
    outputs Y [T, D, batch, H], Y_h, Y_c [D, batch, H] (each optional)."""
    T, batch, I = X.shape
    H = R.shape[1]
    check(_L().i8q_dq_lstm_forward(
        _dev(X, "X", torch.float32), T, batch, I, H, direction, _dev(W, "W", torch.int8),
        _dev(W_scale, "W_scale", torch.float32), _dev(W_zero_point, "W_zero_point"), W_scale.numel(),
        _dev(R, "R", torch.int8), _dev(R_scale, "R_scale", torch.float32), _dev(R_zero_point, "R_zero_point"),
        R_scale.numel(), _dev(B, "B", torch.float32), _dev(h0, "h0", torch.float32), _dev(c0, "c0", torch.float32),
        _dev(Y, "Y", torch.float32), _dev(Y_h, "Y_h", torch.float32), _dev(Y_c, "Y_c", torch.float32),
        _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream)),
        "dq_lstm_forward")
    return Y, Y_h, Y_c


def dq_lstm_forward_ex(X, W, R, W_scale, R_scale, workspace, direction=LSTM_FORWARD, B=None, sequence_lens=None,
                       h0=None, c0=None, P=None, clip=0.0, input_forget=False, Y=None, Y_h=None, Y_c=None,
                       W_zero_point=None, R_zero_point=None, activations=None, activation_alpha=None,
                       activation_beta=None, stream=None):
    """DynamicQuantizeLSTM with the optional inputs and attributes: W, R
    uint8 or int8 (one dtype) with zero points of that dtype ([D] or
    [D, 4H]); sequence_lens int32 [batch]; P [D, 3H]; clip (<= 0: none);
    input_forget; activations: 3 names per direction from
    _lib.LSTM_ACTIVATIONS (None: Sigmoid, Tanh, Tanh) with the
    activation_alpha / activation_beta lists.  Shapes otherwise as
    dq_lstm_forward."""
    T, batch, I = X.shape
    H = R.shape[1]
    if W.dtype != R.dtype or W.dtype not in (torch.uint8, torch.int8):
        raise TypeError("W and R must both be uint8 or both int8")
    for z, n in ((W_zero_point, "W_zero_point"), (R_zero_point, "R_zero_point")):
        if z is not None and z.dtype != W.dtype:
            raise TypeError(f"{n} must have W's dtype")
    kinds = [_lib.LSTM_ACTIVATIONS.index(a) for a in (activations or [])]
    alpha = [float(a) for a in (activation_alpha or [])]
    beta = [float(b) for b in (activation_beta or [])]
    c_kinds = (ctypes.c_int * max(1, len(kinds)))(*kinds)
    c_alpha = (ctypes.c_float * max(1, len(alpha)))(*alpha)
    c_beta = (ctypes.c_float * max(1, len(beta)))(*beta)
    check(_L().i8q_dq_lstm_forward_ex(
        _dev(X, "X", torch.float32), T, batch, I, H, direction, _dev(W, "W"), _dev(R, "R"), _TORCH_TYPE[W.dtype],
        _dev(W_scale, "W_scale", torch.float32), _dev(W_zero_point, "W_zero_point"), W_scale.numel(),
        _dev(R_scale, "R_scale", torch.float32), _dev(R_zero_point, "R_zero_point"), R_scale.numel(),
        _dev(B, "B", torch.float32), _dev(sequence_lens, "sequence_lens", torch.int32),
        _dev(h0, "h0", torch.float32), _dev(c0, "c0", torch.float32), _dev(P, "P", torch.float32), float(clip),
        int(bool(input_forget)), c_kinds, len(kinds), c_alpha, len(alpha), c_beta, len(beta),
        _dev(Y, "Y", torch.float32), _dev(Y_h, "Y_h", torch.float32),
        _dev(Y_c, "Y_c", torch.float32), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream)), "dq_lstm_forward_ex")
    return Y, Y_h, Y_c


def dq_lstm_state_codes(workspace, T, batch, input_size, hidden, direction, which):
    """Test hook: the per-row uint8 codes (as int32 [D * batch, hidden]),
    scales and zero points of a hidden state, read back from the workspace
    of a completed LSTM call (which 0: the state the last step read; 1: the
    final state).  Synchronizes the current stream."""
    codes, scale, zero = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    stride = ctypes.c_int64()
    check(_L().i8q_dq_lstm_state_codes(_dev(workspace, "workspace"), T, batch, input_size, hidden, direction, which,
                                       ctypes.byref(codes), ctypes.byref(scale), ctypes.byref(zero),
                                       ctypes.byref(stride)), "dq_lstm_state_codes")
    D = 2 if direction == LSTM_BIDIRECTIONAL else 1
    base = workspace.data_ptr()
    torch.cuda.current_stream().synchronize()

    def view(ptr, n, dtype, esize):
        off = ptr - base
        if off < 0 or off % esize or off + n * esize > workspace.numel() * workspace.element_size():
            raise ValueError("state codes outside the workspace")
        return workspace.view(torch.uint8)[off:off + n * esize].view(dtype)

    rows = D * batch
    c = view(codes.value, rows * stride.value, torch.bfloat16, 2).view(rows, stride.value)[:, :hidden]
    return (c.float().to(torch.int32) + 128, view(scale.value, rows, torch.float32, 4).clone(),
            view(zero.value, rows, torch.int32, 4).clone())
