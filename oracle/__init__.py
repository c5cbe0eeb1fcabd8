"""Python face of the CPU oracle (ctypes over oracle/oracle.c, numpy arrays).

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``; never by the product package.
It shares no code with the CUDA library.  Each wrapper names the operator
text it follows; the arithmetic itself lives in oracle.c, except for the
compositions below, which only chain oracle.c calls in the order the pages
give.
"""
import ctypes
import os

import numpy as np

from . import build as _build

U8, S8 = 0, 1
ACT_IDENTITY, ACT_RELU, ACT_GELU = 0, 1, 2

_lib = None


def load(path):
    """Open a built oracle library and declare its signatures."""
    l = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    i32 = ctypes.c_int32
    f32 = ctypes.c_float
    c_int = ctypes.c_int
    l.or_quantize_linear.argtypes = [p, i64, i64, i64, p, p, c_int, c_int, p]
    l.or_dequantize_linear.argtypes = [p, c_int, i64, i64, i64, p, p, c_int, p]
    l.or_quantize_rows_u8.argtypes = [p, i64, i64, p, p, p]
    l.or_quantize_cols_s8.argtypes = [p, i64, i64, c_int, p, p]
    l.or_qgemm_dyn_rows.argtypes = [p, p, p, p, p, p, c_int, i64, i64, i64, p, i64, p, p]
    l.or_f32_to_bf16.argtypes = [p, i64, p]
    l.or_f32_to_bf16.restype = None
    l.or_qlinearconv.argtypes = [p, c_int, i64, i64, i64, i64, f32, i32, p, c_int, i64, i64,
                                 i64, p, p, c_int, f32, i32, p, p, p, p, i64, p, c_int]
    l.or_lstm_cell.argtypes = [p, p, p, p, p, p, p, i64, i64]
    l.or_lstm_cell_ex.argtypes = [p, p, p, p, p, f32, c_int, p, p, p, p, p, p, i64, i64]
    l.or_elementary.argtypes = [c_int, p, i64, p]
    l.or_dyn_product_zp.argtypes = [p, p, p, p, c_int, p, i64, p, i64, i64, i64, p]
    l.or_qgemm.argtypes = [p, c_int, c_int, i64, i64, f32, i32, p, c_int, c_int, i64, p, p, i64, p, i64, i64,
                           f32, c_int, f32, i32, c_int, p]
    l.or_matmul_integer_to_float.argtypes = [p, c_int, i64, i64, p, c_int, i64, p, p, i64, p, p, i64, p, p]
    l.or_mul_integer.argtypes = [p, c_int, p, i32, p, c_int, p, i32, p, c_int, p]
    l.or_qlinear_binary.argtypes = [c_int, p, p, f32, i32, p, p, f32, i32, f32, i32, p, c_int, c_int, p]
    l.or_qlinear_unary.argtypes = [c_int, p, i64, c_int, f32, i32, f32, i32, f32, p]
    for fn in ("or_quantize_linear", "or_dequantize_linear", "or_quantize_rows_u8",
               "or_quantize_cols_s8", "or_qgemm_dyn_rows", "or_qlinearconv", "or_lstm_cell", "or_qgemm",
               "or_matmul_integer_to_float", "or_mul_integer", "or_qlinear_binary", "or_qlinear_unary",
               "or_lstm_cell_ex", "or_dyn_product_zp", "or_elementary"):
        getattr(l, fn).restype = ctypes.c_int
    return l


def lib():
    """The oracle library.  ORACLE_LIB_UNDER_TEST names another build of
    oracle.c to load instead; the mutation tests use it to check that the
    pins fail on planted mistakes."""
    global _lib
    if _lib is None:
        _lib = load(os.environ.get("ORACLE_LIB_UNDER_TEST") or _build.build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def _qtype(t):
    return {"u8": U8, "s8": S8, U8: U8, S8: S8}[t]


def _np_qdtype(t):
    return np.uint8 if _qtype(t) == U8 else np.int8


def _axis_view(shape, axis):
    """[outer, axis_len, inner] view of a shape for the per-axis index."""
    rank = len(shape)
    if axis is None:
        n = int(np.prod(shape)) if rank else 1
        return 1, n, 1
    a = axis + rank if axis < 0 else axis
    outer = int(np.prod(shape[:a])) if a > 0 else 1
    inner = int(np.prod(shape[a + 1:])) if a + 1 < rank else 1
    return outer, int(shape[a]), inner


def quantize_linear(x, y_scale, y_zero_point, axis=None, ytype="u8"):
    """QuantizeLinear (ONNX Runtime contrib schema, ver 1): saturating,
    round-half-even x / y_scale plus zero point.  axis=None is per tensor."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s = np.ascontiguousarray(np.atleast_1d(y_scale), dtype=np.float32)
    z = np.ascontiguousarray(np.atleast_1d(y_zero_point), dtype=np.int32)
    outer, alen, inner = _axis_view(x.shape, axis)
    if axis is not None and (s.size != alen or z.size != alen):
        raise ValueError("per-axis scale/zero point length must equal dim[axis]")
    y = np.empty(x.shape, dtype=_np_qdtype(ytype))
    _check(lib().or_quantize_linear(_ptr(x), outer, alen, inner, _ptr(s), _ptr(z),
                                    int(axis is not None), _qtype(ytype), _ptr(y)), "quantize_linear")
    return y


def dequantize_linear(x, x_scale, x_zero_point, axis=None):
    """DequantizeLinear (ONNX Runtime contrib schema, ver 1): (x - zp) * scale."""
    x = np.ascontiguousarray(x)
    xtype = U8 if x.dtype == np.uint8 else S8
    if x.dtype not in (np.uint8, np.int8):
        raise TypeError("x must be uint8 or int8")
    s = np.ascontiguousarray(np.atleast_1d(x_scale), dtype=np.float32)
    z = np.ascontiguousarray(np.atleast_1d(x_zero_point), dtype=np.int32)
    outer, alen, inner = _axis_view(x.shape, axis)
    y = np.empty(x.shape, dtype=np.float32)
    _check(lib().or_dequantize_linear(_ptr(x), xtype, outer, alen, inner, _ptr(s), _ptr(z),
                                      int(axis is not None), _ptr(y)), "dequantize_linear")
    return y


def bf16_bits_to_f32(bits):
    """Exact widening of bf16 (given as uint16 bit patterns) to fp32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x):
    """fp32 -> bf16 bit patterns, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16)
    lib().or_f32_to_bf16(_ptr(x), x.size, _ptr(y))
    return y


def quantize_rows_u8(A):
    """Per-row uint8 dynamic quantization of A (M x K fp32)."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    M, K = A.shape
    uA = np.empty((M, K), dtype=np.uint8)
    sA = np.empty(M, dtype=np.float32)
    zA = np.empty(M, dtype=np.int32)
    _check(lib().or_quantize_rows_u8(_ptr(A), M, K, _ptr(uA), _ptr(sA), _ptr(zA)), "quantize_rows_u8")
    return uA, sA, zA


def quantize_cols_s8(B, avoid_overflow=False):
    """Per-column symmetric int8 quantization of B (K x N fp32)."""
    B = np.ascontiguousarray(B, dtype=np.float32)
    K, N = B.shape
    iB = np.empty((K, N), dtype=np.int8)
    sB = np.empty(N, dtype=np.float32)
    _check(lib().or_quantize_cols_s8(_ptr(B), K, N, int(bool(avoid_overflow)), _ptr(iB), _ptr(sB)),
           "quantize_cols_s8")
    return iB, sB


def qgemm_rows(uA, zA, sA, iB, sB, bias=None, act=ACT_IDENTITY, rows=None):
    """Integer product, dequantization, bias and activation of the Simd
    dynamic quantized inner product, for the listed rows (all if None).
    Returns (int32 sums, fp32 outputs), each len(rows) x N."""
    uA = np.ascontiguousarray(uA, dtype=np.uint8)
    iB = np.ascontiguousarray(iB, dtype=np.int8)
    zA = np.ascontiguousarray(zA, dtype=np.int32)
    sA = np.ascontiguousarray(sA, dtype=np.float32)
    sB = np.ascontiguousarray(sB, dtype=np.float32)
    M, K = uA.shape
    K2, N = iB.shape
    assert K == K2
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else r.size
    acc = np.empty((nr, N), dtype=np.int32)
    C = np.empty((nr, N), dtype=np.float32)
    _check(lib().or_qgemm_dyn_rows(_ptr(uA), _ptr(zA), _ptr(sA), _ptr(iB), _ptr(sB), _ptr(b), act,
                                   M, N, K, _ptr(r), nr, _ptr(acc), _ptr(C)), "qgemm_dyn_rows")
    return acc, C


def dynamic_quantized_inner_product(A, B=None, *, iB=None, scaleB=None, bias=None,
                                    act=ACT_IDENTITY, avoid_overflow=False, typeC="f32",
                                    rows=None):
    """Whole Simd dynamic quantized inner product: quantize A per row, take B
    as given int8 (iB, scaleB) or quantize fp32 B per column, then the
    integer product and its epilogue.  typeC 'bf16' returns bf16 bits.
    A may be fp32, or bf16 bits (uint16), which widen exactly."""
    A = np.asarray(A)
    if A.dtype == np.uint16:
        A = bf16_bits_to_f32(A)
    uA, sA, zA = quantize_rows_u8(A)
    if iB is None:
        Bf = np.asarray(B)
        if Bf.dtype == np.uint16:
            Bf = bf16_bits_to_f32(Bf)
        iB, scaleB = quantize_cols_s8(Bf, avoid_overflow)
    acc, C = qgemm_rows(uA, zA, sA, iB, scaleB, bias, act, rows)
    out = {"uA": uA, "scaleA": sA, "zeroA": zA, "iB": iB, "scaleB": scaleB, "acc": acc, "C32": C}
    out["C"] = f32_to_bf16_bits(C) if typeC == "bf16" else C
    return out


def qlinearconv(x, x_scale, x_zero_point, w, w_scale, w_zero_point, y_scale, y_zero_point,
                B=None, pads=(0, 0, 0, 0), strides=(1, 1), dilations=(1, 1), group=1, ytype=None):
    """2-D QLinearConv (ONNX, since version 10) on NCHW tensors.
    pads = (top, left, bottom, right).  Output type defaults to x's type."""
    x = np.ascontiguousarray(x)
    w = np.ascontiguousarray(w)
    xt = U8 if x.dtype == np.uint8 else S8
    wt = U8 if w.dtype == np.uint8 else S8
    yt = xt if ytype is None else _qtype(ytype)
    N, C, H, W = x.shape
    M, Cg, kH, kW = w.shape
    ws = np.ascontiguousarray(np.atleast_1d(w_scale), dtype=np.float32)
    wz = np.ascontiguousarray(np.atleast_1d(w_zero_point), dtype=np.int32)
    per_ch = int(ws.size == M and M > 1)
    if ws.size not in (1, M) or wz.size != ws.size:
        raise ValueError("w_scale / w_zero_point must be scalars or have M entries")
    if C != Cg * group:
        raise ValueError("x.shape[1] must equal w.shape[1] * group")
    pads = np.asarray(pads, dtype=np.int64)
    strides = np.asarray(strides, dtype=np.int64)
    dil = np.asarray(dilations, dtype=np.int64)
    OH = (H + pads[0] + pads[2] - ((kH - 1) * dil[0] + 1)) // strides[0] + 1
    OW = (W + pads[1] + pads[3] - ((kW - 1) * dil[1] + 1)) // strides[1] + 1
    y = np.empty((N, M, OH, OW), dtype=np.uint8 if yt == U8 else np.int8)
    b = None if B is None else np.ascontiguousarray(B, dtype=np.int32)
    _check(lib().or_qlinearconv(_ptr(x), xt, N, C, H, W, float(x_scale), int(x_zero_point),
                                _ptr(w), wt, M, kH, kW, _ptr(ws), _ptr(wz), per_ch,
                                float(y_scale), int(y_zero_point), _ptr(b), _ptr(pads),
                                _ptr(strides), _ptr(dil), group, _ptr(y), yt), "qlinearconv")
    return y


def qgemm(A, a_scale, a_zero_point, B, b_scale, b_zero_point=None, C=None, alpha=1.0, y_scale=None,
          y_zero_point=None, transA=False, transB=False, ytype=None):
    """QGemm (ONNX Runtime contrib schemas).  A: uint8/int8 (M, K), or (K, M)
    when transA; B: uint8/int8 (K, N), or (N, K) when transB; b_scale and
    b_zero_point: scalars or N entries; C: int32 broadcastable to (M, N)
    ((M, N), (1, N), (N,), (M, 1), (1, 1) or a scalar).  Float output unless
    y_scale is given; the quantized type is y_zero_point's (uint8 when it is
    a plain int and ytype is not given)."""
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    at = U8 if A.dtype == np.uint8 else S8
    bt = U8 if B.dtype == np.uint8 else S8
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    N = B.shape[0] if transB else B.shape[1]
    if (B.shape[1] if transB else B.shape[0]) != K:
        raise ValueError("inner dimensions differ")
    bs = np.ascontiguousarray(np.atleast_1d(b_scale), dtype=np.float32)
    bz = None if b_zero_point is None else np.ascontiguousarray(np.atleast_1d(b_zero_point), dtype=np.int32)
    if bs.size not in (1, N) or (bz is not None and bz.size != bs.size):
        raise ValueError("b_scale / b_zero_point must be scalars or have N entries")
    c = None
    cr = cc = 0
    if C is not None:
        c = np.asarray(C, dtype=np.int32)
        if c.ndim == 0:
            c = c.reshape(1, 1)
        elif c.ndim == 1:
            c = c.reshape(1, -1)
        cr, cc = c.shape
        c = np.ascontiguousarray(c)
    quant = y_scale is not None
    if quant:
        yt = _qtype(ytype) if ytype is not None else (
            S8 if isinstance(y_zero_point, np.integer) and np.asarray(y_zero_point).dtype == np.int8 else U8)
        Y = np.empty((M, N), dtype=np.uint8 if yt == U8 else np.int8)
    else:
        yt = U8
        Y = np.empty((M, N), dtype=np.float32)
    _check(lib().or_qgemm(_ptr(A), at, int(bool(transA)), M, K, float(a_scale), int(a_zero_point), _ptr(B), bt,
                          int(bool(transB)), N, _ptr(bs), _ptr(bz), bs.size, _ptr(c), cr, cc, float(alpha),
                          int(quant), float(y_scale) if quant else 1.0,
                          int(y_zero_point) if quant and y_zero_point is not None else 0, yt, _ptr(Y)), "qgemm")
    return Y


def matmul_integer_to_float(A, B, a_scale, b_scale, a_zero_point=None, b_zero_point=None, bias=None):
    """MatMulIntegerToFloat (ONNX Runtime contrib schemas).  A: uint8/int8
    (..., K), B: uint8/int8 (K, N); a_scale / a_zero_point: 1 entry or one
    per row of A (rows = all leading dimensions); b_scale / b_zero_point: 1
    or N entries; bias: N floats or None.  Returns fp32 (..., N)."""
    A = np.asarray(A)
    lead = A.shape[:-1]
    A2 = np.ascontiguousarray(A.reshape(-1, A.shape[-1]))
    B = np.ascontiguousarray(B)
    M, K = A2.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    at = U8 if A.dtype == np.uint8 else S8
    bt = U8 if B.dtype == np.uint8 else S8
    asc = np.ascontiguousarray(np.atleast_1d(a_scale), dtype=np.float32)
    bsc = np.ascontiguousarray(np.atleast_1d(b_scale), dtype=np.float32)
    az = None if a_zero_point is None else np.ascontiguousarray(np.atleast_1d(a_zero_point), dtype=np.int32)
    bz = None if b_zero_point is None else np.ascontiguousarray(np.atleast_1d(b_zero_point), dtype=np.int32)
    if asc.size not in (1, M) or (az is not None and az.size != asc.size):
        raise ValueError("a_scale / a_zero_point must have 1 entry or one per row of A")
    if bsc.size not in (1, N) or (bz is not None and bz.size != bsc.size):
        raise ValueError("b_scale / b_zero_point must have 1 or N entries")
    bi = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    Y = np.empty((M, N), np.float32)
    _check(lib().or_matmul_integer_to_float(_ptr(A2), at, M, K, _ptr(B), bt, N, _ptr(asc), _ptr(az), asc.size,
                                            _ptr(bsc), _ptr(bz), bsc.size, _ptr(bi), _ptr(Y)),
           "matmul_integer_to_float")
    return Y.reshape(*lead, N)


def dynamic_quantize_matmul(A, B, b_scale, b_zero_point=None, bias=None):
    """DynamicQuantizeMatMul (ONNX Runtime contrib schemas): fp32 A
    (..., K) quantized to uint8 per tensor with the same formula as the rows
    of the dynamic inner product (range widened to contain 0, scale =
    (max - min) / 255, zero point = saturate(rint(-min / scale))), then
    MatMulIntegerToFloat.  Returns {"Y", "uA", "a_scale", "a_zero_point"}."""
    A = np.ascontiguousarray(A, dtype=np.float32)
    uA, s, z = quantize_rows_u8(A.reshape(1, -1))
    uA = uA.reshape(A.shape)
    Y = matmul_integer_to_float(uA, B, s[0], b_scale, np.int32(z[0]), b_zero_point, bias)
    return {"Y": Y, "uA": uA, "a_scale": s[0], "a_zero_point": int(z[0])}


def _bcast_shapes(a, b):
    """Numpy-style broadcast of two shapes: (a_padded, b_padded, out) as int64
    arrays of one rank."""
    out = np.broadcast_shapes(a, b)
    r = max(len(out), 1)
    pad = lambda s: np.array((1,) * (r - len(s)) + tuple(s), dtype=np.int64)  # noqa: E731
    return pad(a), pad(b), pad(out), tuple(out)


def mul_integer(A, B, a_zero_point=0, b_zero_point=0):
    """MulInteger: int32 (A - a_zp) * (B - b_zp), Numpy-style broadcast."""
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    sa, sb, so, out = _bcast_shapes(A.shape, B.shape)
    C = np.empty(out, np.int32)
    _check(lib().or_mul_integer(_ptr(A), U8 if A.dtype == np.uint8 else S8, _ptr(sa), int(a_zero_point), _ptr(B),
                                U8 if B.dtype == np.uint8 else S8, _ptr(sb), int(b_zero_point), _ptr(so), len(so),
                                _ptr(C)), "mul_integer")
    return C


def qlinear_binary(op, A, a_scale, a_zero_point, B, b_scale, b_zero_point, c_scale, c_zero_point):
    """QLinearAdd (op "add") / QLinearMul (op "mul"); A, B, C of one 8-bit
    type, broadcast."""
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    if A.dtype != B.dtype:
        raise ValueError("A and B must have one type")
    sa, sb, so, out = _bcast_shapes(A.shape, B.shape)
    C = np.empty(out, A.dtype)
    _check(lib().or_qlinear_binary({"add": 0, "mul": 1}[op], _ptr(A), _ptr(sa), float(a_scale), int(a_zero_point),
                                   _ptr(B), _ptr(sb), float(b_scale), int(b_zero_point), float(c_scale),
                                   int(c_zero_point), _ptr(so), len(so), U8 if A.dtype == np.uint8 else S8, _ptr(C)),
           "qlinear_binary")
    return C


def qlinear_unary(op, X, x_scale, x_zero_point, y_scale, y_zero_point, alpha=0.01):
    """QLinearLeakyRelu (op "leaky_relu") / QLinearSigmoid (op "sigmoid")."""
    X = np.ascontiguousarray(X)
    Y = np.empty_like(X)
    _check(lib().or_qlinear_unary({"leaky_relu": 0, "sigmoid": 1}[op], _ptr(X), X.size,
                                  U8 if X.dtype == np.uint8 else S8, float(x_scale), int(x_zero_point), float(y_scale),
                                  int(y_zero_point), float(alpha), _ptr(Y)), "qlinear_unary")
    return Y


ELEMENTARY = {"exp": 0, "expm1": 1, "log1p": 2, "sigmoid": 3, "tanh": 4, "softplus": 5}


def elementary(name, x):
    """The oracle's fp32 exp / expm1 / log1p (argument in [0, 1]) / sigmoid /
    tanh / softplus, elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _check(lib().or_elementary(ELEMENTARY[name], _ptr(x), x.size, _ptr(y)), "elementary")
    return y


# The ONNX LSTM activation functions, in the order of the operator's list;
# the value is the index the oracle's C code takes.
LSTM_ACTIVATIONS = ["Relu", "Tanh", "Sigmoid", "Affine", "LeakyRelu", "ThresholdedRelu", "ScaledTanh", "HardSigmoid",
                    "Elu", "Softsign", "Softplus"]
# (alpha, beta) each function takes, with the default of the corresponding
# ONNX operator (None: the function takes no such attribute).  LeakyRelu's
# 0.01 is the one the DynamicQuantizeLSTM pages state; the others are the
# ONNX operators' own defaults, and ScaledTanh (whose operator names none)
# takes 1 and 1, which makes it Tanh.
LSTM_ACTIVATION_PARAMS = {"Relu": (None, None), "Tanh": (None, None), "Sigmoid": (None, None),
                          "Affine": (1.0, 0.0), "LeakyRelu": (0.01, None), "ThresholdedRelu": (1.0, None),
                          "ScaledTanh": (1.0, 1.0), "HardSigmoid": (0.2, 0.5), "Elu": (1.0, None),
                          "Softsign": (None, None), "Softplus": (None, None)}


def resolve_lstm_activations(activations, activation_alpha, activation_beta, D):
    """Per direction, the three (f, g, h) activations as (index, alpha, beta).

    activations: None (Sigmoid, Tanh, Tanh in each direction) or 3*D names.
    activation_alpha / activation_beta are "consumed in the order of
    activation functions": walking the list, each function that takes an
    alpha (beta) takes the next unused value, or its default once the list
    is exhausted."""
    if activations is None:
        activations = ["Sigmoid", "Tanh", "Tanh"] * D
    assert len(activations) == 3 * D, "activations needs 3 entries per direction"
    alphas = list(activation_alpha or [])
    betas = list(activation_beta or [])
    out = []
    for name in activations:
        da, db = LSTM_ACTIVATION_PARAMS[name]
        a = b = 0.0
        if da is not None:
            a = alphas.pop(0) if alphas else da
        if db is not None:
            b = betas.pop(0) if betas else db
        out.append((LSTM_ACTIVATIONS.index(name), float(a), float(b)))
    return [out[3 * d:3 * d + 3] for d in range(D)]


def lstm_cell(Gx, Gh, Wb, Rb, c_prev, P=None, clip=0.0, input_forget=False, acts=None):
    """One DynamicQuantizeLSTM cell update (iofc); P: peepholes (3H, iof) or
    None; clip <= 0: no clip; acts: the (f, g, h) activations as three
    (index, alpha, beta) or None for the defaults."""
    Gx = np.ascontiguousarray(Gx, dtype=np.float32)
    Gh = np.ascontiguousarray(Gh, dtype=np.float32)
    c_prev = np.ascontiguousarray(c_prev, dtype=np.float32)
    batch, H4 = Gx.shape
    H = H4 // 4
    Wb = None if Wb is None else np.ascontiguousarray(Wb, dtype=np.float32)
    Rb = None if Rb is None else np.ascontiguousarray(Rb, dtype=np.float32)
    P = None if P is None else np.ascontiguousarray(P, dtype=np.float32)
    ak = al = be = None
    if acts is not None:
        ak = np.array([a[0] for a in acts], np.int32)
        al = np.array([a[1] for a in acts], np.float32)
        be = np.array([a[2] for a in acts], np.float32)
    h = np.empty((batch, H), dtype=np.float32)
    c = np.empty((batch, H), dtype=np.float32)
    _check(lib().or_lstm_cell_ex(_ptr(Gx), _ptr(Gh), _ptr(Wb), _ptr(Rb), _ptr(P), float(clip), int(bool(input_forget)),
                                 _ptr(ak), _ptr(al), _ptr(be), _ptr(c_prev), _ptr(h), _ptr(c), batch, H), "lstm_cell")
    return h, c


def dyn_product_zp(A, B, scaleB, zeroB=None):
    """The dequantized product of fp32 A (rows quantized to uint8 as in the
    inner product) with 8-bit B (K x N, uint8 or int8) whose zero point is
    per column or per tensor: ((float)sum (uA - zA)(B - zB) * sA) * sB."""
    uA, sA, zA = quantize_rows_u8(A)
    B = np.ascontiguousarray(B)
    M, K = uA.shape
    N = B.shape[1]
    zb = None if zeroB is None else np.ascontiguousarray(np.atleast_1d(zeroB), dtype=np.int32)
    sB = np.ascontiguousarray(np.broadcast_to(np.asarray(scaleB, np.float32), (N,)))
    C = np.empty((M, N), np.float32)
    _check(lib().or_dyn_product_zp(_ptr(uA), _ptr(zA), _ptr(sA), _ptr(B), U8 if B.dtype == np.uint8 else S8, _ptr(zb),
                                   0 if zb is None else zb.size, _ptr(sB), M, N, K, _ptr(C)), "dyn_product_zp")
    return C


def _lstm_product(A, Wq, scale, zero_point):
    """Gx or Gh: the int8-B inner product when W is int8 without zero point,
    else the zero-point product (same arithmetic when the zero point is 0)."""
    if zero_point is None and Wq.dtype == np.int8:
        return dynamic_quantized_inner_product(A, iB=Wq, scaleB=scale)["C32"]
    return dyn_product_zp(A, Wq, scale, zero_point)


def lstm_projection(X, W, W_scale, W_zero_point=None):
    """Input projection of one direction: X (T, batch, I) quantized per row,
    times 8-bit W (I x 4H) with per-column scales (and zero points), no
    bias, fp32 out."""
    T, batch, I = X.shape
    return _lstm_product(X.reshape(T * batch, I), W, W_scale, W_zero_point).reshape(T, batch, -1)


def lstm_step(Gx_t, h_prev, c_prev, R, R_scale, Wb, Rb, R_zero_point=None, P=None, clip=0.0, input_forget=False,
              acts=None):
    """One recurrence step of one direction: quantize h_prev per row, take
    the dequantized product with 8-bit R, then the cell update."""
    Gh = _lstm_product(h_prev, R, R_scale, R_zero_point)
    return lstm_cell(Gx_t, Gh, Wb, Rb, c_prev, P, clip, input_forget, acts)


def dynamic_quantize_lstm(X, W, R, B, W_scale, R_scale, h0=None, c0=None, direction="forward", steps=None,
                          W_zero_point=None, R_zero_point=None, P=None, clip=0.0, input_forget=False,
                          sequence_lens=None, activations=None, activation_alpha=None, activation_beta=None):
    """DynamicQuantizeLSTM (ONNX Runtime contrib schema).  activations: None
    (the defaults) or 3 names per direction, with the alpha/beta attribute
    lists (see resolve_lstm_activations).  X (T, batch, I); W (D, I, 4H) and R (D, H, 4H) uint8 or
    int8 with zero points (D, 4H) / (D,) or None; scales (D, 4H); B (D, 8H)
    or None; P (D, 3H) or None; sequence_lens (batch,) or None.  A batch row
    with length L runs steps t = 0..L-1 (forward) or L-1..0 (reverse); Y is 0
    for t >= L and Y_h, Y_c hold the state after its last step.
    Returns Y (T, D, batch, H), Y_h, Y_c (D, batch, H).  steps (default T)
    limits how many steps each direction runs."""
    T, batch, I = X.shape
    D = W.shape[0]
    H = R.shape[1]
    dirs = {"forward": [0], "reverse": [1], "bidirectional": [0, 1]}[direction]
    assert len(dirs) == D
    S = T if steps is None else steps
    L = np.full(batch, T, np.int64) if sequence_lens is None else np.asarray(sequence_lens, np.int64)
    Y = np.zeros((T, D, batch, H), dtype=np.float32)
    Yh = np.zeros((D, batch, H), dtype=np.float32)
    Yc = np.zeros((D, batch, H), dtype=np.float32)
    zp = lambda z, d: None if z is None else np.asarray(z)[d]  # noqa: E731
    rows = np.arange(batch)
    acts = resolve_lstm_activations(activations, activation_alpha, activation_beta, D)
    for d, kind in enumerate(dirs):
        Gx = lstm_projection(X, W[d], W_scale[d], zp(W_zero_point, d))
        h = np.zeros((batch, H), np.float32) if h0 is None else np.array(h0[d], np.float32)
        c = np.zeros((batch, H), np.float32) if c0 is None else np.array(c0[d], np.float32)
        Wb = None if B is None else B[d, :4 * H]
        Rb = None if B is None else B[d, 4 * H:]
        Pd = None if P is None else P[d]
        for n in range(min(S, T)):
            t_b = np.where(kind == 0, n, L - 1 - n)
            active = n < L
            Gx_t = Gx[np.clip(t_b, 0, T - 1), rows]
            hn, cn = lstm_step(Gx_t, h, c, R[d], R_scale[d], Wb, Rb, zp(R_zero_point, d), Pd, clip, input_forget,
                               acts[d])
            h = np.where(active[:, None], hn, h)
            c = np.where(active[:, None], cn, c)
            for b in np.nonzero(active)[0]:
                Y[t_b[b], d, b] = h[b]
        Yh[d] = h
        Yc[d] = c
    return Y, Yh, Yc


def num_threads():
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else the CPUs this
    process may run on)."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.isdigit():
        return int(env)
    return len(os.sched_getaffinity(0))
