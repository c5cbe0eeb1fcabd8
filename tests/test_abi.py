"""The C ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before launching
anything (these calls reach no CUDA API)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "i8q.h")


@pytest.fixture(scope="module")
def lib():
    from int8_quantized_gb300 import _lib, build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(i8q_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["i8q_qgemm_dyn_init", "i8q_qgemm_dyn_set_params", "i8q_qgemm_dyn_forward", "i8q_quantize_linear",
                 "i8q_dequantize_linear", "i8q_qlinearconv", "i8q_dq_lstm_forward"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from int8_quantized_gb300 import _lib
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in i8q.h but not exported"
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature in the binding"


def test_version(lib):
    assert b"sm_103a" in lib.i8q_version()


def _arr(vals, t=ctypes.c_int64):
    return (t * len(vals))(*vals)


def test_quantize_rejects_bad_axis_and_rank(lib):
    from int8_quantized_gb300 import _lib
    shape = _arr([2, 3, 4])
    rc = lib.i8q_quantize_linear(ctypes.c_void_p(16), shape, 3, 3, ctypes.c_void_p(16), ctypes.c_void_p(16), 4,
                                 _lib.U8, ctypes.c_void_p(16), None)
    assert rc == _lib.ERR_INVALID_ARG and b"axis" in lib.i8q_last_error()
    rc = lib.i8q_quantize_linear(ctypes.c_void_p(16), shape, 9, 0, None, None, 1, _lib.U8, None, None)
    assert rc == _lib.ERR_INVALID_ARG and b"rank" in lib.i8q_last_error()
    # per-axis length must equal dim[axis]
    rc = lib.i8q_quantize_linear(ctypes.c_void_p(16), shape, 3, 1, ctypes.c_void_p(16), ctypes.c_void_p(16), 4,
                                 _lib.U8, ctypes.c_void_p(16), None)
    assert rc == _lib.ERR_INVALID_ARG and b"dim[axis]" in lib.i8q_last_error()
    # per-tensor needs scalars
    rc = lib.i8q_quantize_linear(ctypes.c_void_p(16), shape, 3, _lib.NO_AXIS, ctypes.c_void_p(16),
                                 ctypes.c_void_p(16), 3, _lib.U8, ctypes.c_void_p(16), None)
    assert rc == _lib.ERR_INVALID_ARG and b"scalars" in lib.i8q_last_error()
    rc = lib.i8q_dequantize_linear(ctypes.c_void_p(16), _lib.F32, shape, 3, _lib.NO_AXIS, ctypes.c_void_p(16),
                                   ctypes.c_void_p(16), 1, ctypes.c_void_p(16), None)
    assert rc == _lib.ERR_INVALID_ARG


def test_qgemm_init_validation(lib):
    from int8_quantized_gb300 import _lib
    ctx = ctypes.c_void_p(None)
    assert lib.i8q_qgemm_dyn_init(ctypes.byref(ctx), 0, 8, 8, 0, 0, 0, 1, 1, 0, 0) == _lib.ERR_INVALID_ARG
    assert lib.i8q_qgemm_dyn_init(ctypes.byref(ctx), 4, 8, 70000, 0, 0, 0, 1, 1, 0, 0) == _lib.ERR_UNSUPPORTED
    # int8 B only when constant
    assert lib.i8q_qgemm_dyn_init(ctypes.byref(ctx), 4, 8, 16, _lib.F32, _lib.S8, _lib.F32, 0, 1, 0, 0) == \
        _lib.ERR_INVALID_ARG
    assert lib.i8q_qgemm_dyn_init(ctypes.byref(ctx), 4, 8, 16, _lib.S8, _lib.F32, _lib.F32, 1, 1, 0, 0) == \
        _lib.ERR_INVALID_ARG
    assert lib.i8q_qgemm_dyn_init(ctypes.byref(ctx), 4, 8, 16, _lib.F32, _lib.F32, _lib.F32, 1, 1, 9, 0) == \
        _lib.ERR_UNSUPPORTED
    assert ctx.value is None
    assert lib.i8q_qgemm_dyn_enabled(None) == 0
    assert lib.i8q_qgemm_dyn_info(None) is None
    assert lib.i8q_qgemm_dyn_external_buffer_size(None) == 0
    assert lib.i8q_qgemm_dyn_forward(None, None, None, None, None, None) == _lib.ERR_NOT_INITIALIZED
    assert lib.i8q_qgemm_dyn_set_params(None, None, None, None, None, None) == _lib.ERR_NOT_INITIALIZED
    lib.i8q_qgemm_dyn_clear(None)
    lib.i8q_qgemm_dyn_clear(ctypes.byref(ctx))


def test_qlinearconv_validation(lib):
    from int8_quantized_gb300 import _lib
    xs, ws = _arr([1, 4, 5, 5]), _arr([2, 3, 3, 3])  # C != w.shape[1] * group
    pads, strides, dil = _arr([1, 1, 1, 1]), _arr([1, 1]), _arr([1, 1])
    assert lib.i8q_qlinearconv_workspace_size(xs, ws, pads, strides, dil, 1) == 0
    rc = lib.i8q_qlinearconv(ctypes.c_void_p(16), _lib.U8, xs, 0.1, 0, ctypes.c_void_p(16), _lib.U8, ws,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 0.1, 0, None, pads, strides, dil, 1,
                             ctypes.c_void_p(16), _lib.U8, None, 0, None)
    assert rc == _lib.ERR_INVALID_ARG and b"group" in lib.i8q_last_error()
    ws2 = _arr([2, 4, 3, 3])
    rc = lib.i8q_qlinearconv(ctypes.c_void_p(16), _lib.U8, xs, 0.1, 300, ctypes.c_void_p(16), _lib.U8, ws2,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), 1, 0.1, 0, None, pads, strides, dil, 1,
                             ctypes.c_void_p(16), _lib.U8, None, 0, None)
    assert rc == _lib.ERR_INVALID_ARG and b"zero point" in lib.i8q_last_error()
    rc = lib.i8q_qlinearconv(ctypes.c_void_p(16), _lib.U8, xs, 0.1, 3, ctypes.c_void_p(16), _lib.U8, ws2,
                             ctypes.c_void_p(16), ctypes.c_void_p(16), 3, 0.1, 0, None, pads, strides, dil, 1,
                             ctypes.c_void_p(16), _lib.U8, None, 0, None)
    assert rc == _lib.ERR_INVALID_ARG and b"M entries" in lib.i8q_last_error()


def test_lstm_validation(lib):
    from int8_quantized_gb300 import _lib
    assert lib.i8q_dq_lstm_workspace_size(0, 1, 1, 1, 0) == 0
    assert lib.i8q_dq_lstm_workspace_size(2, 3, 8, 4, 2) > 0
    p = ctypes.c_void_p(256)
    rc = lib.i8q_dq_lstm_forward(p, 2, 3, 8, 4, 2, p, p, None, 3, p, p, None, 2, None, None, None, None, None, None,
                                 p, 1 << 20, None)
    assert rc == _lib.ERR_INVALID_ARG and b"W_scale" in lib.i8q_last_error()
    rc = lib.i8q_dq_lstm_forward(p, 2, 3, 8, 4, 2, p, p, None, 2, p, p, None, 2, None, None, None, None, None, None,
                                 p, 16, None)
    assert rc == _lib.ERR_INVALID_ARG and b"workspace" in lib.i8q_last_error()


def test_lstm_activation_validation(lib):
    """The activations attribute is checked on the host before anything
    runs: 3 entries per direction (or none), each one of the ONNX list."""
    from int8_quantized_gb300 import _lib
    p = ctypes.c_void_p(256)

    def ex(kinds, n):
        arr = (ctypes.c_int * max(1, len(kinds)))(*kinds)
        return lib.i8q_dq_lstm_forward_ex(p, 2, 3, 8, 4, 0, p, p, _lib.S8, p, None, 1, p, None, 1, None, None, None,
                                          None, None, 0.0, 0, arr, n, None, 0, None, 0, None, None, None, p,
                                          1 << 20, None)
    assert ex([2, 1], 2) == _lib.ERR_INVALID_ARG and b"3 entries" in lib.i8q_last_error()
    assert ex([2, 1, 11], 3) == _lib.ERR_INVALID_ARG and b"unknown activation" in lib.i8q_last_error()
    assert ex([2, 1, -1], 3) == _lib.ERR_INVALID_ARG


def test_lstm_state_codes_layout(lib):
    """The hook only computes addresses inside the workspace: the two
    parities are one block of D * batch code rows apart, and which = 0 / 1
    swap with the parity of T (step s reads parity (s + 1) % 2 and writes
    parity s % 2)."""
    from int8_quantized_gb300 import _lib
    ws = 1 << 20
    out = [ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_int64()]

    def codes(T, which):
        rc = lib.i8q_dq_lstm_state_codes(ctypes.c_void_p(ws), T, 3, 8, 40, _lib.LSTM_BIDIRECTIONAL, which,
                                         *[ctypes.byref(o) for o in out])
        assert rc == 0
        return out[0].value, out[1].value, out[3].value
    c0, s0, stride = codes(4, 0)
    c1, s1, _ = codes(4, 1)
    assert stride == 64 and abs(c1 - c0) == 2 * 3 * 64 * 2 and abs(s1 - s0) == 2 * 3 * 4
    assert c1 - c0 == 2 * 3 * 64 * 2                   # T even: the last step read parity 0, wrote parity 1
    d0, _, _ = codes(5, 0)
    d1, _, _ = codes(5, 1)
    assert d0 - d1 == 2 * 3 * 64 * 2                   # T odd: the other way round
    assert ws < min(c0, c1) < ws + lib.i8q_dq_lstm_workspace_size(4, 3, 8, 40, _lib.LSTM_BIDIRECTIONAL)
    assert lib.i8q_dq_lstm_state_codes(None, 4, 3, 8, 40, 2, 0, *[ctypes.byref(o) for o in out]) == \
        _lib.ERR_INVALID_ARG
    assert lib.i8q_dq_lstm_state_codes(ctypes.c_void_p(ws), 4, 3, 8, 40, 2, 2, *[ctypes.byref(o) for o in out]) == \
        _lib.ERR_INVALID_ARG


def test_wait_probe_validation(lib):
    from int8_quantized_gb300 import _lib
    assert lib.i8q_debug_wait_timeout(2, 3_000_000, None) == _lib.ERR_INVALID_ARG
    assert lib.i8q_debug_wait_timeout(0, 10, None) == _lib.ERR_INVALID_ARG


def test_qgemm_validation(lib):
    from int8_quantized_gb300 import _lib
    p = ctypes.c_void_p(256)
    assert lib.i8q_qgemm_workspace_size(0, 4, 4) == 0
    assert lib.i8q_qgemm_workspace_size(3, 5, 7) > 0

    def call(atype=_lib.U8, btype=_lib.S8, M=4, K=8, N=3, za=0, n_b=1, C=None, cr=0, cc=0, quant=0, yzp=0,
             ytype=_lib.U8, ws=1 << 20):
        return lib.i8q_qgemm(p, atype, 0, M, K, 0.1, za, p, btype, 0, N, p, None, n_b, C, cr, cc, 1.0, quant, 0.5, yzp,
                             ytype, p, p, ws, None)
    assert call(atype=_lib.F32) == _lib.ERR_INVALID_ARG and b"U8 or I8Q_S8" in lib.i8q_last_error()
    assert call(n_b=2) == _lib.ERR_INVALID_ARG and b"b_scale" in lib.i8q_last_error()
    assert call(za=256) == _lib.ERR_INVALID_ARG and b"a_zero_point" in lib.i8q_last_error()
    assert call(atype=_lib.S8, za=200) == _lib.ERR_INVALID_ARG
    assert call(C=p, cr=2, cc=3) == _lib.ERR_INVALID_ARG and b"broadcastable" in lib.i8q_last_error()
    assert call(quant=1, ytype=_lib.F32) == _lib.ERR_INVALID_ARG
    assert call(quant=1, ytype=_lib.S8, yzp=128) == _lib.ERR_INVALID_ARG
    assert call(ws=16) == _lib.ERR_INVALID_ARG and b"workspace" in lib.i8q_last_error()
    assert call(K=70000) == _lib.ERR_UNSUPPORTED


def test_matmul_integer_validation(lib):
    from int8_quantized_gb300 import _lib
    p = ctypes.c_void_p(256)
    assert lib.i8q_matmul_integer_workspace_size(3, 5, 7) == lib.i8q_qgemm_workspace_size(3, 5, 7)
    rc = lib.i8q_matmul_integer_to_float(p, _lib.U8, 4, 8, p, _lib.S8, 3, p, None, 2, p, None, 1, None, p, p, 1 << 20,
                                         None)
    assert rc == _lib.ERR_INVALID_ARG and b"one per row" in lib.i8q_last_error()
    rc = lib.i8q_matmul_integer_to_float(p, _lib.F32, 4, 8, p, _lib.S8, 3, p, None, 1, p, None, 1, None, p, p, 1 << 20,
                                         None)
    assert rc == _lib.ERR_INVALID_ARG
    rc = lib.i8q_dynamic_quantize_matmul(p, 4, 8, p, _lib.S8, 3, p, None, 3, None, p, None, None, p, 16, None)
    assert rc == _lib.ERR_INVALID_ARG and b"workspace" in lib.i8q_last_error()
    rc = lib.i8q_dynamic_quantize_matmul(p, 4, 8, p, _lib.S8, 3, p, None, 2, None, p, None, None, p, 1 << 20, None)
    assert rc == _lib.ERR_INVALID_ARG and b"b_scale" in lib.i8q_last_error()


def test_qlinear_elementwise_validation(lib):
    from int8_quantized_gb300 import _lib
    p = ctypes.c_void_p(256)
    s34, s54 = _arr([3, 4]), _arr([5, 4])
    rc = lib.i8q_qlinear_binary(0, p, s34, 2, 0.1, 0, p, s54, 2, 0.1, 0, 0.1, 0, _lib.U8, p, None)
    assert rc == _lib.ERR_INVALID_ARG and b"broadcastable" in lib.i8q_last_error()
    rc = lib.i8q_qlinear_binary(7, p, s34, 2, 0.1, 0, p, s34, 2, 0.1, 0, 0.1, 0, _lib.U8, p, None)
    assert rc == _lib.ERR_INVALID_ARG and b"op" in lib.i8q_last_error()
    rc = lib.i8q_qlinear_binary(1, p, s34, 2, 0.1, 0, p, s34, 2, 0.1, 0, 0.1, -1, _lib.U8, p, None)
    assert rc == _lib.ERR_INVALID_ARG and b"zero point" in lib.i8q_last_error()
    rc = lib.i8q_mul_integer(p, _lib.F32, s34, 2, 0, p, _lib.U8, s34, 2, 0, p, None)
    assert rc == _lib.ERR_INVALID_ARG
    rc = lib.i8q_qlinear_unary(1, p, 10, _lib.S8, 0.1, 0, 0.1, 200, 0.01, p, None)
    assert rc == _lib.ERR_INVALID_ARG and b"zero point" in lib.i8q_last_error()
    assert lib.i8q_qlinear_unary(0, None, 0, _lib.U8, 0.1, 0, 0.1, 0, 0.01, None, None) == _lib.OK
