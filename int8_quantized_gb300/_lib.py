"""ctypes declarations of libi8q.so (include/i8q.h).  Loading fails loudly
when the library has not been built: there is no other implementation."""
import ctypes
import os

from . import build as _build

F32, BF16, S8, U8, S32 = 0, 1, 2, 3, 4
ACT_IDENTITY, ACT_RELU, ACT_GELU = 0, 1, 2
NO_AXIS = -(2 ** 31)
LSTM_FORWARD, LSTM_REVERSE, LSTM_BIDIRECTIONAL = 0, 1, 2
# I8Q_LSTM_ACT_*: the ONNX LSTM activation functions, in the operator's order
LSTM_ACTIVATIONS = ["Relu", "Tanh", "Sigmoid", "Affine", "LeakyRelu", "ThresholdedRelu", "ScaledTanh", "HardSigmoid",
                    "Elu", "Softsign", "Softplus"]

OK = 0
ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NOT_INITIALIZED, ERR_ALLOC, ERR_CUDA, ERR_DEVICE_TIMEOUT = -1, -2, -3, -4, -5, -6

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f = ctypes.c_float

# name -> (restype, argtypes); mirrors include/i8q.h
SIGNATURES = {
    "i8q_last_error": (ctypes.c_char_p, []),
    "i8q_version": (ctypes.c_char_p, []),
    "i8q_qgemm_dyn_init": (_i, [ctypes.POINTER(_p), _sz, _sz, _sz, _i, _i, _i, _i, _i, _i, _i]),
    "i8q_qgemm_dyn_enabled": (_i, [_p]),
    "i8q_qgemm_dyn_internal_buffer_size": (_sz, [_p]),
    "i8q_qgemm_dyn_external_buffer_size": (_sz, [_p]),
    "i8q_qgemm_dyn_info": (ctypes.c_char_p, [_p]),
    "i8q_qgemm_dyn_set_params": (_i, [_p, _p, _p, _p, _p, _p]),
    "i8q_qgemm_dyn_forward": (_i, [_p, _p, _p, _p, _p, _p]),
    "i8q_qgemm_dyn_forward_host": (_i, [_p, _p, _p, _p]),
    "i8q_qgemm_dyn_forward_s32": (_i, [_p, _p, _p, _p, _p, _p]),
    "i8q_qgemm_dyn_buf_views": (_i, [_p, _p, ctypes.POINTER(_p), ctypes.POINTER(_sz), ctypes.POINTER(_p),
                                     ctypes.POINTER(_p)]),
    "i8q_qgemm_dyn_weight_views": (_i, [_p, _p, ctypes.POINTER(_p), ctypes.POINTER(_p), ctypes.POINTER(_sz),
                                        ctypes.POINTER(_p), ctypes.POINTER(_p)]),
    "i8q_qgemm_dyn_clear": (None, [ctypes.POINTER(_p)]),
    "i8q_quantize_linear": (_i, [_p, _p, _i, _i, _p, _p, _sz, _i, _p, _p]),
    "i8q_dequantize_linear": (_i, [_p, _i, _p, _i, _i, _p, _p, _sz, _p, _p]),
    "i8q_qlinearconv": (_i, [_p, _i, _p, _f, _i, _p, _i, _p, _p, _p, _sz, _f, _i, _p, _p, _p, _p, _i64, _p, _i, _p,
                             _sz, _p]),
    "i8q_qlinearconv_workspace_size": (_sz, [_p, _p, _p, _p, _p, _i64]),
    "i8q_qgemm": (_i, [_p, _i, _i, _i64, _i64, _f, _i, _p, _i, _i, _i64, _p, _p, _sz, _p, _i64, _i64, _f, _i, _f,
                       _i, _i, _p, _p, _sz, _p]),
    "i8q_qgemm_workspace_size": (_sz, [_i64, _i64, _i64]),
    "i8q_matmul_integer_to_float": (_i, [_p, _i, _i64, _i64, _p, _i, _i64, _p, _p, _sz, _p, _p, _sz, _p, _p, _p, _sz,
                                         _p]),
    "i8q_dynamic_quantize_matmul": (_i, [_p, _i64, _i64, _p, _i, _i64, _p, _p, _sz, _p, _p, _p, _p, _p, _sz, _p]),
    "i8q_matmul_integer_workspace_size": (_sz, [_i64, _i64, _i64]),
    "i8q_dq_lstm_forward_ex": (_i, [_p, _i64, _i64, _i64, _i64, _i, _p, _p, _i, _p, _p, _sz, _p, _p, _sz, _p, _p, _p,
                                    _p, _p, _f, _i, _p, _sz, _p, _sz, _p, _sz, _p, _p, _p, _p, _sz, _p]),
    "i8q_dq_lstm_state_codes": (_i, [_p, _i64, _i64, _i64, _i64, _i, _i, ctypes.POINTER(_p), ctypes.POINTER(_p),
                                     ctypes.POINTER(_p), ctypes.POINTER(_i64)]),
    "i8q_qlinear_binary": (_i, [_i, _p, _p, _i, _f, _i, _p, _p, _i, _f, _i, _f, _i, _i, _p, _p]),
    "i8q_mul_integer": (_i, [_p, _i, _p, _i, _i, _p, _i, _p, _i, _i, _p, _p]),
    "i8q_qlinear_unary": (_i, [_i, _p, _i64, _i, _f, _i, _f, _i, _f, _p, _p]),
    "i8q_dq_lstm_forward": (_i, [_p, _i64, _i64, _i64, _i64, _i, _p, _p, _p, _sz, _p, _p, _p, _sz, _p, _p, _p, _p,
                                 _p, _p, _p, _sz, _p]),
    "i8q_dq_lstm_workspace_size": (_sz, [_i64, _i64, _i64, _i64, _i]),
    "i8q_sync_status": (_i, [_p]),
    "i8q_debug_wait_timeout": (_i, [_i, _i64, _p]),
    "i8q_profile_enable": (_i, [_i]),
    "i8q_profile_collect": (_i, []),
    "i8q_profile_entry": (_i, [_i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_longlong),
                               ctypes.POINTER(ctypes.c_double)]),
    "i8q_measure_int8_mma_peak": (_i, [_i64, _p, ctypes.POINTER(ctypes.c_double)]),
    "i8q_qgemm_dyn_static": (_i, [_sz, _sz, _sz, _i, _p, _p, _p, _p, _i, _i, _p, _p]),
    "i8q_qgemm_dyn_static_scratch_bytes": (_sz, [_sz, _sz, _sz]),
    "i8q_qgemm_dyn_static_scratch_capacity": (_sz, []),
}

_lib = None


def lib_path():
    return _build.LIB


def load(path=None):
    """Load libi8q.so and declare every exported signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libi8q.so is not built ({p}); run int8_quantized_gb300.build.build() first")
    l = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(l, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = l
    return l


def last_error():
    return load().i8q_last_error().decode(errors="replace")


class I8QError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where} failed ({code}): {last_error()}")


def check(rc, where):
    if rc != OK:
        raise I8QError(rc, where)
    return rc
