"""The allocation-free entry point i8q_qgemm_dyn_static, through the C ABI.

It serves callers that may not allocate device memory (code inside a host
application that owns all device memory through its own pool, or code that
cannot take cudaMalloc's possible synchronization).  Its result must match
the context-based Forward on the same inputs, on two calls in a row: the
second call reuses the static scratch array the first one left behind.
This file sorts last so a run that stops at the first failure has run every
other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from conftest import bf16_ulp_distance, max_rel_err
from int8_quantized_gb300 import _lib

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(rng, M, N, K, typeA, typeC, act, dev):
    A = torch.from_numpy(rng.normal(0, 1, (M, K)).astype(np.float32)).to(dev)
    if typeA == q.BF16:
        A = A.to(torch.bfloat16)
    B = torch.from_numpy(rng.integers(-128, 128, (K, N)).astype(np.int8)).to(dev)
    sB = torch.from_numpy(rng.uniform(1e-3, 1e-2, N).astype(np.float32)).to(dev)
    bias = torch.from_numpy(rng.normal(0, 0.02, N).astype(np.float32)).to(dev)
    ctype = torch.bfloat16 if typeC == q.BF16 else torch.float32
    return A, B, sB, bias, torch.empty(M, N, dtype=ctype, device=dev), torch.empty(M, N, dtype=ctype, device=dev)


def _compare(got, ref, typeC):
    if typeC == q.BF16:
        d = bf16_ulp_distance(got.cpu().view(torch.int16).numpy().view(np.uint16),
                              ref.cpu().view(torch.int16).numpy().view(np.uint16))
        assert d.max() <= 1
    else:
        assert max_rel_err(got.cpu().numpy(), ref.cpu().numpy()) <= 1e-6


def test_static_entry_point_matches_forward_twice(dev):
    lib = _lib.load()
    rng = np.random.default_rng(20)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [(300, 200, 1000, q.F32, q.F32, q.ACT_IDENTITY), (64, 128, 256, q.BF16, q.BF16, q.ACT_GELU)]
    for M, N, K, tA, tC, act in cases:
        A, B, sB, bias, C_static, C_ref = _case(rng, M, N, K, tA, tC, act, dev)
        assert lib.i8q_qgemm_dyn_static_scratch_bytes(M, N, K) <= lib.i8q_qgemm_dyn_static_scratch_capacity()
        rc = lib.i8q_qgemm_dyn_static(M, N, K, tA, _ptr(A), _ptr(B), _ptr(sB), _ptr(bias), act, tC, _ptr(C_static),
                                      stream)
        assert rc == 0, lib.i8q_last_error()
        ctx = q.QGemmDyn(M, N, K, tA, q.S8, tC, constB=True, bias=True, activation=act)
        ctx.set_params(B, sB, bias)
        ctx.forward(A, C_ref)
        q.sync_status()
        _compare(C_static, C_ref, tC)
        ctx.clear()


def test_static_entry_point_rejects_oversize(dev):
    lib = _lib.load()
    cap = lib.i8q_qgemm_dyn_static_scratch_capacity()
    assert cap == 32 << 20
    M = N = 8192
    K = 4096
    assert lib.i8q_qgemm_dyn_static_scratch_bytes(M, N, K) > cap
    p = ctypes.c_void_p(256)
    rc = lib.i8q_qgemm_dyn_static(M, N, K, q.F32, p, p, p, None, q.ACT_IDENTITY, q.F32, p, None)
    assert rc == _lib.ERR_UNSUPPORTED
    assert b"static array" in lib.i8q_last_error()
