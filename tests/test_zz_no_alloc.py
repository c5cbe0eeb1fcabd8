"""The allocation-free entry point i8q_qgemm_dyn_static, through the C ABI.

It serves callers that may not allocate device memory (code inside a host
application that owns all device memory through its own pool, or code that
cannot take cudaMalloc's possible synchronization).  Its result must match
the CPU oracle, and the context-based Forward, on the same inputs, on two
calls in a row: the second call reuses the static scratch array the first
one left behind.  The cases take both of its routes: the fused dp4a kernel
and the row kernel with the mma.sync core.
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


def _case(rng, M, N, K, typeA, typeC, dev):
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    if typeA == q.BF16:
        A = (A.view(np.uint32) & 0xFFFF0000).view(np.float32)   # exactly representable in bf16
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    sB = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = rng.normal(0, 0.02, N).astype(np.float32)
    At = torch.from_numpy(A).to(dev)
    if typeA == q.BF16:
        At = At.to(torch.bfloat16)
    ctype = torch.bfloat16 if typeC == q.BF16 else torch.float32
    return A, B, sB, bias, At, torch.empty(M, N, dtype=ctype, device=dev)


def _compare(got, ref, typeC):
    """fp32 within 1e-6 relative, bf16 within one ulp, of the oracle's
    output (ref: fp32 output, or bf16 bit patterns)."""
    if typeC == q.BF16:
        d = bf16_ulp_distance(got.cpu().view(torch.int16).numpy().view(np.uint16), ref)
        assert d.max() <= 1
    else:
        assert max_rel_err(got.cpu().numpy(), ref) <= 1e-6


# (M, N, K, typeA, typeC, activation): the first two take the fused dp4a
# kernel (Kp <= 8192 and at most 2^27 multiply-adds); the others the row
# kernel and the mma.sync core: K above 8192, and a product too large for
# the small kernel though its K is short.
CASES = [(300, 200, 1000, q.F32, q.F32, q.ACT_IDENTITY), (64, 128, 256, q.BF16, q.BF16, q.ACT_GELU),
         (64, 128, 9000, q.F32, q.F32, q.ACT_RELU), (64, 128, 9000, q.BF16, q.BF16, q.ACT_GELU),
         (512, 640, 1024, q.F32, q.BF16, q.ACT_IDENTITY)]


@pytest.mark.parametrize("M,N,K,tA,tC,act", CASES)
def test_static_entry_point_matches_oracle_twice(orc, dev, M, N, K, tA, tC, act):
    """Two calls in a row (the second reuses the array the first left
    behind), each against the CPU oracle, and against the context-based
    Forward on the same inputs."""
    lib = _lib.load()
    rng = np.random.default_rng(20 + K)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.i8q_qgemm_dyn_static_scratch_bytes(M, N, K) <= lib.i8q_qgemm_dyn_static_scratch_capacity()
    ref = None
    for call in range(2):
        A, B, sB, bias, At, C = _case(rng, M, N, K, tA, tC, dev)
        Bt, sBt, biast = (torch.from_numpy(v).to(dev) for v in (B, sB, bias))
        rc = lib.i8q_qgemm_dyn_static(M, N, K, tA, _ptr(At), _ptr(Bt), _ptr(sBt), _ptr(biast), act, tC, _ptr(C),
                                      stream)
        assert rc == 0, lib.i8q_last_error()
        q.sync_status()
        ref = orc.dynamic_quantized_inner_product(A, iB=B, scaleB=sB, bias=bias, act=act,
                                                  typeC="bf16" if tC == q.BF16 else "f32")
        _compare(C, ref["C"], tC)
        # the context-based Forward on the same inputs gives the same output
        ctx = q.QGemmDyn(M, N, K, tA, q.S8, tC, constB=True, bias=True, activation=act)
        ctx.set_params(Bt, sBt, biast)
        C2 = torch.empty_like(C)
        ctx.forward(At, C2)
        q.sync_status()
        assert torch.equal(C.view(torch.int16) if tC == q.BF16 else C, C2.view(torch.int16) if tC == q.BF16 else C2)
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
