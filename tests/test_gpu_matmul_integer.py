"""MatMulIntegerToFloat and DynamicQuantizeMatMul (ONNX Runtime contrib
schemas) on the GPU vs the CPU oracle.

fp32 outputs must be equal (the integer sum, the scale product, the multiply
and the bias add are the same fp32 operations on both sides); the per-tensor
quantization of DynamicQuantizeMatMul must give the same scale and zero point
bit for bit.  Every case runs on the single-CTA and the CTA-pair kernels.
"""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from conftest import read_golden
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["tc1", "tc2"], autouse=True)
def kernel(request, monkeypatch):
    monkeypatch.setenv("I8Q_FORCE_CORE", request.param)
    return request.param


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_mitf(orc, dev, A, B, a_scale, b_scale, az=None, bz=None, bias=None):
    A = np.asarray(A)
    Y = torch.empty(*A.shape[:-1], B.shape[1], dtype=torch.float32, device=dev)
    asc = np.atleast_1d(np.asarray(a_scale, np.float32))
    bsc = np.atleast_1d(np.asarray(b_scale, np.float32))
    azp = None if az is None else np.atleast_1d(np.asarray(az)).astype(A.dtype)
    bzp = None if bz is None else np.atleast_1d(np.asarray(bz)).astype(B.dtype)
    q.matmul_integer_to_float(_t(A, dev), _t(B, dev), _t(asc, dev), _t(bsc, dev), Y,
                              a_zero_point=None if azp is None else _t(azp, dev),
                              b_zero_point=None if bzp is None else _t(bzp, dev),
                              bias=None if bias is None else _t(np.asarray(bias, np.float32), dev))
    q.sync_status()
    ref = orc.matmul_integer_to_float(A, B, asc, bsc, azp, bzp, bias)
    got = Y.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} of {got.size} differ"
    return got


def test_worked_example(orc, dev):
    g = read_golden("matmul_integer_to_float_example.txt")
    A = np.array(g["A_u8"], np.int64).astype(np.uint8).reshape(2, 2)
    B = np.array(g["B_s8"], np.int64).astype(np.int8).reshape(2, 2)
    y = run_mitf(orc, dev, A, B, float(g["a_scale"][0]), np.array(g["b_scale"], np.float32), int(g["a_zero_point"][0]),
                 np.array(g["b_zero_point"], np.int64), np.array(g["bias"], np.float32))
    assert np.array_equal(y.ravel(), np.array(g["Y"], np.float32))


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (5, 17, 9), (70, 130, 260), (257, 300, 129)])
@pytest.mark.parametrize("atype,btype", [("u8", "s8"), ("s8", "u8"), ("u8", "u8"), ("s8", "s8")])
@pytest.mark.parametrize("a_rows", [False, True])
def test_types_shapes_and_granularity(orc, dev, M, K, N, atype, btype, a_rows):
    w = workloads.qgemm(seed=M * 3 + K + N, M=M, K=K, N=N, atype=atype, btype=btype)
    rng = np.random.default_rng(M + N)
    lo, hi = (0, 256) if atype == "u8" else (-128, 128)
    as_ = rng.uniform(0.01, 0.05, M).astype(np.float32) if a_rows else np.float32(w["a_scale"])
    az = rng.integers(lo, hi, M) if a_rows else w["a_zero_point"]
    bias = rng.normal(0, 0.5, N).astype(np.float32)
    run_mitf(orc, dev, w["A"], w["B"], as_, w["b_scale"], az, w["b_zero_point"], bias)
    run_mitf(orc, dev, w["A"], w["B"], as_, w["b_scale"][:1])  # no zero points, per-tensor B, no bias


def test_n_dimensional_A(orc, dev):
    rng = np.random.default_rng(31)
    A = rng.integers(0, 256, (3, 4, 50)).astype(np.uint8)
    B = rng.integers(-128, 128, (50, 70)).astype(np.int8)
    y = run_mitf(orc, dev, A, B, np.float32(0.03), rng.uniform(1e-3, 1e-2, 70).astype(np.float32), 120)
    assert y.shape == (3, 4, 70)


def test_worst_case_magnitudes(orc, dev):
    M, K, N = 64, 8192, 256
    A = np.full((M, K), 255, np.uint8)
    A[1::2] = 0
    B = np.where(np.arange(N) % 2 == 0, 0, 255).astype(np.uint8)[None, :].repeat(K, 0)
    bz = np.where(np.arange(N) % 2 == 0, 255, 0)
    y = run_mitf(orc, dev, A, B, np.float32(1.0), np.ones(N, np.float32), 0, bz)
    assert np.abs(y).max() == 255 * 255 * K


@pytest.mark.parametrize("M,K,N", [(1, 1, 1), (7, 33, 20), (130, 300, 270), (512, 1024, 1024)])
@pytest.mark.parametrize("btype", ["s8", "u8"])
def test_dynamic_quantize_matmul(orc, dev, M, K, N, btype):
    w = workloads.qgemm(seed=M + 2 * K + N, M=M, K=K, N=N, btype=btype)
    rng = np.random.default_rng(K)
    A = rng.normal(0, 2, (M, K)).astype(np.float32)
    bias = rng.normal(0, 0.1, N).astype(np.float32)
    Y = torch.empty(M, N, dtype=torch.float32, device=dev)
    s_out = torch.empty(1, dtype=torch.float32, device=dev)
    z_out = torch.empty(1, dtype=torch.uint8, device=dev)
    q.dynamic_quantize_matmul(_t(A, dev), _t(w["B"], dev), _t(w["b_scale"], dev), Y,
                              b_zero_point=_t(w["b_zero_point"], dev), bias=_t(bias, dev), a_scale_out=s_out,
                              a_zero_point_out=z_out)
    q.sync_status()
    ref = orc.dynamic_quantize_matmul(A, w["B"], w["b_scale"], w["b_zero_point"], bias)
    assert s_out.cpu().numpy()[0] == ref["a_scale"] and int(z_out.cpu().numpy()[0]) == ref["a_zero_point"]
    got = Y.cpu().numpy()
    assert np.array_equal(got, ref["Y"]), f"{np.count_nonzero(got != ref['Y'])} of {got.size} differ"


def test_dynamic_quantize_matmul_degenerate_and_one_sided(orc, dev):
    """An all-zero A (scale 1, zero point 0), an all-positive A (zero point 0)
    and an all-negative A (zero point 255)."""
    rng = np.random.default_rng(5)
    B = rng.integers(-128, 128, (40, 30)).astype(np.int8)
    bs = rng.uniform(1e-3, 1e-2, 30).astype(np.float32)
    for A in (np.zeros((6, 40), np.float32), np.abs(rng.normal(0, 1, (6, 40))).astype(np.float32),
              -np.abs(rng.normal(0, 1, (6, 40))).astype(np.float32)):
        Y = torch.empty(6, 30, dtype=torch.float32, device=dev)
        q.dynamic_quantize_matmul(_t(A, dev), _t(B, dev), _t(bs, dev), Y)
        q.sync_status()
        ref = orc.dynamic_quantize_matmul(A, B, bs)
        assert np.array_equal(Y.cpu().numpy(), ref["Y"])


@pytest.mark.parametrize("scale", [1.0, 0.5, 2.0])
def test_dynamic_quantize_matmul_quantization_ties(orc, dev, scale):
    """A spanning exactly [0, 255 * scale] gives the scale `scale` and zero
    point 0, and inputs at (j + 1/2) * scale put every quotient on a tie
    (round half to even decides), others just beside one."""
    rng = np.random.default_rng(int(scale * 10))
    M, K, N = 40, 96, 48
    j = rng.integers(0, 255, (M, K)).astype(np.float32)
    A = ((j + 0.5) * np.float32(scale)).astype(np.float32)
    A[1::3] = np.nextafter(A[1::3], np.float32(0))
    A[0, 0], A[0, 1] = 0.0, np.float32(255 * scale)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    bs = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    Y = torch.empty(M, N, dtype=torch.float32, device=dev)
    q.dynamic_quantize_matmul(_t(A, dev), _t(B, dev), _t(bs, dev), Y)
    q.sync_status()
    ref = orc.dynamic_quantize_matmul(A, B, bs)
    assert ref["a_scale"] == np.float32(scale) and ref["a_zero_point"] == 0
    assert np.array_equal(Y.cpu().numpy(), ref["Y"])


def test_dynamic_quantize_matmul_full_size_sampled(orc, dev):
    """M=8192 K=4096 N=14336: the per-tensor parameters, and sampled output
    rows recomputed by the oracle from those rows of A with the same
    parameters."""
    w = workloads.qgemm(seed=5, btype="s8")
    A = workloads.large_gemm(seed=2, M=8192, K=4096, N=16)["A_bf16"]
    A = (A.astype(np.uint32) << 16).view(np.float32)
    Y = torch.empty(8192, 14336, dtype=torch.float32, device=dev)
    s_out = torch.empty(1, dtype=torch.float32, device=dev)
    z_out = torch.empty(1, dtype=torch.uint8, device=dev)
    q.dynamic_quantize_matmul(_t(A, dev), _t(w["B"], dev), _t(w["b_scale"], dev), Y,
                              b_zero_point=_t(w["b_zero_point"], dev), a_scale_out=s_out, a_zero_point_out=z_out)
    q.sync_status()
    uA, s, z = orc.quantize_rows_u8(A.reshape(1, -1))
    assert s_out.cpu().numpy()[0] == s[0] and int(z_out.cpu().numpy()[0]) == z[0]
    rows = np.array([0, 1, 4095, 8191])
    ref = orc.matmul_integer_to_float(uA.reshape(A.shape)[rows], w["B"], s[0], w["b_scale"], np.int32(z[0]),
                                      w["b_zero_point"])
    assert np.array_equal(Y.cpu().numpy()[rows], ref)
