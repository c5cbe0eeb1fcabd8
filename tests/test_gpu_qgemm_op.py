"""QGemm (ONNX Runtime contrib schema) on the GPU vs the CPU oracle.

Bit-exact for quantized outputs (the integer sum, the fp32 rescale and the
division by y_scale are one fixed sequence on both sides) and exactly equal
for fp32 outputs.  Every case runs on the single-CTA and the CTA-pair
tensor-core kernels.
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


def run(orc, dev, A, a_scale, za, B, b_scale, zb=None, C=None, alpha=1.0, y_scale=None, yzp=0, ytype="u8",
        transA=False, transB=False, rows=None):
    M = A.shape[1] if transA else A.shape[0]
    N = B.shape[0] if transB else B.shape[1]
    if y_scale is None:
        Y = torch.empty(M, N, dtype=torch.float32, device=dev)
    else:
        Y = torch.empty(M, N, dtype=torch.uint8 if ytype == "u8" else torch.int8, device=dev)
    bs = np.atleast_1d(np.asarray(b_scale, np.float32))
    bz = None if zb is None else np.atleast_1d(np.asarray(zb)).astype(B.dtype)
    q.qgemm(_t(A, dev), a_scale, za, _t(B, dev), _t(bs, dev), Y, b_zero_point=None if bz is None else _t(bz, dev),
            C=None if C is None else _t(np.asarray(C, np.int32), dev), alpha=alpha, y_scale=y_scale, y_zero_point=yzp,
            transA=transA, transB=transB)
    q.sync_status()
    got = Y.cpu().numpy()
    if rows is not None:
        # rows of the output depend only on the same rows of A (and of C)
        A = A[:, rows] if transA else A[rows]
        if C is not None and np.asarray(C).ndim == 2 and np.asarray(C).shape[0] > 1:
            C = np.asarray(C)[rows]
        got = got[rows]
    ref = orc.qgemm(A, a_scale, za, B, bs, bz, C=C, alpha=alpha, y_scale=y_scale, y_zero_point=yzp, transA=transA,
                    transB=transB, ytype=ytype)
    assert got.dtype == ref.dtype
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} of {got.size} differ"
    return got


@pytest.mark.parametrize("transA,transB", [(False, False), (True, False), (False, True), (True, True)])
def test_worked_example(orc, dev, transA, transB):
    g = read_golden("qgemm_small_example.txt")
    M, K = map(int, g["M_K"])
    N = int(g["K_N"][1])
    A = np.array(g["A_u8"], np.int64).astype(np.uint8).reshape(M, K)
    B = np.array(g["B_s8"], np.int64).astype(np.int8).reshape(K, N)
    a = A.T.copy() if transA else A
    b = B.T.copy() if transB else B
    kw = dict(zb=np.array(g["b_zero_point"], np.int64), C=np.array([g["C_1xN"]], np.int32), alpha=float(g["alpha"][0]),
              transA=transA, transB=transB)
    y = run(orc, dev, a, float(g["a_scale"][0]), int(g["a_zero_point"][0]), b, np.array(g["b_scale"], np.float32),
            **kw)
    assert np.array_equal(y.ravel(), np.array(g["y_float"], np.float32))
    yq = run(orc, dev, a, float(g["a_scale"][0]), int(g["a_zero_point"][0]), b, np.array(g["b_scale"], np.float32),
             y_scale=float(g["y_scale"][0]), yzp=int(g["y_zero_point"][0]), **kw)
    assert np.array_equal(yq.ravel(), np.array(g["y_u8"], np.int64))


SHAPES = [(1, 1, 1), (3, 5, 7), (64, 70, 130), (129, 257, 200), (300, 520, 1000)]


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("atype,btype", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8")])
def test_ragged_shapes_and_types(orc, dev, M, K, N, atype, btype):
    w = workloads.qgemm(seed=M + K + N, M=M, K=K, N=N, atype=atype, btype=btype)
    yt = "u8" if atype == "u8" else "s8"
    run(orc, dev, w["A"], w["a_scale"], w["a_zero_point"], w["B"], w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"], ytype=yt)
    run(orc, dev, w["A"], w["a_scale"], w["a_zero_point"], w["B"], w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]))


@pytest.mark.parametrize("c_shape", [None, "MN", "1N", "N", "M1", "11"])
@pytest.mark.parametrize("per_column", [True, False])
def test_bias_shapes_and_parameter_kinds(orc, dev, c_shape, per_column):
    w = workloads.qgemm(seed=11, M=150, K=333, N=270, per_column=per_column, c_shape=c_shape)
    run(orc, dev, w["A"], w["a_scale"], w["a_zero_point"], w["B"], w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"])


@pytest.mark.parametrize("transA,transB", [(True, False), (False, True), (True, True)])
def test_transposed_operands(orc, dev, transA, transB):
    w = workloads.qgemm(seed=12, M=200, K=300, N=260, atype="s8", btype="u8")
    A = w["A"].T.copy() if transA else w["A"]
    B = w["B"].T.copy() if transB else w["B"]
    run(orc, dev, A, w["a_scale"], w["a_zero_point"], B, w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"], ytype="s8", transA=transA,
        transB=transB)


@pytest.mark.parametrize("transA,transB", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("atype,btype", [("u8", "s8"), ("s8", "u8")])
def test_tiled_transposing_centring(orc, dev, transA, transB, atype, btype):
    """Operands whose K is the slow index and whose other extent is a
    multiple of 16 are centred in 128 x 128 tiles turned by byte permutes:
    M = 80 and N = 272 leave partial tiles, K = 200 a partial K tile and
    the padding up to 256."""
    w = workloads.qgemm(seed=14, M=80, K=200, N=272, atype=atype, btype=btype)
    A = w["A"].T.copy() if transA else w["A"]
    B = w["B"].T.copy() if transB else w["B"]
    yt = "u8" if atype == "u8" else "s8"
    run(orc, dev, A, w["a_scale"], w["a_zero_point"], B, w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"], ytype=yt, transA=transA,
        transB=transB)
    run(orc, dev, A, w["a_scale"], w["a_zero_point"], B, w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), transA=transA, transB=transB)


def test_no_zero_point_and_unit_parameters(orc, dev):
    w = workloads.qgemm(seed=13, M=96, K=64, N=128)
    run(orc, dev, w["A"], 1.0, 0, w["B"], np.float32(1.0))


def test_worst_case_magnitudes(orc, dev):
    """|A - a_zero_point| = 255 and |B - b_zero_point| = 255 in every term,
    K = 8192: |acc| reaches 5.3e8, the centred products stay at 2^14."""
    M, K, N = 130, 8192, 260
    A = np.full((M, K), 255, np.uint8)
    A[1::2] = 0
    B = np.zeros((K, N), np.uint8)
    B[:, 1::2] = 255
    zb = np.where(np.arange(N) % 2 == 0, 255, 0).astype(np.uint8)
    y = run(orc, dev, A, 1.0, 0, B, np.ones(N, np.float32), zb)
    assert np.abs(y).max() == 255 * 255 * K
    run(orc, dev, A, 1.0, 255, B, np.full(N, 2.0 ** -20, np.float32), zb, y_scale=1.0, yzp=0)


@pytest.mark.parametrize("y_scale", [2.0, 0.5, 3.0, 0.1, 1e-30, 1e30, 3e38])
def test_requantization_ties(orc, dev, y_scale):
    """Unit scales make every rescaled sum an integer, so y_scale 2 puts half
    the quotients exactly on a tie (round half to even decides them); the
    other scales give exact, inexact, saturating, vanishing quotients and one
    whose reciprocal is not a normal number."""
    rng = np.random.default_rng(31)
    M, K, N = 300, 4, 520
    A = rng.integers(0, 16, (M, K)).astype(np.uint8)
    B = rng.integers(-8, 8, (K, N)).astype(np.int8)
    run(orc, dev, A, 1.0, 0, B, np.ones(N, np.float32), y_scale=y_scale, yzp=0, ytype="s8")


def test_mid_size_full(orc, dev):
    w = workloads.qgemm(seed=14, M=512, K=2048, N=1024)
    run(orc, dev, w["A"], w["a_scale"], w["a_zero_point"], w["B"], w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"])


def test_full_size_sampled_rows(orc, dev):
    """M=8192 K=4096 N=14336, u8 output: sampled rows against the oracle."""
    w = workloads.qgemm(seed=5)
    rows = np.array([0, 1, 255, 256, 4095, 4096, 8191])
    run(orc, dev, w["A"], w["a_scale"], w["a_zero_point"], w["B"], w["b_scale"], w["b_zero_point"], C=w["C"],
        alpha=float(w["alpha"]), y_scale=float(w["y_scale"]), yzp=w["y_zero_point"], rows=rows)


def test_rejects_bad_arguments(dev):
    A = torch.zeros(4, 8, dtype=torch.uint8, device=dev)
    B = torch.zeros(8, 3, dtype=torch.int8, device=dev)
    Y = torch.empty(4, 3, dtype=torch.float32, device=dev)
    with pytest.raises(q.I8QError):
        q.qgemm(A, 1.0, 0, B, torch.ones(2, device=dev), Y)              # b_scale neither 1 nor N entries
    with pytest.raises(q.I8QError):
        q.qgemm(A, 1.0, 300, B, torch.ones(1, device=dev), Y)            # a_zero_point out of range
    with pytest.raises(q.I8QError):
        q.qgemm(A, 1.0, 0, B, torch.ones(1, device=dev), Y,
                C=torch.zeros(2, 3, dtype=torch.int32, device=dev))      # C not broadcastable
    with pytest.raises(q.I8QError):
        q.qgemm(A, 1.0, 0, B, torch.ones(1, device=dev), Y, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
