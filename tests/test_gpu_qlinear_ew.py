"""MulInteger, QLinearAdd, QLinearMul, QLinearLeakyRelu and QLinearSigmoid
on the GPU vs the CPU oracle: bit-exact, except QLinearSigmoid, whose expf
may differ by an ulp between the libraries and so move a code that lies at
a rounding boundary (allowed there only, by one step)."""

import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from conftest import read_golden

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["table", "arithmetic"], autouse=True)
def binary_path(request, monkeypatch):
    """Large QLinearAdd / QLinearMul run through the 256 x 256 code table,
    and with the per-element arithmetic."""
    if request.param == "arithmetic":
        monkeypatch.setenv("I8Q_QEW_NO_TABLE", "1")
    return request.param


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def binary(orc, dev, op, A, sa, za, B, sb, zb, sc, zc):
    out = np.broadcast_shapes(A.shape, B.shape)
    C = torch.empty(out, dtype=torch.uint8 if A.dtype == np.uint8 else torch.int8, device=dev)
    q.qlinear_binary(op, _t(A, dev), sa, za, _t(B, dev), sb, zb, sc, zc, C)
    q.sync_status()
    ref = orc.qlinear_binary(op, A, sa, za, B, sb, zb, sc, zc)
    got = C.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} of {got.size} differ"
    return got


def test_worked_cases(orc, dev):
    g = read_golden("qlinear_elementwise_cases.txt")
    A = np.array(g["A"], np.int64).astype(np.uint8).reshape(2, 2)
    B = np.array(g["B"], np.int64).astype(np.uint8)
    y = binary(orc, dev, "add", A, 0.5, 10, B, 0.25, 100, 1.0, 128)
    assert np.array_equal(y.ravel(), np.array(g["add"], np.int64))
    y = binary(orc, dev, "mul", A, 0.5, 10, B, 0.25, 100, 2.0, 128)
    assert np.array_equal(y.ravel(), np.array(g["mul"], np.int64))
    C = torch.empty(2, 2, dtype=torch.int32, device=dev)
    q.mul_integer(_t(A, dev), 10, _t(B, dev), 100, C)
    assert np.array_equal(C.cpu().numpy().ravel(), np.array(g["mul_integer"], np.int64))
    X = np.array(g["leaky_x"], np.int64).astype(np.uint8)
    Y = torch.empty(8, dtype=torch.uint8, device=dev)
    q.qlinear_unary("leaky_relu", _t(X, dev), 0.5, 128, 0.5, 128, Y, alpha=0.25)
    assert np.array_equal(Y.cpu().numpy(), np.array(g["leaky_y"], np.int64))


@pytest.mark.parametrize("qt", ["u8", "s8"])
@pytest.mark.parametrize("op", ["add", "mul"])
@pytest.mark.parametrize("n", [1, 15, 16, 17, 1000, 65543])
def test_same_shape(orc, dev, qt, op, n):
    rng = np.random.default_rng(n)
    lo, hi, dt = (0, 256, np.uint8) if qt == "u8" else (-128, 128, np.int8)
    A = rng.integers(lo, hi, n).astype(dt)
    B = rng.integers(lo, hi, n).astype(dt)
    za, zb, zc = (int(v) for v in rng.integers(lo, hi, 3))
    binary(orc, dev, op, A, 0.0371, za, B, 0.0213, zb, 0.0457 if op == "add" else 0.31, zc)


BCAST = [((4, 5, 64), (64,)), ((4, 5, 64), (5, 64)), ((3, 1, 7), (1, 4, 1)), ((2, 3, 16), ()), ((), (9, 33)),
         ((8, 1), (8, 32)), ((1, 48), (6, 48)), ((2, 1, 3, 1), (1, 5, 1, 7))]


@pytest.mark.parametrize("sa,sb", BCAST)
def test_broadcasting(orc, dev, sa, sb):
    rng = np.random.default_rng(len(sa) * 10 + len(sb))
    A = rng.integers(0, 256, sa).astype(np.uint8)
    B = rng.integers(0, 256, sb).astype(np.uint8)
    for op in ("add", "mul"):
        binary(orc, dev, op, A, 0.05, 100, B, 0.02, 31, 0.09 if op == "add" else 0.4, 127)
    C = torch.empty(np.broadcast_shapes(sa, sb), dtype=torch.int32, device=dev)
    q.mul_integer(_t(A, dev), 100, _t(B, dev), 31, C)
    q.sync_status()
    assert np.array_equal(C.cpu().numpy(), orc.mul_integer(A, B, 100, 31))


def test_mul_integer_mixed_types_and_unaligned(orc, dev):
    rng = np.random.default_rng(3)
    A = rng.integers(-128, 128, 1001).astype(np.int8)
    B = rng.integers(0, 256, 1001).astype(np.uint8)
    Ad = torch.empty(1002, dtype=torch.int8, device=dev)[1:]
    Ad.copy_(_t(A, dev))
    C = torch.empty(1001, dtype=torch.int32, device=dev)
    q.mul_integer(Ad, -5, _t(B, dev), 200, C)
    q.sync_status()
    assert np.array_equal(C.cpu().numpy(), orc.mul_integer(A, B, -5, 200))


def test_large_same_shape(orc, dev):
    rng = np.random.default_rng(4)
    A = rng.integers(0, 256, (4, 1024, 4096)).astype(np.uint8)
    B = rng.integers(0, 256, (4, 1024, 4096)).astype(np.uint8)
    binary(orc, dev, "add", A, 0.02, 128, B, 0.03, 120, 0.04, 125)
    binary(orc, dev, "mul", A, 0.02, 128, B, 0.03, 120, 0.05, 125)


def test_table_cache_hits_and_overflow(orc, dev, monkeypatch):
    """The code tables kept across calls: the same parameters twice (the
    second call reuses the first call's table), from a second stream, and
    more distinct parameter sets than the kept slots (the rest compute their
    table inside the kernel); every result against the oracle."""
    rng = np.random.default_rng(21)
    A = rng.integers(0, 256, (1 << 20,)).astype(np.uint8)
    B = rng.integers(0, 256, (1 << 20,)).astype(np.uint8)
    for k in range(20):
        cs = 0.04 + 0.001 * k
        binary(orc, dev, "add", A, 0.02, 128, B, 0.03, 120, cs, 125)
        if k % 7 == 0:
            binary(orc, dev, "add", A, 0.02, 128, B, 0.03, 120, cs, 125)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        binary(orc, dev, "mul", A, 0.02, 128, B, 0.03, 120, 0.041, 125)
    binary(orc, dev, "mul", A, 0.02, 128, B, 0.03, 120, 0.041, 125)
    monkeypatch.setenv("I8Q_QEW_NO_TABLE_CACHE", "1")
    binary(orc, dev, "add", A, 0.02, 128, B, 0.03, 120, 0.04, 125)


@pytest.mark.parametrize("qt", ["u8", "s8"])
@pytest.mark.parametrize("bshape", [(), (4096,), (1024, 4096)])
def test_large_broadcast(orc, dev, qt, bshape):
    """2^24 outputs: B a single value, a repeating row, or a repeating
    matrix; both operand types."""
    rng = np.random.default_rng(len(bshape) + 10 * (qt == "s8"))
    lo, hi, dt = (0, 256, np.uint8) if qt == "u8" else (-128, 128, np.int8)
    A = rng.integers(lo, hi, (4, 1024, 4096)).astype(dt)
    B = rng.integers(lo, hi, bshape).astype(dt)
    for op in ("add", "mul"):
        binary(orc, dev, op, A, 0.021, int(rng.integers(lo, hi)), B, 0.033, int(rng.integers(lo, hi)),
               0.05 if op == "add" else 0.3, int(rng.integers(lo, hi)))


@pytest.mark.parametrize("qt", ["u8", "s8"])
def test_leaky_relu_every_code(orc, dev, qt):
    lo, hi, dt = (0, 256, np.uint8) if qt == "u8" else (-128, 128, np.int8)
    X = np.arange(lo, hi).astype(dt)
    for zx, zy, alpha in ((lo + 90, lo + 10, 0.01), (lo + 200, lo + 255, 0.7)):
        Y = torch.empty(256, dtype=torch.uint8 if qt == "u8" else torch.int8, device=dev)
        q.qlinear_unary("leaky_relu", _t(X, dev), 0.0437, zx, 0.0311, zy, Y, alpha=alpha)
        q.sync_status()
        assert np.array_equal(Y.cpu().numpy(), orc.qlinear_unary("leaky_relu", X, 0.0437, zx, 0.0311, zy, alpha))


@pytest.mark.parametrize("qt", ["u8", "s8"])
@pytest.mark.parametrize("xs,ys", [(0.061, 1.0 / 255), (0.0123, 1.0 / 256), (0.5, 0.25), (0.002, 1e-3)])
def test_sigmoid_every_code(orc, dev, qt, xs, ys):
    """Every code, bit for bit: both sides use the same fixed-sequence fp32
    sigmoid, so even values at a rounding boundary take the same code."""
    lo, hi, dt = (0, 256, np.uint8) if qt == "u8" else (-128, 128, np.int8)
    X = np.arange(lo, hi).astype(dt)
    zx, zy = lo + 120, lo
    Y = torch.empty(256, dtype=torch.uint8 if qt == "u8" else torch.int8, device=dev)
    q.qlinear_unary("sigmoid", _t(X, dev), xs, zx, ys, zy, Y)
    q.sync_status()
    assert np.array_equal(Y.cpu().numpy(), orc.qlinear_unary("sigmoid", X, xs, zx, ys, zy))


def test_unary_large_and_unaligned(orc, dev):
    rng = np.random.default_rng(6)
    X = rng.integers(0, 256, 3 * 1024 * 1024 + 7).astype(np.uint8)
    Xd = torch.empty(X.size + 1, dtype=torch.uint8, device=dev)[1:]
    Xd.copy_(_t(X, dev))
    Y = torch.empty(X.size, dtype=torch.uint8, device=dev)
    q.qlinear_unary("leaky_relu", Xd, 0.02, 128, 0.015, 100, Y, alpha=0.1)
    q.sync_status()
    assert np.array_equal(Y.cpu().numpy(), orc.qlinear_unary("leaky_relu", X, 0.02, 128, 0.015, 100, 0.1))
    Y2 = torch.empty(X.size, dtype=torch.uint8, device=dev)
    q.qlinear_unary("leaky_relu", _t(X, dev), 0.02, 128, 0.015, 100, Y2, alpha=0.1)
    assert torch.equal(Y, Y2)


def test_rejects_bad_arguments(dev):
    A = torch.zeros(3, 4, dtype=torch.uint8, device=dev)
    B = torch.zeros(5, 4, dtype=torch.uint8, device=dev)
    C = torch.empty(3, 4, dtype=torch.uint8, device=dev)
    with pytest.raises(q.I8QError):
        q.qlinear_binary("add", A, 0.1, 0, B, 0.1, 0, 0.1, 0, C)     # not broadcastable
    with pytest.raises(q.I8QError):
        q.qlinear_binary("add", A, 0.1, 300, A, 0.1, 0, 0.1, 0, C)   # zero point out of range
    with pytest.raises(q.I8QError):
        q.qlinear_unary("sigmoid", A, 0.1, 0, 0.1, -1, C)            # zero point out of range
