"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something the pages or the mathematics
fix: the worked examples the QLinearConv page prints, hand-worked closed
forms of QuantizeLinear/DequantizeLinear, lossless special cases whose exact
result is a textbook fp64 product, error bounds, invariants and library
routines.  The choice is meant to catch a dropped term, a wrong sign or
index, or a transposed operand anywhere in the oracle.
"""
import math
import zlib
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden, read_golden_rows
from int8_quantized_gb300 import workloads


def _qdt(t):
    return np.uint8 if t == "u8" else np.int8


# ----------------------------------------------------------------------------
# QLinearConv: the two printed examples, bit for bit
# ----------------------------------------------------------------------------

def _run_conv_golden(orc, name, xdt, wdt, xshape, wshape):
    g = read_golden(name)
    x = np.array([int(v) for v in g["x"]], dtype=xdt).reshape(xshape)
    w = np.array([int(v) for v in g["w"]], dtype=wdt).reshape(wshape)
    y = orc.qlinearconv(x, np.float32(g["x_scale"][0]), int(g["x_zero_point"][0]), w,
                        np.array([float(g["w_scale"][0])], np.float32),
                        np.array([int(g["w_zero_point"][0])]),
                        np.float32(g["y_scale"][0]), int(g["y_zero_point"][0]))
    expect = np.array([int(v) for v in g["y"]], dtype=xdt)
    return y.reshape(-1), expect


def test_qlinearconv_printed_uint8_example(orc):
    y, expect = _run_conv_golden(orc, "qlinearconv_u8_7x7.txt", np.uint8, np.uint8, (1, 1, 7, 7), (1, 1, 1, 1))
    assert np.array_equal(y, expect)


def test_qlinearconv_printed_int8_example(orc):
    y, expect = _run_conv_golden(orc, "qlinearconv_s8_2x2.txt", np.int8, np.int8, (1, 1, 2, 2), (1, 1, 2, 2))
    assert y.shape == (1,) and np.array_equal(y, expect)


# ----------------------------------------------------------------------------
# QuantizeLinear / DequantizeLinear closed forms
# ----------------------------------------------------------------------------

def test_quantize_linear_closed_form_cases(orc):
    for x, s, zp, t, y in read_golden_rows("quantize_linear_cases.txt"):
        got = orc.quantize_linear(np.array([float(x)], np.float32), np.float32(s), int(zp), None, t)
        assert got.dtype == _qdt(t)
        assert int(got[0]) == int(y), (x, s, zp, t, y, got)


def test_dequantize_linear_closed_form_cases(orc):
    for x, s, zp, t, y in read_golden_rows("dequantize_linear_cases.txt"):
        got = orc.dequantize_linear(np.array([int(x)], _qdt(t)), np.float32(s), int(zp))
        assert got.dtype == np.float32
        assert got[0] == np.float32(y), (x, s, zp, t, y, got)


@pytest.mark.parametrize("t", ["u8", "s8"])
def test_quantize_power_of_two_scales_match_exact_rational_rounding(orc, t):
    """With a power-of-two scale x/scale is exact, so the operator reduces to
    Python's round() (half to even) on exact rationals, then clamp."""
    rng = np.random.default_rng(11)
    lo, hi = (0, 255) if t == "u8" else (-128, 127)
    for e in (-7, -3, 0, 2):
        s = np.float32(2.0 ** e)
        zp = int(rng.integers(lo, hi + 1))
        k = rng.integers(-400, 400, size=500)
        frac = rng.choice([0.0, 0.25, 0.5, 0.75], size=500)
        x = ((k + frac) * float(s)).astype(np.float32)
        got = orc.quantize_linear(x, s, zp, None, t)
        for xi, gi in zip(x, got):
            r = round(Fraction(float(xi)) / Fraction(float(s))) + zp
            assert int(gi) == min(max(r, lo), hi)


def test_quantize_per_axis_equals_per_tensor_slices(orc):
    """Per-axis quantization along axis a is per-tensor quantization of each
    slice taken along a with that slice's scale and zero point."""
    rng = np.random.default_rng(5)
    x = rng.normal(0, 2, size=(3, 5, 7)).astype(np.float32)
    for axis in (0, 1, 2, -1):
        n = x.shape[axis]
        s = rng.uniform(0.005, 0.05, size=n).astype(np.float32)
        z = rng.integers(0, 256, size=n)
        y = orc.quantize_linear(x, s, z, axis, "u8")
        for c in range(n):
            ref = orc.quantize_linear(np.take(x, c, axis=axis), s[c], z[c], None, "u8")
            assert np.array_equal(np.take(y, c, axis=axis), ref)
        d = orc.dequantize_linear(y, s, z, axis)
        for c in range(n):
            ref = orc.dequantize_linear(np.take(y, c, axis=axis), s[c], z[c], None)
            assert np.array_equal(np.take(d, c, axis=axis), ref)


def test_qdq_ties_round_to_even(orc):
    """The tie positions the workload plants sit exactly at k + 0.5 after the
    fp32 division; QuantizeLinear must send each to the even neighbour."""
    w = workloads.qdq(seed=1, shape=(4, 8, 64), tie_fraction=0.2)
    x, s, zp = w["x"], w["scale"], w["zero_point"]
    y = orc.quantize_linear(x, s, zp, axis=2, ytype="u8")
    flat_x = x.reshape(-1)
    flat_y = y.reshape(-1).astype(np.int64)
    pos = w["tie_positions"]
    assert pos.size > 50
    ch = pos % 64
    q = (flat_x[pos] / s[ch]).astype(np.float32).astype(np.float64)
    assert np.all(q - np.floor(q) == 0.5)
    v = flat_y[pos] - zp[ch].astype(np.int64)
    assert np.all(v % 2 == 0)
    assert np.all(np.abs(v - q) == 0.5)


def test_qdq_roundtrip_error_within_half_scale(orc):
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, size=(64, 33)).astype(np.float32)
    s = rng.uniform(0.005, 0.05, size=33).astype(np.float32)
    z = rng.integers(0, 256, size=33)
    y = orc.quantize_linear(x, s, z, axis=1, ytype="u8")
    d = orc.dequantize_linear(y, s, z, axis=1)
    lo = (0 - z) * s.astype(np.float64)
    hi = (255 - z) * s.astype(np.float64)
    inside = (x >= lo) & (x <= hi)
    err = np.abs(d.astype(np.float64) - x)
    assert np.all(err[inside] <= 0.5 * s[np.nonzero(inside)[1]] * (1 + 1e-5))
    # outside the representable range the result saturates at the nearer end
    assert np.all(y[x > hi + s] == 255) and np.all(y[x < lo - s] == 0)


# ----------------------------------------------------------------------------
# Row / column quantization invariants
# ----------------------------------------------------------------------------

def test_row_quantization_invariants(orc):
    rng = np.random.default_rng(7)
    A = rng.normal(0, 1, size=(40, 97)).astype(np.float32)
    A[3] = np.abs(A[3])          # all non-negative: zero point 0
    A[4] = -np.abs(A[4])         # all non-positive: zero point 255
    A[5] = 0.0                   # degenerate row
    uA, sA, zA = orc.quantize_rows_u8(A)
    assert sA[5] == 1.0 and zA[5] == 0 and np.all(uA[5] == 0)
    assert zA[3] == 0 and zA[4] == 255
    for i in range(40):
        if i == 5:
            continue
        mn, mx = min(0.0, float(A[i].min())), max(0.0, float(A[i].max()))
        assert abs(float(sA[i]) - (mx - mn) / 255) <= 1e-6 * (mx - mn) / 255
        deq = (uA[i].astype(np.float64) - zA[i]) * float(sA[i])
        assert np.max(np.abs(deq - A[i])) <= 0.5 * float(sA[i]) * (1 + 1e-4)
        # the zero point is the code of real 0, the extremes map to the ends
        if mn < 0:
            assert uA[i, np.argmin(A[i])] == 0
        if mx > 0:
            assert uA[i, np.argmax(A[i])] >= 254


@pytest.mark.parametrize("avoid", [False, True])
def test_column_quantization_invariants(orc, avoid):
    rng = np.random.default_rng(8)
    B = rng.normal(0, 0.05, size=(77, 19)).astype(np.float32)
    B[:, 4] = 0.0
    iB, sB = orc.quantize_cols_s8(B, avoid)
    qmax = 63 if avoid else 127
    assert iB.min() >= (-64 if avoid else -128) and iB.max() <= qmax
    assert sB[4] == 1.0 and np.all(iB[:, 4] == 0)
    for j in range(19):
        if j == 4:
            continue
        m = np.abs(B[:, j]).max()
        assert abs(float(sB[j]) - m / qmax) <= 1e-6 * m / qmax
        assert abs(int(iB[np.argmax(np.abs(B[:, j])), j])) == qmax
        deq = iB[:, j].astype(np.float64) * float(sB[j])
        assert np.max(np.abs(deq - B[:, j])) <= 0.5 * float(sB[j]) * (1 + 1e-4)


# ----------------------------------------------------------------------------
# Dynamic quantized inner product
# ----------------------------------------------------------------------------

def lossless_A(rng, M, K):
    """Rows on the grid (q - z) * 2^e with a 0 and a 255 code present: the
    row scale (max - min) / 255 is exactly 2^e and the zero point exactly z,
    so quantization loses nothing."""
    A = np.empty((M, K), np.float32)
    for i in range(M):
        s = 2.0 ** int(rng.integers(-9, -4))
        z = int(rng.integers(0, 256))
        q = rng.integers(0, 256, size=K)
        if K == 1:
            q[0] = 255 if z == 0 else 0
            z = 0 if q[0] == 255 else 255
        else:
            lo_pos, hi_pos = rng.choice(K, size=2, replace=False)
            q[lo_pos], q[hi_pos] = 0, 255
        A[i] = (q - z) * s
    return A


def lossless_B(rng, K, N, qmax=127):
    B = np.empty((K, N), np.float32)
    for j in range(N):
        t = 2.0 ** int(rng.integers(-10, -5))
        v = rng.integers(-qmax, qmax + 1, size=K)
        v[rng.integers(0, K)] = qmax if rng.random() < 0.5 else -qmax
        B[:, j] = v * t
    return B


@pytest.mark.parametrize("M,N,K", [(1, 1, 2), (3, 5, 7), (8, 8, 16), (7, 13, 63), (17, 9, 129), (5, 33, 500)])
@pytest.mark.parametrize("avoid", [False, True])
def test_inner_product_lossless_grid_equals_fp64_product(orc, M, N, K, avoid):
    """Lossless special case: the method's result must equal the textbook
    fp64 product A @ B + bias, rounded once to fp32."""
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A = lossless_A(rng, M, K)
    B = lossless_B(rng, K, N, 63 if avoid else 127)
    bias = rng.uniform(-0.1, 0.1, size=N).astype(np.float32)
    out = orc.dynamic_quantized_inner_product(A, B, bias=bias, avoid_overflow=avoid)
    ref = (A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)).astype(np.float32)
    assert np.array_equal(out["C"], ref)
    relu = orc.dynamic_quantized_inner_product(A, B, bias=bias, act=orc.ACT_RELU, avoid_overflow=avoid)
    assert np.array_equal(relu["C"], np.where(ref > 0, ref, np.float32(0)))


def test_inner_product_gelu_matches_erf_definition(orc):
    rng = np.random.default_rng(21)
    A = lossless_A(rng, 9, 40)
    B = lossless_B(rng, 40, 11)
    bias = rng.uniform(-0.5, 0.5, size=11).astype(np.float32)
    out = orc.dynamic_quantized_inner_product(A, B, bias=bias, act=orc.ACT_GELU)
    v = (A.astype(np.float64) @ B.astype(np.float64) + bias).astype(np.float32).astype(np.float64)
    ref = np.vectorize(lambda t: 0.5 * t * math.erfc(-t / math.sqrt(2.0)))(v)
    err = np.abs(out["C"].astype(np.float64) - ref)
    # fp32 evaluation without cancellation: a few ulps of the result, plus
    # the rounding of the argument t = x / sqrt 2, which erfc(-t) amplifies
    # by about 2 t^2 in relative terms
    t2 = v * v / 2
    tol = np.abs(ref) * (8 + 2 * t2) * 2.0 ** -24 + 1e-44
    assert np.all(err <= tol)
    # the same values through the 1 + erf form agree to its own accuracy
    ref2 = np.vectorize(lambda t: 0.5 * t * (1.0 + math.erf(t / math.sqrt(2.0))))(v)
    assert np.all(np.abs(ref2 - ref) <= 1e-15 * np.maximum(np.abs(v), 1))


def _error_bound(A, B, bias, qmax):
    A64, B64 = A.astype(np.float64), B.astype(np.float64)
    rng_A = np.maximum(A64.max(1), 0) - np.minimum(A64.min(1), 0)
    eA = 0.5 * rng_A / 255 * (1 + 1e-3)
    eB = 0.5 * np.abs(B64).max(0) / qmax * (1 + 1e-3)
    ref = A64 @ B64 + bias
    bound = (np.abs(A64) @ np.ones_like(B64)) * eB[None, :] + eA[:, None] * (np.ones_like(A64) @ np.abs(B64)) \
        + A.shape[1] * eA[:, None] * eB[None, :] + 4 * 2.0 ** -24 * (np.abs(ref) + np.abs(bias)) + 1e-30
    return ref, bound


@pytest.mark.parametrize("avoid", [False, True])
def test_inner_product_within_quantization_error_bound(orc, avoid):
    w = workloads.inner_product(seed=0)
    out = orc.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"], avoid_overflow=avoid)
    ref, bound = _error_bound(w["A"], w["B"], w["bias"], 63 if avoid else 127)
    assert np.all(np.abs(out["C"] - ref) <= bound)
    # and the bound is not vacuous: the error is well below the result scale
    assert np.max(np.abs(out["C"] - ref)) < 0.05 * np.max(np.abs(ref))


@pytest.mark.parametrize("avoid", [True, False])
def test_usage_ramp_example_within_bound(orc, avoid):
    """The Simd usage example (M=4 N=8 K=16 ramps, bias 0.1, constant B,
    identity, fp32, avoidOverflow as printed = true).  The page prints no
    outputs, so the bound is the pin."""
    w = workloads.usage_ramp()
    out = orc.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"], avoid_overflow=avoid)
    ref, bound = _error_bound(w["A"], w["B"], w["bias"], 63 if avoid else 127)
    assert np.all(np.abs(out["C"] - ref) <= bound)
    assert np.all(out["zeroA"] == 0)                 # all-positive rows
    assert out["iB"].min() >= 0 and out["iB"].max() == (63 if avoid else 127)


def test_inner_product_zero_point_identity(orc):
    """sum_k (u - z) b == sum_k u b - z * colsum(b), checked in int64."""
    w = workloads.inner_product(seed=0, M=16, N=24, K=96)
    out = orc.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"])
    u = out["uA"].astype(np.int64)
    b = out["iB"].astype(np.int64)
    z = out["zeroA"].astype(np.int64)
    assert np.array_equal(out["acc"].astype(np.int64), u @ b - z[:, None] * b.sum(0)[None, :])


def test_degenerate_rows_give_activated_bias(orc):
    A = np.zeros((3, 10), np.float32)
    rng = np.random.default_rng(2)
    B = rng.normal(0, 0.05, (10, 6)).astype(np.float32)
    bias = np.array([-0.3, -0.1, 0.0, 0.1, 0.2, 0.7], np.float32)
    out = orc.dynamic_quantized_inner_product(A, B, bias=bias, act=orc.ACT_RELU)
    assert np.array_equal(out["C"], np.tile(np.maximum(bias, 0), (3, 1)))
    assert np.all(out["acc"] == 0)


def test_bf16_conversion_matches_torch(orc):
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.normal(0, 1, 5000), rng.normal(0, 1e30, 100), [0.0, -0.0, 1e-40, 3.0e38, -3.4e38]])
    x = x.astype(np.float32)
    # values exactly halfway between bf16 neighbours
    halves = (np.arange(200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, halves, -halves])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f32_to_bf16_bits(x), ref)


def test_bf16_input_widening_is_exact(orc):
    rng = np.random.default_rng(9)
    a = rng.normal(0, 3, 1000).astype(np.float32)
    bits = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(orc.bf16_bits_to_f32(bits), ref)


# ----------------------------------------------------------------------------
# QLinearConv invariants
# ----------------------------------------------------------------------------

def _small_conv(rng, N=2, C=4, H=6, W=5, M=3, k=3, group=1):
    x = rng.integers(0, 256, size=(N, C, H, W)).astype(np.uint8)
    w = rng.integers(0, 256, size=(M, C // group, k, k)).astype(np.uint8)
    ws = rng.uniform(0.001, 0.01, size=M).astype(np.float32)
    wz = rng.integers(100, 157, size=M)
    B = rng.integers(-5000, 5001, size=M).astype(np.int32)
    return x, w, ws, wz, B


def test_conv_padding_is_real_zero(orc):
    """A padded position holds real 0, i.e. the code x_zero_point: padding
    by p equals an unpadded conv over x framed with x_zero_point."""
    rng = np.random.default_rng(1)
    x, w, ws, wz, B = _small_conv(rng)
    y = orc.qlinearconv(x, np.float32(0.0037), 132, w, ws, wz, np.float32(0.05), 128, B, pads=(1, 2, 1, 0))
    xp = np.full((2, 4, 8, 7), 132, np.uint8)
    xp[:, :, 1:7, 2:7] = x
    y2 = orc.qlinearconv(xp, np.float32(0.0037), 132, w, ws, wz, np.float32(0.05), 128, B)
    assert np.array_equal(y, y2)


def test_depthwise_equals_block_diagonal_dense(orc):
    rng = np.random.default_rng(2)
    C = 5
    x, w, ws, wz, B = _small_conv(rng, C=C, M=C, group=C)
    y = orc.qlinearconv(x, np.float32(0.0037), 132, w, ws, wz, np.float32(0.05), 128, B,
                        pads=(1, 1, 1, 1), group=C)
    dense = np.empty((C, C, 3, 3), np.uint8)
    for m in range(C):
        dense[m] = wz[m]              # off-diagonal taps contribute w - w_zp = 0
        dense[m, m] = w[m, 0]
    y2 = orc.qlinearconv(x, np.float32(0.0037), 132, dense, ws, wz, np.float32(0.05), 128, B,
                         pads=(1, 1, 1, 1))
    assert np.array_equal(y, y2)


def test_conv_power_of_two_scales_equal_fp64_path(orc):
    """With power-of-two scales the requantization is exact, so QLinearConv
    equals DequantizeLinear -> float convolution (fp64) -> QuantizeLinear."""
    rng = np.random.default_rng(3)
    x, w, _, wz, B = _small_conv(rng, N=2, C=3, H=7, W=6, M=4)
    xs, ws, ys = 2.0 ** -6, np.array([2.0 ** -7, 2.0 ** -8, 2.0 ** -6, 2.0 ** -9], np.float32), 2.0 ** -1
    y = orc.qlinearconv(x, np.float32(xs), 120, w, ws, wz, np.float32(ys), 128, B, pads=(1, 1, 1, 1))
    ref = _fp64_conv_path(x, xs, 120, w, ws, wz, ys, 128, B, pad=1)
    assert np.array_equal(y, ref)


def _fp64_conv_path(x, xs, xz, w, ws, wz, ys, yz, B, pad):
    xd = (x.astype(np.float64) - xz) * xs
    N, C, H, W = x.shape
    M, _, k, _ = w.shape
    wd = (w.astype(np.float64) - np.asarray(wz, np.float64)[:, None, None, None]) * \
        np.asarray(ws, np.float64)[:, None, None, None]
    xp = np.zeros((N, C, H + 2 * pad, W + 2 * pad))
    xp[:, :, pad:pad + H, pad:pad + W] = xd
    OH, OW = H + 2 * pad - k + 1, W + 2 * pad - k + 1
    out = np.zeros((N, M, OH, OW))
    for kh in range(k):
        for kw in range(k):
            out += np.einsum("nchw,mc->nmhw", xp[:, :, kh:kh + OH, kw:kw + OW], wd[:, :, kh, kw])
    out += (B.astype(np.float64) * xs * np.asarray(ws, np.float64))[None, :, None, None]
    q = np.rint(out / ys) + yz
    return np.clip(q, 0, 255).astype(np.uint8)


def test_conv_general_scales_near_fp64_path(orc):
    rng = np.random.default_rng(4)
    x, w, ws, wz, B = _small_conv(rng, N=2, C=8, H=9, W=7, M=6)
    y = orc.qlinearconv(x, np.float32(0.0037), 132, w, ws, wz, np.float32(0.05), 128, B, pads=(1, 1, 1, 1))
    ref = _fp64_conv_path(x, float(np.float32(0.0037)), 132, w, ws, wz, float(np.float32(0.05)), 128, B, 1)
    d = np.abs(y.astype(int) - ref.astype(int))
    assert d.max() <= 1 and np.mean(d == 0) > 0.98


# ----------------------------------------------------------------------------
# DynamicQuantizeLSTM
# ----------------------------------------------------------------------------

def _sig(v):
    return 1.0 / (1.0 + np.exp(-v))


def _textbook_lstm(X, Wf, Rf, B, direction_rev=False):
    """fp64 unquantized LSTM, default activations, gate columns i, o, f, c."""
    T, b, _ = X.shape
    H = Rf.shape[0]
    h = np.zeros((b, H))
    c = np.zeros((b, H))
    Y = np.zeros((T, b, H))
    order = range(T - 1, -1, -1) if direction_rev else range(T)
    for t in order:
        g = X[t] @ Wf + h @ Rf + B[:4 * H] + B[4 * H:]
        i, o, f, ct = _sig(g[:, :H]), _sig(g[:, H:2 * H]), _sig(g[:, 2 * H:3 * H]), np.tanh(g[:, 3 * H:])
        c = f * c + i * ct
        h = o * np.tanh(c)
        Y[t] = h
    return Y


def test_lstm_first_step_lossless_equals_textbook(orc):
    """Step 0 with h0 = 0: the recurrent product is exactly 0 and, with X on
    the lossless grid and power-of-two W scales, the input projection is
    exact, so the first hidden state is the textbook LSTM cell."""
    rng = np.random.default_rng(6)
    T, b, I, H = 1, 4, 24, 8
    X = lossless_A(rng, T * b, I).reshape(T, b, I)
    W = rng.integers(-128, 128, size=(1, I, 4 * H)).astype(np.int8)
    R = rng.integers(-128, 128, size=(1, H, 4 * H)).astype(np.int8)
    Ws = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Rs = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Bb = rng.normal(0, 0.1, size=(1, 8 * H)).astype(np.float32)
    Y, Yh, Yc = orc.dynamic_quantize_lstm(X, W, R, Bb, Ws, Rs)
    ref = _textbook_lstm(X.astype(np.float64), W[0] * Ws[0].astype(np.float64), R[0] * Rs[0].astype(np.float64),
                         Bb[0].astype(np.float64))
    assert np.allclose(Y[0, 0], ref[0], rtol=2e-6, atol=2e-7)
    assert np.array_equal(Yh[0], Y[0, 0])


@pytest.mark.parametrize("direction", ["forward", "reverse", "bidirectional"])
def test_lstm_within_quantization_error_of_textbook(orc, direction):
    w = workloads.lstm(seed=4, T=6, batch=3, I=32, H=16, D=2 if direction == "bidirectional" else 1)
    Y, Yh, Yc = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                          direction=direction)
    dirs = {"forward": [False], "reverse": [True], "bidirectional": [False, True]}[direction]
    for d, rev in enumerate(dirs):
        ref = _textbook_lstm(w["X"].astype(np.float64), w["W"][d] * w["W_scale"][d].astype(np.float64),
                             w["R"][d] * w["R_scale"][d].astype(np.float64), w["B"][d].astype(np.float64), rev)
        err = np.abs(Y[:, d] - ref)
        assert err.max() < 0.02, err.max()
        assert np.abs(ref).max() > 0.2        # non-trivial activations
        last = 0 if rev else -1
        assert np.array_equal(Yh[d], Y[last, d])


# ---- QGemm (ONNX Runtime contrib schema "QGemm") -----------------------------

def _qgemm_golden():
    g = read_golden("qgemm_small_example.txt")
    M, K = map(int, g["M_K"])
    K2, N = map(int, g["K_N"])
    A = np.array(g["A_u8"], dtype=np.int64).astype(np.uint8).reshape(M, K)
    B = np.array(g["B_s8"], dtype=np.int64).astype(np.int8).reshape(K2, N)
    return g, A, B


@pytest.mark.parametrize("transA,transB", [(False, False), (True, False), (False, True), (True, True)])
def test_qgemm_worked_example(orc, transA, transB):
    g, A, B = _qgemm_golden()
    a = A.T.copy() if transA else A
    b = B.T.copy() if transB else B
    kw = dict(b_zero_point=np.array(g["b_zero_point"], np.int32), C=np.array([g["C_1xN"]], np.int32),
              alpha=float(g["alpha"][0]), transA=transA, transB=transB)
    bs = np.array(g["b_scale"], np.float32)
    y = orc.qgemm(a, float(g["a_scale"][0]), int(g["a_zero_point"][0]), b, bs, **kw)
    assert np.array_equal(y.ravel(), np.array(g["y_float"], np.float32))
    yq = orc.qgemm(a, float(g["a_scale"][0]), int(g["a_zero_point"][0]), b, bs, y_scale=float(g["y_scale"][0]),
                   y_zero_point=int(g["y_zero_point"][0]), **kw)
    assert yq.dtype == np.uint8 and np.array_equal(yq.ravel(), np.array(g["y_u8"], np.int64))


def _exact_qgemm(A, za, B, zb, C, alpha, a_s, b_s):
    """fp64 textbook: alpha * a_scale * b_scale * (sum (A - za)(B - zb) + C)."""
    acc = (A.astype(np.int64) - za) @ (B.astype(np.int64) - np.asarray(zb, np.int64).reshape(1, -1))
    if C is not None:
        acc = acc + np.asarray(C, np.int64)
    return acc, alpha * a_s * np.asarray(b_s, np.float64).reshape(1, -1) * acc


@pytest.mark.parametrize("atype,btype", [("u8", "s8"), ("s8", "s8"), ("u8", "u8"), ("s8", "u8")])
@pytest.mark.parametrize("cshape", [None, "MN", "1N", "N", "M1", "11"])
def test_qgemm_power_of_two_scales_exact(orc, atype, btype, cshape):
    """With power-of-two scales and alpha and |acc| < 2^24 every fp32 step
    is exact, so the float output equals the fp64 textbook value."""
    rng = np.random.default_rng(zlib.crc32(f"{atype}{btype}{cshape}".encode()))
    M, K, N = 5, 37, 6
    lo = {"u8": (0, 256), "s8": (-128, 128)}
    dt = {"u8": np.uint8, "s8": np.int8}
    A = rng.integers(*lo[atype], (M, K)).astype(dt[atype])
    B = rng.integers(*lo[btype], (K, N)).astype(dt[btype])
    za = int(rng.integers(*lo[atype]))
    zb = rng.integers(*lo[btype], N).astype(np.int32)
    bs = np.float32(2.0) ** rng.integers(-8, -2, N).astype(np.float32)
    C = {None: None, "MN": rng.integers(-999, 999, (M, N)), "1N": rng.integers(-999, 999, (1, N)),
         "N": rng.integers(-999, 999, N), "M1": rng.integers(-999, 999, (M, 1)),
         "11": rng.integers(-999, 999, (1, 1))}[cshape]
    y = orc.qgemm(A, 0.25, za, B, bs, zb, C=C, alpha=0.5)
    acc, ref = _exact_qgemm(A, za, B, zb, None if C is None else np.broadcast_to(np.asarray(C).reshape(
        (1, -1) if np.asarray(C).ndim == 1 else np.asarray(C).shape), (M, N)), 0.5, 0.25, bs)
    assert np.abs(acc).max() < 2**24
    assert np.array_equal(y.astype(np.float64), ref)


def test_qgemm_quantized_output_is_quantize_linear_of_float_output(orc):
    """The quantized output is QuantizeLinear of the float output (same
    fp32 value divided by y_scale), for both output types."""
    rng = np.random.default_rng(3)
    A = rng.integers(0, 256, (9, 70)).astype(np.uint8)
    B = rng.integers(-128, 128, (70, 11)).astype(np.int8)
    bs = rng.uniform(1e-3, 1e-2, 11).astype(np.float32)
    y = orc.qgemm(A, 0.02, 131, B, bs, alpha=1.5)
    for zp, t in ((np.uint8(120), "u8"), (np.int8(-3), "s8")):
        yq = orc.qgemm(A, 0.02, 131, B, bs, alpha=1.5, y_scale=0.37, y_zero_point=int(zp), ytype=t)
        ref = orc.quantize_linear(y, np.float32(0.37), np.array(zp), ytype=t)
        assert np.array_equal(yq, ref)


def test_qgemm_brute_force_matches_integer_definition(orc):
    """Tiny shapes, every combination of per-tensor / per-column B
    parameters: the integer sum before rescaling, recovered with unit scales,
    equals the definition evaluated directly in int64."""
    rng = np.random.default_rng(8)
    for M, K, N in [(1, 1, 1), (2, 3, 4), (3, 1, 2), (4, 5, 1)]:
        A = rng.integers(-128, 128, (M, K)).astype(np.int8)
        B = rng.integers(0, 256, (K, N)).astype(np.uint8)
        for per_col in (False, True):
            zb = rng.integers(0, 256, N if per_col else 1).astype(np.int32)
            bs = np.ones(N if per_col else 1, np.float32)
            y = orc.qgemm(A, 1.0, -7, B, bs, zb)
            ref = np.zeros((M, N), np.int64)
            for i in range(M):
                for j in range(N):
                    z = int(zb[j if per_col else 0])
                    ref[i, j] = sum((int(A[i, k]) + 7) * (int(B[k, j]) - z) for k in range(K))
            assert np.array_equal(y.astype(np.int64), ref)


# ---- MatMulIntegerToFloat / DynamicQuantizeMatMul (contrib schemas) -------

def test_matmul_integer_to_float_worked_example(orc):
    g = read_golden("matmul_integer_to_float_example.txt")
    A = np.array(g["A_u8"], np.int64).astype(np.uint8).reshape(2, 2)
    B = np.array(g["B_s8"], np.int64).astype(np.int8).reshape(2, 2)
    Y = orc.matmul_integer_to_float(A, B, float(g["a_scale"][0]), np.array(g["b_scale"], np.float32),
                                    np.int32(int(g["a_zero_point"][0])), np.array(g["b_zero_point"], np.int32),
                                    np.array(g["bias"], np.float32))
    assert np.array_equal(Y.ravel(), np.array(g["Y"], np.float32))


@pytest.mark.parametrize("atype,btype", [("u8", "s8"), ("s8", "u8"), ("u8", "u8"), ("s8", "s8")])
@pytest.mark.parametrize("a_rows,b_cols", [(False, False), (True, True), (True, False), (False, True)])
def test_matmul_integer_to_float_power_of_two_exact(orc, atype, btype, a_rows, b_cols):
    """Power-of-two scales and bias on a 2^-4 grid: every fp32 step is exact,
    so Y equals the fp64 textbook value."""
    rng = np.random.default_rng(zlib.crc32(f"mitf{atype}{btype}{a_rows}{b_cols}".encode()))
    M, K, N = 6, 45, 7
    lo = {"u8": (0, 256), "s8": (-128, 128)}
    dt = {"u8": np.uint8, "s8": np.int8}
    A = rng.integers(*lo[atype], (M, K)).astype(dt[atype])
    B = rng.integers(*lo[btype], (K, N)).astype(dt[btype])
    na, nb = (M if a_rows else 1), (N if b_cols else 1)
    az = rng.integers(*lo[atype], na).astype(np.int32)
    bz = rng.integers(*lo[btype], nb).astype(np.int32)
    as_ = (2.0 ** rng.integers(-6, -1, na)).astype(np.float32)
    bs = (2.0 ** rng.integers(-6, -1, nb)).astype(np.float32)
    bias = (rng.integers(-64, 64, N) / 16.0).astype(np.float32)
    Y = orc.matmul_integer_to_float(A, B, as_, bs, az, bz, bias)
    acc = (A.astype(np.int64) - az.reshape(-1, 1)) @ (B.astype(np.int64) - bz.reshape(1, -1))
    assert np.abs(acc).max() < 2**24
    ref = acc * (as_.astype(np.float64).reshape(-1, 1) * bs.astype(np.float64).reshape(1, -1)) + bias
    assert np.array_equal(Y.astype(np.float64), ref)


def test_matmul_integer_to_float_per_row_equals_per_tensor_rows(orc):
    """With one scale and zero point per row of A, each output row equals the
    per-tensor product of that row alone; an N-D A equals its flattened
    rows."""
    rng = np.random.default_rng(21)
    A = rng.integers(0, 256, (2, 3, 40)).astype(np.uint8)
    B = rng.integers(-128, 128, (40, 9)).astype(np.int8)
    as_ = rng.uniform(0.01, 0.1, 6).astype(np.float32)
    az = rng.integers(0, 256, 6).astype(np.int32)
    bs = rng.uniform(1e-3, 1e-2, 9).astype(np.float32)
    Y = orc.matmul_integer_to_float(A, B, as_, bs, az, None, None)
    assert Y.shape == (2, 3, 9)
    flat = A.reshape(6, 40)
    for i in range(6):
        yi = orc.matmul_integer_to_float(flat[i:i + 1], B, as_[i], bs, np.int32(az[i]))
        assert np.array_equal(Y.reshape(6, 9)[i], yi[0])


def test_dynamic_quantize_matmul_lossless_grid(orc):
    """A on the grid k * 2^-7 spanning exactly [-128, 127] * 2^-7 quantizes
    losslessly (scale 2^-7, zero point 128), so with power-of-two b_scale Y is
    the fp64 textbook A (B - zb) b_scale + bias."""
    rng = np.random.default_rng(22)
    M, K, N = 5, 64, 6
    k = rng.integers(-128, 128, (M, K))
    k[0, 0], k[0, 1] = -128, 127
    A = (k * 2.0 ** -7).astype(np.float32)
    B = rng.integers(-128, 128, (K, N)).astype(np.int8)
    bz = rng.integers(-128, 128, N).astype(np.int32)
    bs = (2.0 ** rng.integers(-8, -3, N)).astype(np.float32)
    bias = (rng.integers(-64, 64, N) / 8.0).astype(np.float32)
    out = orc.dynamic_quantize_matmul(A, B, bs, bz, bias)
    assert out["a_scale"] == np.float32(2.0 ** -7) and out["a_zero_point"] == 128
    ref = A.astype(np.float64) @ ((B.astype(np.int64) - bz) * bs.astype(np.float64)) + bias
    assert np.array_equal(out["Y"].astype(np.float64), ref)


def test_dynamic_quantize_matmul_tensor_quantization_invariants(orc):
    rng = np.random.default_rng(23)
    A = rng.normal(0, 2, (7, 33)).astype(np.float32)
    A[3, 4] = 9.5
    out = orc.dynamic_quantize_matmul(A, rng.integers(-128, 128, (33, 4)).astype(np.int8), np.float32(0.01))
    s, z, uA = out["a_scale"], out["a_zero_point"], out["uA"].astype(np.int64)
    assert s == np.float32((np.float32(9.5) - np.float32(A.min())) / np.float32(255))
    assert uA.max() == 255 and uA.min() == 0
    assert np.all(np.abs((uA - z) * np.float64(s) - A) <= np.float64(s) / 2 * (1 + 1e-6))


# ---- QLinear elementwise family (contrib schemas) ---------------------------

def _golden_ints(g, key, dt=np.int64):
    return np.array(g[key], np.int64).astype(dt)


def test_qlinear_elementwise_worked_cases(orc):
    g = read_golden("qlinear_elementwise_cases.txt")
    A = _golden_ints(g, "A", np.uint8).reshape(2, 2)
    B = _golden_ints(g, "B", np.uint8)
    assert np.array_equal(orc.mul_integer(A, B, 10, 100).ravel(), _golden_ints(g, "mul_integer"))
    cs, cz = g["add_c_scale_zp"]
    assert np.array_equal(orc.qlinear_binary("add", A, 0.5, 10, B, 0.25, 100, float(cs), int(cz)).ravel(),
                          _golden_ints(g, "add"))
    cs, cz = g["mul_c_scale_zp"]
    assert np.array_equal(orc.qlinear_binary("mul", A, 0.5, 10, B, 0.25, 100, float(cs), int(cz)).ravel(),
                          _golden_ints(g, "mul"))
    y = orc.qlinear_unary("leaky_relu", _golden_ints(g, "leaky_x", np.uint8), 0.5, 128, 0.5, 128, 0.25)
    assert np.array_equal(y, _golden_ints(g, "leaky_y"))


def _half_even(fr):
    """Round a Fraction to the nearest integer, ties to even."""
    f = math.floor(fr)
    d = fr - f
    if d > Fraction(1, 2) or (d == Fraction(1, 2) and f % 2 == 1):
        return f + 1
    return f


@pytest.mark.parametrize("qt", ["u8", "s8"])
@pytest.mark.parametrize("op", ["add", "mul"])
def test_qlinear_binary_power_of_two_exact(orc, qt, op):
    """Power-of-two scales: each fp32 step is exact, so every code equals the
    rational formula rounded half to even and saturated."""
    rng = np.random.default_rng(zlib.crc32(f"qbin{qt}{op}".encode()))
    lo, hi, dt = (0, 255, np.uint8) if qt == "u8" else (-128, 127, np.int8)
    A = rng.integers(lo, hi + 1, (7, 9)).astype(dt)
    B = rng.integers(lo, hi + 1, (7, 9)).astype(dt)
    za, zb, zc = (int(v) for v in rng.integers(lo, hi + 1, 3))
    sa, sb, sc = Fraction(1, 8), Fraction(1, 4), (Fraction(1, 2) if op == "add" else Fraction(16))
    C = orc.qlinear_binary(op, A, float(sa), za, B, float(sb), zb, float(sc), zc)
    for (i, j), c in np.ndenumerate(C):
        a, b = int(A[i, j]) - za, int(B[i, j]) - zb
        v = (sa * a + sb * b) / sc if op == "add" else (a * b) * (sa * sb) / sc
        assert int(c) == min(max(_half_even(v) + zc, lo), hi)


@pytest.mark.parametrize("shapes", [((3, 4, 5), (5,)), ((3, 1, 5), (1, 4, 1)), ((1,), (2, 3)), ((2, 3), ())])
def test_qlinear_broadcast_equals_explicit(orc, shapes):
    rng = np.random.default_rng(7)
    sa, sb = shapes
    A = rng.integers(0, 256, sa).astype(np.uint8)
    B = rng.integers(0, 256, sb).astype(np.uint8)
    out = np.broadcast_shapes(sa, sb)
    Ae, Be = np.broadcast_to(A, out).copy(), np.broadcast_to(B, out).copy()
    for op in ("add", "mul"):
        assert np.array_equal(orc.qlinear_binary(op, A, 0.03, 7, B, 0.02, 250, 0.07, 3),
                              orc.qlinear_binary(op, Ae, 0.03, 7, Be, 0.02, 250, 0.07, 3))
    assert np.array_equal(orc.mul_integer(A, B, 7, 250), orc.mul_integer(Ae, Be, 7, 250))


def test_mul_integer_exact(orc):
    rng = np.random.default_rng(8)
    A = rng.integers(-128, 128, (6, 1, 8)).astype(np.int8)
    B = rng.integers(0, 256, (5, 1)).astype(np.uint8)
    C = orc.mul_integer(A, B, -3, 200)
    ref = (A.astype(np.int64) + 3) * (B.astype(np.int64) - 200)
    assert C.shape == ref.shape and np.array_equal(C, ref)


@pytest.mark.parametrize("qt", ["u8", "s8"])
def test_qlinear_leaky_relu_power_of_two_exact(orc, qt):
    lo, hi, dt = (0, 255, np.uint8) if qt == "u8" else (-128, 127, np.int8)
    X = np.arange(lo, hi + 1).astype(dt)
    zx, zy = (100, 30) if qt == "u8" else (-20, 5)
    Y = orc.qlinear_unary("leaky_relu", X, 0.25, zx, 0.125, zy, 0.375)
    for x, y in zip(X.astype(np.int64), Y.astype(np.int64)):
        d = Fraction(int(x) - zx, 4)
        f = d * Fraction(3, 8) if d < 0 else d
        assert int(y) == min(max(_half_even(f * 8) + zy, lo), hi)


def test_qlinear_sigmoid_against_fp64(orc):
    """Every code equals the fp64 sigmoid quantized, except where the fp64
    value lies within 1e-5 of a rounding boundary (the fp32 exp may move it
    across); outputs are non-decreasing in the input."""
    X = np.arange(256).astype(np.uint8)
    xs, zx, ys, zy = 0.07, 131, 1.0 / 256, 0
    Y = orc.qlinear_unary("sigmoid", X, xs, zx, ys, zy).astype(np.int64)
    assert np.all(np.diff(Y) >= 0)
    for x, y in zip(range(256), Y):
        d = float(np.float32((x - zx) * np.float32(xs)))
        t = 1.0 / (1.0 + math.exp(-d)) / ys
        exact = min(max(int(np.rint(t)) + zy, 0), 255)
        if abs(t - math.floor(t) - 0.5) > 1e-5:
            assert y == exact
        else:
            assert abs(y - exact) <= 1


# ---- DynamicQuantizeLSTM variants ------------------------------------------

def _textbook_cell(gx, c0, Bv, H, P=None, clip=0.0, input_forget=False):
    """fp64 ONNX LSTM cell from pre-activation products gx (b, 4H) and c0,
    peepholes P (3H, iof), clip and coupled gates."""
    Wb, Rb = Bv[:4 * H], Bv[4 * H:]
    cl = (lambda v: np.clip(v, -clip, clip)) if clip > 0 else (lambda v: v)  # noqa: E731
    pi = 0 if P is None else P[:H] * c0
    pf = 0 if P is None else P[2 * H:] * c0
    i = _sig(cl(gx[:, :H] + pi + Wb[:H] + Rb[:H]))
    f = 1 - i if input_forget else _sig(cl(gx[:, 2 * H:3 * H] + pf + Wb[2 * H:3 * H] + Rb[2 * H:3 * H]))
    ct = np.tanh(cl(gx[:, 3 * H:] + Wb[3 * H:] + Rb[3 * H:]))
    c = f * c0 + i * ct
    po = 0 if P is None else P[H:2 * H] * c
    o = _sig(cl(gx[:, H:2 * H] + po + Wb[H:2 * H] + Rb[H:2 * H]))
    return o * np.tanh(c), c


@pytest.mark.parametrize("peep,clip,coupled", [(True, 0.0, False), (False, 0.7, False), (False, 0.0, True),
                                               (True, 1.3, True)])
def test_lstm_variant_first_step_equals_textbook(orc, peep, clip, coupled):
    """Step 0 with h0 = 0 (Gh exactly 0) and X on the lossless grid with
    power-of-two W scales (Gx exact): the cell with peepholes, clip or
    coupled gates is the fp64 textbook cell to fp32 rounding."""
    rng = np.random.default_rng(61)
    T, b, I, H = 1, 4, 24, 8
    X = lossless_A(rng, T * b, I).reshape(T, b, I)
    W = rng.integers(-128, 128, size=(1, I, 4 * H)).astype(np.int8)
    R = rng.integers(-128, 128, size=(1, H, 4 * H)).astype(np.int8)
    Ws = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Rs = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Bb = rng.normal(0, 0.1, size=(1, 8 * H)).astype(np.float32)
    c0 = rng.normal(0, 1, size=(1, b, H)).astype(np.float32)
    P = rng.normal(0, 0.5, size=(1, 3 * H)).astype(np.float32) if peep else None
    Y, Yh, Yc = orc.dynamic_quantize_lstm(X, W, R, Bb, Ws, Rs, c0=c0, P=P, clip=clip, input_forget=coupled)
    gx = X[0].astype(np.float64) @ (W[0] * Ws[0].astype(np.float64))
    h, c = _textbook_cell(gx, c0[0].astype(np.float64), Bb[0].astype(np.float64), H,
                          None if P is None else P[0].astype(np.float64), clip, coupled)
    assert np.allclose(Yc[0], c, rtol=4e-6, atol=4e-7)
    assert np.allclose(Yh[0], h, rtol=4e-6, atol=4e-7)


def test_lstm_variant_neutral_settings(orc):
    """Zero peepholes equal none; a clip above every gate input equals none."""
    w = workloads.lstm(seed=4, T=4, batch=3, I=32, H=16, D=1)
    base = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"])
    zp = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                   P=np.zeros((1, 48), np.float32))
    cl = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"], clip=1e30)
    for a, b_, c_ in zip(base, zp, cl):
        assert np.array_equal(a, b_) and np.array_equal(a, c_)
    lim = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"], clip=0.05)
    assert not np.array_equal(lim[0], base[0])


def test_lstm_uint8_weights_with_zero_point_equal_shifted_int8(orc):
    """uint8 W, R with zero point 128 per channel give the same sums as the
    int8 codes W - 128 without zero point, so the same outputs."""
    w = workloads.lstm(seed=4, T=5, batch=2, I=32, H=16, D=2)
    Wu = (w["W"].astype(np.int16) + 128).astype(np.uint8)
    Ru = (w["R"].astype(np.int16) + 128).astype(np.uint8)
    z = np.full((2, 64), 128, np.int32)
    a = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"], direction="bidirectional")
    b_ = orc.dynamic_quantize_lstm(w["X"], Wu, Ru, w["B"], w["W_scale"], w["R_scale"], direction="bidirectional",
                                   W_zero_point=z, R_zero_point=z)
    for x, y in zip(a, b_):
        assert np.array_equal(x, y)


def test_dyn_product_zero_point_brute_force(orc):
    rng = np.random.default_rng(62)
    A = rng.normal(0, 1, (5, 13)).astype(np.float32)
    B = rng.integers(0, 256, (13, 7)).astype(np.uint8)
    zb = rng.integers(0, 256, 7).astype(np.int32)
    sb = np.full(7, 0.25, np.float32)
    C = orc.dyn_product_zp(A, B, sb, zb)
    uA, sA, zA = orc.quantize_rows_u8(A)
    acc = (uA.astype(np.int64) - zA[:, None]) @ (B.astype(np.int64) - zb[None, :])
    ref = ((acc.astype(np.float32) * sA[:, None]).astype(np.float32) * sb[None, :]).astype(np.float32)
    assert np.array_equal(C, ref)
    iB = rng.integers(-128, 128, (13, 7)).astype(np.int8)
    assert np.array_equal(orc.dyn_product_zp(A, iB, sb), orc.dynamic_quantized_inner_product(A, iB=iB, scaleB=sb)["C32"])


@pytest.mark.parametrize("direction", ["forward", "reverse"])
def test_lstm_sequence_lens_equal_truncated_runs(orc, direction):
    """A batch row of length L gives the run over its first L inputs alone;
    Y is zero from t = L on; rows of full length are unchanged."""
    w = workloads.lstm(seed=4, T=6, batch=4, I=32, H=16, D=1)
    sel = slice(0, 1)
    lens = np.array([6, 3, 1, 0])
    Y, Yh, Yc = orc.dynamic_quantize_lstm(w["X"], w["W"][sel], w["R"][sel], w["B"][sel], w["W_scale"][sel],
                                          w["R_scale"][sel], direction=direction, sequence_lens=lens)
    Yf, Yhf, Ycf = orc.dynamic_quantize_lstm(w["X"], w["W"][sel], w["R"][sel], w["B"][sel], w["W_scale"][sel],
                                             w["R_scale"][sel], direction=direction)
    assert np.array_equal(Y[:, :, 0], Yf[:, :, 0]) and np.array_equal(Yh[:, 0], Yhf[:, 0])
    for b, L in enumerate(lens):
        assert np.all(Y[L:, :, b] == 0)
        if L == 0:
            assert np.all(Yh[:, b] == 0) and np.all(Yc[:, b] == 0)
            continue
        Yb, Yhb, Ycb = orc.dynamic_quantize_lstm(w["X"][:L, b:b + 1], w["W"][sel], w["R"][sel], w["B"][sel],
                                                 w["W_scale"][sel], w["R_scale"][sel], direction=direction)
        assert np.array_equal(Y[:L, :, b], Yb[:, :, 0])
        assert np.array_equal(Yh[:, b], Yhb[:, 0]) and np.array_equal(Yc[:, b], Ycb[:, 0])


# ---- fp32 elementary functions (exp, expm1, log1p, sigmoid, tanh, softplus) --

def _ulps(y, ref):
    """|y - ref| in fp32 ulps of ref (the spacing of fp32 at |ref|; the least
    subnormal below the normal range)."""
    sp = np.maximum(np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64), 2.0 ** -149)
    return np.abs(y.astype(np.float64) - ref) / sp


def _sweep(lo, hi, n=200_000, seed=0):
    rng = np.random.default_rng(seed)
    return np.concatenate([np.linspace(lo, hi, n), rng.uniform(lo, hi, n)]).astype(np.float32)


@pytest.mark.parametrize("name,lo,hi,ref,bound", [
    ("exp", -103.0, 88.7, np.exp, 1.0),
    ("expm1", -20.0, 20.0, np.expm1, 2.0),
    ("expm1", -1e-3, 1e-3, np.expm1, 2.0),
    ("log1p", 0.0, 1.0, np.log1p, 3.0),
    ("sigmoid", -87.0, 100.0, lambda v: 1.0 / (1.0 + np.exp(-v)), 3.0),
    ("tanh", -12.0, 12.0, np.tanh, 3.5),
    ("tanh", -1e-3, 1e-3, np.tanh, 3.5),
    ("softplus", -100.0, 100.0, lambda v: np.logaddexp(0.0, v), 3.5),
])
def test_elementary_functions_within_ulps_of_fp64(orc, name, lo, hi, ref, bound):
    """Each fp32 function is within a few ulps of the fp64 library value
    (numpy's exp, expm1, log1p, tanh, logaddexp) over its range."""
    x = _sweep(lo, hi)
    err = _ulps(orc.elementary(name, x), ref(x.astype(np.float64)))
    assert err.max() <= bound, (name, float(err.max()), float(x[np.argmax(err)]))


def test_elementary_special_values(orc):
    e = orc.elementary
    assert e("exp", [0.0])[0] == 1.0
    assert e("exp", [89.0])[0] == np.inf and e("exp", [-104.0])[0] == 0.0
    assert np.isfinite(e("exp", [88.72])[0])
    # exact powers of two: e^(k ln 2) rounds to 2^k within an ulp
    k = np.arange(-120, 127)
    assert np.all(_ulps(e("exp", (k * math.log(2)).astype(np.float32)), np.exp((k * math.log(2)).astype(np.float32)
                                                                                 .astype(np.float64))) <= 1.0)
    assert e("sigmoid", [0.0])[0] == 0.5
    assert e("sigmoid", [200.0])[0] == 1.0 and e("sigmoid", [-200.0])[0] == 0.0
    t = e("tanh", [0.0, -0.0, 9.6, -9.6, 1e-30])
    assert t[0] == 0.0 and np.signbit(t[1]) and t[2] == 1.0 and t[3] == -1.0 and t[4] == np.float32(1e-30)
    assert e("expm1", [0.0])[0] == 0.0 and e("expm1", [-30.0])[0] == -1.0
    assert e("log1p", [0.0])[0] == 0.0 and abs(float(e("log1p", [1.0])[0]) - math.log(2)) <= 6e-8
    assert e("softplus", [0.0])[0] == np.float32(math.log(2))
    assert e("softplus", [100.0])[0] == 100.0 and e("softplus", [-100.0])[0] > 0.0


def test_elementary_symmetries(orc):
    """tanh is odd bit for bit (it is evaluated on |x|); sigmoid(x) +
    sigmoid(-x) = 1 and softplus(x) - softplus(-x) = x to rounding; exp
    and sigmoid are non-decreasing on a fine grid (tanh and softplus, each
    a quotient or sum of separately rounded terms, may step back by an
    ulp)."""
    x = _sweep(-15.0, 15.0, n=20_000)
    assert np.array_equal(orc.elementary("tanh", -x), -orc.elementary("tanh", x))
    s = orc.elementary("sigmoid", x).astype(np.float64) + orc.elementary("sigmoid", -x)
    assert np.abs(s - 1.0).max() <= 2.5e-7
    d = orc.elementary("softplus", x).astype(np.float64) - orc.elementary("softplus", -x)
    assert np.abs(d - x).max() <= 1e-5 * np.abs(x).max()
    g = np.sort(x)
    for name in ("sigmoid", "exp"):
        assert np.all(np.diff(orc.elementary(name, g).astype(np.float64)) >= 0), name


# ---- DynamicQuantizeLSTM activations ("activations", "activation_alpha/beta") --

_F64_ACT = {
    "Relu": lambda x, a, b: np.maximum(x, 0.0),
    "Tanh": lambda x, a, b: np.tanh(x),
    "Sigmoid": lambda x, a, b: 1.0 / (1.0 + np.exp(-x)),
    "Affine": lambda x, a, b: a * x + b,
    "LeakyRelu": lambda x, a, b: np.where(x >= 0, x, a * x),
    "ThresholdedRelu": lambda x, a, b: np.where(x > a, x, 0.0),
    "ScaledTanh": lambda x, a, b: a * np.tanh(b * x),
    "HardSigmoid": lambda x, a, b: np.clip(a * x + b, 0.0, 1.0),
    "Elu": lambda x, a, b: np.where(x >= 0, x, a * np.expm1(np.minimum(x, 0.0))),
    "Softsign": lambda x, a, b: x / (1.0 + np.abs(x)),
    "Softplus": lambda x, a, b: np.logaddexp(0.0, x),
}


def test_lstm_activation_attribute_lists_are_consumed_in_order(orc):
    """alpha / beta values go, in order, to the functions that take them;
    functions past the end of a list take the ONNX operators' defaults
    (LeakyRelu 0.01 as the pages state)."""
    r = orc.resolve_lstm_activations(["LeakyRelu", "Tanh", "HardSigmoid", "Elu", "Softplus", "ScaledTanh"],
                                     [0.3, 0.4], [0.6], 2)
    A = orc.LSTM_ACTIVATIONS.index
    assert r == [[(A("LeakyRelu"), 0.3, 0.0), (A("Tanh"), 0.0, 0.0),
                  (A("HardSigmoid"), pytest.approx(0.4), pytest.approx(0.6))],
                 [(A("Elu"), 1.0, 0.0), (A("Softplus"), 0.0, 0.0), (A("ScaledTanh"), 1.0, 1.0)]]
    assert orc.resolve_lstm_activations(["LeakyRelu"] * 3, None, None, 1)[0][0] == (A("LeakyRelu"), 0.01, 0.0)
    d = orc.resolve_lstm_activations(None, None, None, 1)[0]
    assert [k for k, _, _ in d] == [A("Sigmoid"), A("Tanh"), A("Tanh")]


@pytest.mark.parametrize("slot", [0, 1, 2])
@pytest.mark.parametrize("name", sorted(_F64_ACT))
def test_lstm_activation_first_step_equals_textbook(orc, slot, name):
    """Step 0 with h0 = 0 (Gh exactly 0) and X on the lossless grid with
    power-of-two W scales (Gx exact): with `name` as f (slot 0: the i, o, f
    gates), g (slot 1: the cell candidate) or h (slot 2: the output), the
    cell is the fp64 ONNX LSTM cell with that function, to fp32 rounding."""
    rng = np.random.default_rng(70 + slot)
    T, b, I, H = 1, 4, 24, 8
    X = lossless_A(rng, T * b, I).reshape(T, b, I)
    W = rng.integers(-128, 128, size=(1, I, 4 * H)).astype(np.int8)
    R = rng.integers(-128, 128, size=(1, H, 4 * H)).astype(np.int8)
    Ws = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Rs = (2.0 ** rng.integers(-9, -6, size=(1, 4 * H))).astype(np.float32)
    Bb = rng.normal(0, 0.1, size=(1, 8 * H)).astype(np.float32)
    c0 = rng.normal(0, 1, size=(1, b, H)).astype(np.float32)
    names = ["Sigmoid", "Tanh", "Tanh"]
    names[slot] = name
    alpha, beta = [0.7, 1.3, 0.9], [0.25, 0.5, 0.75]   # each slot's values, whether used or not
    al = [alpha[k] for k in range(3) if orc.LSTM_ACTIVATION_PARAMS[names[k]][0] is not None]
    be = [beta[k] for k in range(3) if orc.LSTM_ACTIVATION_PARAMS[names[k]][1] is not None]
    Y, Yh, Yc = orc.dynamic_quantize_lstm(X, W, R, Bb, Ws, Rs, c0=c0, activations=names, activation_alpha=al,
                                          activation_beta=be)
    gx = X[0].astype(np.float64) @ (W[0] * Ws[0].astype(np.float64))
    Bd = Bb[0].astype(np.float64)
    g = gx + Bd[:4 * H] + Bd[4 * H:]
    fa = [lambda v, k=k: _F64_ACT[names[k]](v, alpha[k], beta[k]) for k in range(3)]
    i, o, f = fa[0](g[:, :H]), fa[0](g[:, H:2 * H]), fa[0](g[:, 2 * H:3 * H])
    c = f * c0[0] + i * fa[1](g[:, 3 * H:])
    h = o * fa[2](c)
    assert np.allclose(Yc[0], c, rtol=1e-5, atol=1e-6)
    assert np.allclose(Yh[0], h, rtol=1e-5, atol=1e-6)
