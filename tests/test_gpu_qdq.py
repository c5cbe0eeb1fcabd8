"""QuantizeLinear / DequantizeLinear on the GPU vs the CPU oracle: bit-exact
(integer codes, and fp32 dequantized values, which the operator fixes to one
rounding)."""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu


def _run_q(orc, dev, x, s, z, axis, t):
    zt = np.asarray(z).astype(np.uint8 if t == "u8" else np.int8)
    ref = orc.quantize_linear(x, s, zt.astype(np.int32), axis, t)
    xd = torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    y = torch.empty(x.shape, dtype=torch.uint8 if t == "u8" else torch.int8, device=dev)
    q.quantize_linear(xd, torch.from_numpy(np.atleast_1d(s).astype(np.float32)).to(dev),
                      torch.from_numpy(np.atleast_1d(zt)).to(dev), y, axis=axis)
    got = y.cpu().numpy()
    assert np.array_equal(got, ref)
    deq_ref = orc.dequantize_linear(ref, s, zt.astype(np.int32), axis)
    yd = torch.empty(x.shape, dtype=torch.float32, device=dev)
    q.dequantize_linear(y, torch.from_numpy(np.atleast_1d(s).astype(np.float32)).to(dev),
                        torch.from_numpy(np.atleast_1d(zt)).to(dev), yd, axis=axis)
    assert np.array_equal(yd.cpu().numpy(), deq_ref)


@pytest.mark.parametrize("shape", [(1,), (7,), (16,), (33,), (3, 5, 17), (2, 33, 64), (4, 16, 48), (2, 3, 32, 16)])
@pytest.mark.parametrize("t", ["u8", "s8"])
def test_small_shapes_every_axis(orc, dev, shape, t):
    rng = np.random.default_rng(sum(shape) + len(t))
    x = rng.normal(0, 2, size=shape).astype(np.float32)
    lo, hi = (0, 256) if t == "u8" else (-128, 128)
    # per tensor
    _run_q(orc, dev, x, np.float32(rng.uniform(0.005, 0.05)), rng.integers(lo, hi), None, t)
    for axis in range(-len(shape), len(shape)):
        n = shape[axis]
        _run_q(orc, dev, x, rng.uniform(0.005, 0.05, n).astype(np.float32), rng.integers(lo, hi, n), axis, t)


def test_ties_and_saturation(orc, dev):
    d = workloads.qdq(seed=7, shape=(8, 16, 128), tie_fraction=0.3)
    x = d["x"].copy()
    x.reshape(-1)[:50] = 1e6      # saturate high
    x.reshape(-1)[50:100] = -1e6  # saturate low
    _run_q(orc, dev, x, d["scale"], d["zero_point"], 2, "u8")
    _run_q(orc, dev, x, np.float32(0.02), 0, None, "s8")


def test_extreme_scales(orc, dev):
    """Per-channel scales whose reciprocal is not a normal number (subnormal
    and near the largest float) next to ordinary ones, inputs with zeros,
    tiny and huge magnitudes, and exact ties."""
    rng = np.random.default_rng(12)
    C = 64
    s = rng.uniform(0.005, 0.05, C).astype(np.float32)
    s[:8] = [1e-39, 5e-40, 2.9e-39, 3e38, 1e38, 1e-30, 1e30, 7e-45]
    x = rng.normal(0, 2, (40, C)).astype(np.float32)
    x[0] = 0.0
    x[1] = 1e-40
    x[2] = -3e38
    x[3] = 3e38
    x[4:8, 8:] = (np.round(x[4:8, 8:] / s[8:]) + 0.5) * s[8:]  # ties on the ordinary channels
    for t, lo, hi in (("u8", 0, 256), ("s8", -128, 128)):
        _run_q(orc, dev, x, s, rng.integers(lo, hi, C), 1, t)
        for sc in (np.float32(1e-39), np.float32(3e38), np.float32(0.02)):
            _run_q(orc, dev, x, sc, 0, None, t)


def test_closed_form_golden_cases(orc, dev):
    from conftest import read_golden_rows
    for x, s, zp, t, y in read_golden_rows("quantize_linear_cases.txt"):
        xd = torch.tensor([float(x)], dtype=torch.float32, device=dev)
        out = torch.empty(1, dtype=torch.uint8 if t == "u8" else torch.int8, device=dev)
        q.quantize_linear(xd, torch.tensor([float(s)], device=dev),
                          torch.tensor([int(zp)], dtype=out.dtype, device=dev), out)
        assert int(out.item()) == int(y), (x, s, zp, t, y)


def test_unaligned_and_empty(orc, dev):
    rng = np.random.default_rng(3)
    base = torch.from_numpy(rng.normal(0, 2, 1000).astype(np.float32)).to(dev)
    x = base[1:1 + 512]  # 4-byte offset: not 16-byte aligned
    ref = orc.quantize_linear(x.cpu().numpy(), np.float32(0.01), 3, None, "u8")
    ybuf = torch.empty(600, dtype=torch.uint8, device=dev)
    y = ybuf[3:3 + 512]
    q.quantize_linear(x, torch.tensor([0.01], device=dev), torch.tensor([3], dtype=torch.uint8, device=dev), y)
    assert np.array_equal(y.cpu().numpy(), ref)
    e = torch.empty((0, 5), dtype=torch.float32, device=dev)
    ye = torch.empty((0, 5), dtype=torch.uint8, device=dev)
    q.quantize_linear(e, torch.tensor([0.1], device=dev), torch.tensor([0], dtype=torch.uint8, device=dev), ye)
    q.sync_status()


def test_full_size_round_trip(orc, dev):
    """[32,1024,4096] per-axis uint8 (axis 2) and per-tensor int8, every
    element compared."""
    d = workloads.qdq(seed=1)
    x = d["x"]
    xd = torch.from_numpy(x).to(dev)
    for t, s, z, axis in (("u8", d["scale"], d["zero_point"], 2), ("s8", np.float32(0.02), np.int8(0), None)):
        st = torch.from_numpy(np.atleast_1d(s).astype(np.float32)).to(dev)
        zt = torch.from_numpy(np.atleast_1d(z)).to(dev)
        y = torch.empty(x.shape, dtype=zt.dtype, device=dev)
        q.quantize_linear(xd, st, zt, y, axis=axis)
        ref = orc.quantize_linear(x, s, np.atleast_1d(z).astype(np.int32), axis, t)
        got = y.cpu().numpy()
        assert np.array_equal(got, ref), f"{t}: {np.count_nonzero(got != ref)} codes differ"
        yd = torch.empty(x.shape, dtype=torch.float32, device=dev)
        q.dequantize_linear(y, st, zt, yd, axis=axis)
        dref = orc.dequantize_linear(ref, s, np.atleast_1d(z).astype(np.int32), axis)
        assert np.array_equal(yd.cpu().numpy(), dref)
        del y, yd


@pytest.mark.parametrize("shape,axis", [((3, 700, 4096), 2), ((5000, 768), 1), ((20000, 48), 1), ((300, 1000), 1),
                                        ((64, 12, 1000), 1), ((3, 700, 4096), None)])
def test_mid_size_vector_paths(orc, dev, shape, axis):
    """Sizes between the small cases and the full one: several waves of
    blocks with a ragged last round, last axes whose length does or does not
    divide the grid stride, an inner axis, and the per-tensor form."""
    rng = np.random.default_rng(sum(shape))
    x = rng.normal(0, 2, size=shape).astype(np.float32)
    if axis is None:
        _run_q(orc, dev, x, np.float32(0.02), 0, None, "s8")
        _run_q(orc, dev, x, np.float32(0.013), 77, None, "u8")
    else:
        n = shape[axis]
        _run_q(orc, dev, x, rng.uniform(0.005, 0.05, n).astype(np.float32), rng.integers(0, 256, n), axis, "u8")
        _run_q(orc, dev, x, rng.uniform(0.005, 0.05, n).astype(np.float32), rng.integers(-128, 128, n), axis, "s8")
