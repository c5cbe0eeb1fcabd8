"""QLinearConv on the GPU vs the CPU oracle: output codes bit-exact."""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from conftest import read_golden
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def run_conv(orc, dev, x, xs, xz, w, ws, wz, ys, yz, B=None, pads=(0, 0, 0, 0), strides=(1, 1), dil=(1, 1), group=1,
             ytype=None):
    ref = orc.qlinearconv(x, xs, xz, w, ws, wz, ys, yz, B, pads=pads, strides=strides, dilations=dil, group=group,
                          ytype=ytype)
    y = torch.empty(ref.shape, dtype=torch.uint8 if ref.dtype == np.uint8 else torch.int8, device=dev)
    ws_bytes = q.qlinearconv_workspace_size(x.shape, w.shape, pads, strides, dil, group)
    wsp = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev) if ws_bytes else None
    q.qlinearconv(_t(x, dev), float(xs), int(xz), _t(w, dev), _t(np.atleast_1d(ws).astype(np.float32), dev),
                  _t(np.atleast_1d(wz).astype(w.dtype), dev), float(ys), int(yz), y,
                  B=None if B is None else _t(B, dev), pads=pads, strides=strides, dilations=dil, group=group,
                  workspace=wsp)
    q.sync_status()
    got = y.cpu().numpy()
    assert np.array_equal(got, ref), f"{np.count_nonzero(got != ref)} of {ref.size} codes differ"
    return got


def test_printed_examples(orc, dev):
    g = read_golden("qlinearconv_u8_7x7.txt")
    x = np.array([int(v) for v in g["x"]], np.uint8).reshape(1, 1, 7, 7)
    y = run_conv(orc, dev, x, np.float32(g["x_scale"][0]), int(g["x_zero_point"][0]), np.zeros((1, 1, 1, 1), np.uint8),
                 np.float32(g["w_scale"][0]), int(g["w_zero_point"][0]), np.float32(g["y_scale"][0]),
                 int(g["y_zero_point"][0]))
    assert np.array_equal(y.reshape(-1), np.array([int(v) for v in g["y"]], np.uint8))
    g = read_golden("qlinearconv_s8_2x2.txt")
    x = np.array([int(v) for v in g["x"]], np.int8).reshape(1, 1, 2, 2)
    y = run_conv(orc, dev, x, np.float32(g["x_scale"][0]), int(g["x_zero_point"][0]), np.ones((1, 1, 2, 2), np.int8),
                 np.float32(1.0), 0, np.float32(1.0), -10)
    assert int(y.reshape(-1)[0]) == -2


CASES = [
    # N, C, H, W, M, k, pads, strides, dil, group
    (1, 3, 7, 5, 4, 3, (1, 1, 1, 1), (1, 1), (1, 1), 1),
    (2, 8, 9, 11, 6, 3, (0, 0, 0, 0), (1, 1), (1, 1), 1),
    (2, 8, 10, 9, 6, 3, (1, 2, 0, 1), (2, 1), (1, 1), 2),
    (1, 6, 12, 12, 6, 3, (2, 2, 2, 2), (1, 1), (2, 2), 6),
    (3, 16, 14, 13, 16, 3, (1, 1, 1, 1), (1, 1), (1, 1), 16),
    (1, 4, 5, 5, 8, 1, (0, 0, 0, 0), (1, 1), (1, 1), 1),
    (1, 5, 17, 3, 7, 5, (2, 2, 2, 2), (3, 2), (1, 1), 1),
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8"), ("u8", "s8", "u8"), ("s8", "u8", "s8")])
def test_shapes_and_types(orc, dev, case, types):
    N, C, H, W, M, k, pads, strides, dil, group = case
    rng = np.random.default_rng(N * 100 + C * 10 + M + k)
    dt = {"u8": (np.uint8, 0, 256), "s8": (np.int8, -128, 128)}
    xt, wt, yt = (dt[t] for t in types)
    x = rng.integers(xt[1], xt[2], (N, C, H, W)).astype(xt[0])
    w = rng.integers(wt[1], wt[2], (M, C // group, k, k)).astype(wt[0])
    ws = rng.uniform(0.001, 0.01, M).astype(np.float32)
    wz = rng.integers(wt[1], wt[2], M)
    B = rng.integers(-5000, 5001, M).astype(np.int32)
    run_conv(orc, dev, x, np.float32(0.0037), int(rng.integers(xt[1], xt[2])), w, ws, wz, np.float32(0.05),
             int(rng.integers(yt[1], yt[2])), B, pads, strides, dil, group, ytype=types[2])
    # per-tensor weight parameters, no bias
    run_conv(orc, dev, x, np.float32(0.02), int(rng.integers(xt[1], xt[2])), w, np.float32(0.004),
             int(rng.integers(wt[1], wt[2])), np.float32(0.3), int(rng.integers(yt[1], yt[2])), None, pads, strides,
             dil, group, ytype=types[2])


TC_CASES = [
    # N, C, H, W, M, k, pads: output rows that tile into 224-pixel tiles
    (2, 64, 14, 14, 130, 3, (1, 1, 1, 1)),   # OW 14: 16 rows per tile > OH (partial), M tail
    (1, 72, 10, 28, 40, 3, (1, 1, 1, 1)),    # C not a multiple of 64, OW 28
    (2, 32, 7, 56, 96, 1, (0, 0, 0, 0)),     # 1x1
    (1, 16, 9, 56, 64, 5, (2, 2, 2, 2)),     # 5x5
    (1, 8, 6, 58, 24, 3, (0, 0, 0, 0)),      # unpadded, OW 56 from W 58
    (3, 128, 8, 56, 256, 3, (1, 1, 1, 1)),   # two output-channel tiles, partial row group
    (1, 72, 7, 56, 40, 3, (1, 1, 1, 1)),     # W % 8 == 0 with C not a multiple of 64
    (1, 40, 6, 112, 48, 3, (1, 1, 1, 1)),    # OW 112: two rows per tile, several column rounds
    (2, 37, 5, 56, 40, 3, (1, 1, 1, 1)),     # odd C: a channel pair half in the padding
    # H % 8 == 0: the input centred in blocks of 8 rows x 64 channels
    (2, 72, 16, 28, 40, 3, (1, 1, 1, 1)),    # C not a multiple of 64
    (1, 37, 8, 56, 40, 3, (1, 1, 1, 1)),     # odd C
    (1, 64, 16, 14, 64, 3, (1, 1, 1, 1)),    # rows of 14 pixels, 8 rows a block
    (1, 24, 6, 56, 40, 3, (1, 1, 1, 1)),     # planes of 336 pixels: bulk stores, last row group half empty
]


@pytest.mark.parametrize("case", TC_CASES)
@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8"), ("u8", "s8", "s8")])
@pytest.mark.parametrize("store", ["bulk", "direct"])
def test_tensor_core_path(orc, dev, monkeypatch, case, types, store):
    """y by bulk tensor stores of 32 channels x 224 pixels where the planes
    allow (16-byte multiples, whole rows per tile), else (and forced) by
    the epilogue threads' own stores."""
    if store == "direct":
        monkeypatch.setenv("I8Q_CONV_DIRECT_STORE", "1")
    N, C, H, W, M, k, pads = case
    rng = np.random.default_rng(N * 1000 + C + M + k)
    dt = {"u8": (np.uint8, 0, 256), "s8": (np.int8, -128, 128)}
    xt, wt, yt = (dt[t] for t in types)
    x = rng.integers(xt[1], xt[2], (N, C, H, W)).astype(xt[0])
    w = rng.integers(wt[1], wt[2], (M, C, k, k)).astype(wt[0])
    ws = rng.uniform(0.001, 0.01, M).astype(np.float32)
    wz = rng.integers(wt[1], wt[2], M)
    B = rng.integers(-5000, 5001, M).astype(np.int32)
    assert q.qlinearconv_workspace_size(x.shape, w.shape, pads) > 0, "shape should take the tensor-core path"
    q.profile_enable(True)
    run_conv(orc, dev, x, np.float32(0.0037), int(rng.integers(xt[1], xt[2])), w, ws, wz, np.float32(0.05),
             int(rng.integers(yt[1], yt[2])), B, pads, ytype=types[2])
    # extreme zero points: the widest centered range (|x - x_zp| up to 255)
    run_conv(orc, dev, x, np.float32(0.02), xt[1], w, np.float32(0.004), wt[2] - 1, np.float32(0.3),
             int(rng.integers(yt[1], yt[2])), None, pads, ytype=types[2])
    prof = q.profile_collect()
    q.profile_enable(False)
    assert prof.get("qlinearconv_tc", (0,))[0] == 2


@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8")])
def test_row_centring_forced(orc, dev, monkeypatch, types):
    """The operands centred by the row kernel (shared-memory transpose) and
    a separate filter launch on a shape the one-launch form also takes."""
    monkeypatch.setenv("I8Q_CONV_CENTER_ROW", "1")
    N, C, H, W, M, k, pads = 2, 72, 7, 56, 40, 3, (1, 1, 1, 1)
    rng = np.random.default_rng(29)
    dt = {"u8": (np.uint8, 0, 256), "s8": (np.int8, -128, 128)}
    xt, wt, yt = (dt[t] for t in types)
    x = rng.integers(xt[1], xt[2], (N, C, H, W)).astype(xt[0])
    w = rng.integers(wt[1], wt[2], (M, C, k, k)).astype(wt[0])
    ws = rng.uniform(0.001, 0.01, M).astype(np.float32)
    wz = rng.integers(wt[1], wt[2], M)
    B = rng.integers(-5000, 5001, M).astype(np.int32)
    run_conv(orc, dev, x, np.float32(0.0037), int(rng.integers(xt[1], xt[2])), w, ws, wz, np.float32(0.05),
             int(rng.integers(yt[1], yt[2])), B, pads, ytype=types[2])


def test_direct_path_forced(orc, dev, monkeypatch):
    monkeypatch.setenv("I8Q_FORCE_CONV", "direct")
    N, C, H, W, M, k, pads = TC_CASES[0]
    rng = np.random.default_rng(3)
    x = rng.integers(0, 256, (N, C, H, W)).astype(np.uint8)
    w = rng.integers(0, 256, (M, C, k, k)).astype(np.uint8)
    assert q.qlinearconv_workspace_size(x.shape, w.shape, pads) == 0
    run_conv(orc, dev, x, np.float32(0.0037), 132, w, rng.uniform(0.001, 0.01, M).astype(np.float32),
             rng.integers(100, 157, M), np.float32(0.05), 128, None, pads)


def test_full_size_dense_sampled(orc, dev):
    """x [32,256,56,56], w [256,256,3,3]: the whole output on the GPU,
    compared for 2 images x 24 output channels (each output depends only on
    its image and its channel's filter)."""
    c = workloads.qlinearconv(seed=3)
    x, w = c["x"], c["w"]
    ref_shape = (32, 256, 56, 56)
    y = torch.empty(ref_shape, dtype=torch.uint8, device=dev)
    ws_bytes = q.qlinearconv_workspace_size(x.shape, w.shape, c["pads"], (1, 1), (1, 1), 1)
    wsp = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    q.qlinearconv(_t(x, dev), float(c["x_scale"]), c["x_zero_point"], _t(w, dev), _t(c["w_scale"], dev),
                  _t(c["w_zero_point"], dev), float(c["y_scale"]), c["y_zero_point"], y, B=_t(c["B"], dev),
                  pads=c["pads"], workspace=wsp)
    q.sync_status()
    got = y.cpu().numpy()
    rng = np.random.default_rng(0)
    imgs = [0, 31]
    chans = np.sort(rng.choice(256, 24, replace=False))
    for n in imgs:
        ref = orc.qlinearconv(x[n:n + 1], c["x_scale"], c["x_zero_point"], w[chans], c["w_scale"][chans],
                              c["w_zero_point"][chans], c["y_scale"], c["y_zero_point"], c["B"][chans],
                              pads=c["pads"])
        assert np.array_equal(got[n][chans], ref[0])


def test_full_size_depthwise(orc, dev):
    c = workloads.qlinearconv(seed=3, depthwise=True)
    run_conv(orc, dev, c["x"], c["x_scale"], c["x_zero_point"], c["w"], c["w_scale"], c["w_zero_point"],
             c["y_scale"], c["y_zero_point"], c["B"], c["pads"], group=c["group"])


DW_CASES = [
    # N, C, H, W, k, pads
    (2, 8, 56, 56, 3, (1, 1, 1, 1)),
    (1, 5, 17, 23, 3, (0, 2, 1, 0)),
    (3, 4, 9, 16, 5, (2, 2, 2, 2)),
    (1, 6, 30, 7, 5, (0, 0, 0, 0)),
    (2, 3, 8, 8, 3, (2, 1, 0, 2)),
    (1, 7, 56, 56, 3, (1, 1, 1, 1)),     # planes not a multiple of the planes per CTA
    (1, 3, 130, 130, 3, (1, 1, 1, 1)),   # more items per plane than threads
    (2, 5, 33, 21, 5, (2, 2, 2, 2)),     # rows of W % 4 != 0 bytes
    (1, 4, 12, 12, 3, (1, 1, 1, 1)),     # rows of whole words, not 8-byte pieces
]


def force_dw_kernel(monkeypatch, kernel):
    """rows: the persistent row kernel; halo: the halo-tile kernel."""
    if kernel == "halo":
        monkeypatch.setenv("I8Q_FORCE_CONV_HALO", "1")


DW_KERNELS = ["rows", "halo"]


@pytest.mark.parametrize("kernel", DW_KERNELS)
@pytest.mark.parametrize("case", DW_CASES)
@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8"), ("u8", "s8", "s8")])
def test_depthwise_kernels(orc, dev, monkeypatch, kernel, case, types):
    force_dw_kernel(monkeypatch, kernel)
    N, C, H, W, k, pads = case
    rng = np.random.default_rng(N * 100 + C * 10 + k)
    rg = {"u8": (0, 256, np.uint8), "s8": (-128, 128, np.int8)}
    xt, wt, yt = (rg[t] for t in types)
    x = rng.integers(xt[0], xt[1], (N, C, H, W)).astype(xt[2])
    w = rng.integers(wt[0], wt[1], (C, 1, k, k)).astype(wt[2])
    ws = rng.uniform(0.001, 0.01, C).astype(np.float32)
    wz = rng.integers(wt[0], wt[1], C)
    B = rng.integers(-5000, 5001, C).astype(np.int32)
    run_conv(orc, dev, x, np.float32(0.0037), int(rng.integers(xt[0], xt[1])), w, ws, wz, np.float32(0.05),
             int(rng.integers(yt[0], yt[1])), B, pads, group=C, ytype=types[2])


@pytest.mark.parametrize("kernel", DW_KERNELS)
@pytest.mark.parametrize("ys", [2.0, 0.5, 3.0, 0.1, 1e-30, 1e30, 3e38])
def test_depthwise_requantization_ties(orc, dev, monkeypatch, kernel, ys):
    """Unit input and filter scales make every rescaled sum an integer, so
    y_scale 2 puts half the quotients exactly on a tie (round half to even
    decides them); the other scales give exact, inexact, saturating,
    vanishing quotients and one whose reciprocal is not a normal number."""
    force_dw_kernel(monkeypatch, kernel)
    rng = np.random.default_rng(int(ys * 7) % 1000 if ys < 1e3 else 5)
    N, C, H, W, k = 2, 6, 20, 24, 3
    x = rng.integers(0, 16, (N, C, H, W)).astype(np.uint8)
    w = rng.integers(-8, 8, (C, 1, k, k)).astype(np.int8)
    B = rng.integers(-50, 51, C).astype(np.int32)
    run_conv(orc, dev, x, np.float32(1.0), 3, w, np.ones(C, np.float32), np.zeros(C, np.int64), np.float32(ys), 0, B,
             (1, 1, 1, 1), group=C, ytype="s8")


@pytest.mark.parametrize("kernel", DW_KERNELS)
@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8")])
def test_depthwise_large_bias(orc, dev, monkeypatch, kernel, types):
    """Biases around 2^24 and 2^30: int32 sums whose conversion to fp32
    rounds, with unit scales and y_scale 2^17 so that the codes still move
    with the tap sums."""
    force_dw_kernel(monkeypatch, kernel)
    rng = np.random.default_rng(11)
    rg = {"u8": (0, 256, np.uint8), "s8": (-128, 128, np.int8)}
    xt, wt, yt = (rg[t] for t in types)
    N, C, H, W, k = 2, 8, 19, 24, 3
    x = rng.integers(xt[0], xt[1], (N, C, H, W)).astype(xt[2])
    w = rng.integers(wt[0], wt[1], (C, 1, k, k)).astype(wt[2])
    wz = rng.integers(wt[0], wt[1], C)
    B = np.array([2 ** 24, -2 ** 24, 2 ** 24 - 2 ** 21, -(2 ** 24 - 2 ** 21), 2 ** 24 - 2 ** 21 + 1, 2 ** 30,
                  -2 ** 30, 12345], np.int32)
    # unit scales and y_scale 2^17: codes near +-128 that move with the tap sums
    run_conv(orc, dev, x, np.float32(1.0), int(rng.integers(xt[0], xt[1])), w, np.ones(C, np.float32), wz,
             np.float32(2.0 ** 17), 128 if types[2] == "u8" else 0, B, (1, 1, 1, 1), group=C, ytype=types[2])


@pytest.mark.parametrize("kernel", DW_KERNELS)
@pytest.mark.parametrize("types", [("u8", "u8", "u8"), ("s8", "s8", "s8")])
@pytest.mark.parametrize("ys", [2.0 ** 15, 2.0 ** 17, 4.00001, 3.99999, 4.0])
def test_depthwise_sum_range_edges(orc, dev, monkeypatch, kernel, types, ys):
    """Sums that reach +-(2^22 - 1) and +-2^22 (the row kernel carries sums
    below 2^22 as exact floats and takes larger ones another way), and
    quotients around 2^20 in magnitude, where the same switch happens for
    the rounded codes: every channel's filter is one centred value +-200,
    its bias puts the largest possible sum at the edge, and most inputs sit
    at the end of their range that reaches it."""
    force_dw_kernel(monkeypatch, kernel)
    rng = np.random.default_rng(17)
    s8 = types[0] == "s8"
    xmax = 128 if s8 else 255
    xz = -3 if s8 else 10
    N, C, H, W, k = 2, 8, 13, 24, 3
    wz = np.array([-128, 127] * 4 if s8 else [0, 200] * 4, np.int64)
    wc = wz + np.array([200, -200] * 4)           # centred filter +200 or -200 at every tap
    w = np.repeat(wc, k * k).reshape(C, 1, k, k).astype(np.int8 if s8 else np.uint8)
    wsum = 9 * (wc - wz)
    edge = np.array([2 ** 22 - 1, 2 ** 22 - 1, 2 ** 22, 2 ** 22, 2 ** 22 - 2, 2 ** 22 + 1, 2 ** 21, 2 ** 22 - 1])
    # |k0| + xmax * sum |w'| = edge, with k0 of the sign that the extreme inputs push further
    sign = np.sign(wc - wz) * (-1 if s8 else 1)
    k0 = sign * (edge - xmax * np.abs(wsum))
    B = (k0 + xz * wsum).astype(np.int32)
    # inputs at the extreme code (x_max for u8, -128 for s8) with a sprinkling of others
    lo, hi = (-128, 128) if s8 else (0, 256)
    x = np.full((N, C, H, W), -128 if s8 else 255, np.int64)
    m = rng.random(x.shape) < 0.3
    x[m] = rng.integers(lo, hi, int(m.sum()))
    x = x.astype(np.int8 if s8 else np.uint8)
    run_conv(orc, dev, x, np.float32(1.0), xz, w, np.ones(C, np.float32), wz, np.float32(ys), 0 if s8 else 128, B,
             (1, 1, 1, 1), group=C, ytype=types[2])
