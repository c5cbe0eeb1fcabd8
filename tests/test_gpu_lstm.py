"""DynamicQuantizeLSTM on the GPU vs the CPU oracle, bit for bit.

Both sides evaluate sigmoid and tanh as the same fixed sequence of fp32
operations, so every step computes the same bits: the hidden and cell
states, and the uint8 codes, scales and zero points of the hidden state that
the next step's product reads (read back from the workspace through the
i8q_dq_lstm_state_codes hook).  Checked step-locally from a given (h, c),
over whole sequences, and at the full size: sampled steps of the 512-step
run from their GPU states, the codes of the state each sampled step read,
and a whole 32-step sequence at the full width.
"""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu

DIRS = {"forward": q.LSTM_FORWARD, "reverse": q.LSTM_REVERSE, "bidirectional": q.LSTM_BIDIRECTIONAL}


@pytest.fixture(params=["imma", "tc", "tc_steps"], autouse=True)
def core(request, monkeypatch):
    """Every case runs with the recurrent product on the int8 mma.sync core
    and on the exact-integer tcgen05 core, the latter both as the
    persistent recurrence (one launch, where the layer fits) and as one
    launch per step."""
    monkeypatch.setenv("I8Q_FORCE_CORE", "imma" if request.param == "imma" else "tc")
    if request.param == "tc_steps":
        monkeypatch.setenv("I8Q_LSTM_STEPS", "1")
    return request.param


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def gpu_lstm(dev, w, direction, X=None, h0=None, c0=None, per_channel=True, codes=False):
    X = w["X"] if X is None else X
    T, batch, I = X.shape
    D = 2 if direction == "bidirectional" else 1
    # the workload holds two directions: a reverse-only run uses the second
    sel = slice(1, 2) if direction == "reverse" else slice(0, D)
    H = w["R"].shape[1]
    ws = torch.empty(q.dq_lstm_workspace_size(T, batch, I, H, DIRS[direction]), dtype=torch.uint8, device=dev)
    Y = torch.empty(T, D, batch, H, device=dev)
    Yh = torch.empty(D, batch, H, device=dev)
    Yc = torch.empty(D, batch, H, device=dev)
    Ws = w["W_scale"][sel] if per_channel else w["W_scale"][sel, 0].copy()
    Rs = w["R_scale"][sel] if per_channel else w["R_scale"][sel, 0].copy()
    q.dq_lstm_forward(_t(X, dev), _t(w["W"][sel], dev), _t(w["R"][sel], dev), _t(Ws, dev), _t(Rs, dev), ws,
                      direction=DIRS[direction], B=_t(w["B"][sel], dev),
                      h0=None if h0 is None else _t(h0, dev), c0=None if c0 is None else _t(c0, dev),
                      Y=Y, Y_h=Yh, Y_c=Yc, W_zero_point=_t(np.zeros(Ws.size, np.int8), dev),
                      R_zero_point=_t(np.zeros(Rs.size, np.int8), dev))
    q.sync_status()
    out = (Y.cpu().numpy(), Yh.cpu().numpy(), Yc.cpu().numpy())
    if codes:
        # codes of the state the last step read, and of the final state
        out += tuple(tuple(a.cpu().numpy() for a in q.dq_lstm_state_codes(ws, T, batch, I, H, DIRS[direction], k))
                     for k in (0, 1))
    return out


def assert_codes(orc, got, h, d, batch):
    """The GPU's codes, scale and zero point of direction d's rows equal the
    oracle's per-row quantization of h."""
    uh, sh, zh = got
    rows = slice(d * batch, (d + 1) * batch)
    u, s, z = orc.quantize_rows_u8(h)
    assert np.array_equal(uh[rows], u.astype(np.int32))
    assert np.array_equal(sh[rows], s)
    assert np.array_equal(zh[rows], z)


def oracle_step(orc, w, d, X_t, h, c):
    """One oracle step of direction d from state (h, c)."""
    H = w["R"].shape[1]
    Gx = orc.dynamic_quantized_inner_product(X_t, iB=w["W"][d], scaleB=w["W_scale"][d])["C32"]
    return orc.lstm_step(Gx, h, c, w["R"][d], w["R_scale"][d], w["B"][d, :4 * H], w["B"][d, 4 * H:])


@pytest.mark.parametrize("direction", ["forward", "reverse", "bidirectional"])
def test_single_step_from_given_state(orc, dev, direction):
    w = workloads.lstm(seed=4, T=1, batch=5, I=96, H=40)
    rng = np.random.default_rng(1)
    D = 2 if direction == "bidirectional" else 1
    h0 = rng.uniform(-0.9, 0.9, (D, 5, 40)).astype(np.float32)
    c0 = rng.normal(0, 1, (D, 5, 40)).astype(np.float32)
    Y, Yh, Yc, c_in, c_out = gpu_lstm(dev, w, direction, h0=h0, c0=c0, codes=True)
    for d in range(D):
        widx = 1 if direction == "reverse" else d
        assert_codes(orc, c_in, h0[d], d, 5)
        h, c = oracle_step(orc, w, widx, w["X"][0], h0[d], c0[d])
        assert np.array_equal(Y[0, d], h)
        assert np.array_equal(Yc[d], c)
        assert np.array_equal(Yh[d], Y[0, d])
        assert_codes(orc, c_out, h, d, 5)


@pytest.mark.parametrize("direction", ["forward", "reverse", "bidirectional"])
@pytest.mark.parametrize("per_channel", [True, False])
def test_short_sequence(orc, dev, direction, per_channel):
    w = workloads.lstm(seed=4, T=7, batch=3, I=64, H=32)
    if not per_channel:
        w["W_scale"][:] = w["W_scale"][:, :1]
        w["R_scale"][:] = w["R_scale"][:, :1]
    D = 2 if direction == "bidirectional" else 1
    Y, Yh, Yc, c_in, c_out = gpu_lstm(dev, w, direction, per_channel=per_channel, codes=True)
    sl = slice(0, D) if direction != "reverse" else slice(1, 2)
    ref = orc.dynamic_quantize_lstm(w["X"], w["W"][sl], w["R"][sl], w["B"][sl], w["W_scale"][sl], w["R_scale"][sl],
                                    direction=direction)
    assert np.array_equal(Y, ref[0])
    assert np.array_equal(Yh, ref[1])
    assert np.array_equal(Yc, ref[2])
    for d in range(D):
        rev = direction == "reverse" or d == 1
        assert_codes(orc, c_in, Y[1 if rev else 5, d], d, 3)   # the state the last step read
        assert_codes(orc, c_out, Yh[d], d, 3)


def test_nonzero_zero_point(orc, dev):
    """int8 W, R with nonzero per-channel zero points through the plain
    entry point (they run on the general tensor-core path)."""
    w = workloads.lstm(seed=4, T=3, batch=2, I=16, H=8, D=1)
    ws = torch.empty(q.dq_lstm_workspace_size(3, 2, 16, 8, q.LSTM_FORWARD), dtype=torch.uint8, device=dev)
    zp = np.zeros((1, 32), np.int8)
    zp[0, 3] = 1
    zp[0, 17] = -5
    Y = torch.empty(3, 1, 2, 8, device=dev)
    q.dq_lstm_forward(_t(w["X"], dev), _t(w["W"], dev), _t(w["R"], dev), _t(w["W_scale"], dev),
                      _t(w["R_scale"], dev), ws, B=_t(w["B"], dev), Y=Y, W_zero_point=_t(zp, dev),
                      R_zero_point=_t(zp, dev))
    q.sync_status()
    ref = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                    W_zero_point=zp.astype(np.int32), R_zero_point=zp.astype(np.int32))
    assert np.array_equal(Y.cpu().numpy(), ref[0])


@pytest.mark.parametrize("H,batch", [(144, 64), (336, 17), (512, 64), (1088, 64)])
def test_slab_counts(orc, dev, H, batch):
    """Hidden sizes padded to 3, 6, 8 and 17 slabs of 64 (8: one round of
    the persistent kernel's ring per step; 17: too wide for its shared
    memory, one launch per step), whole sequences bit for bit."""
    w = workloads.lstm(seed=5, T=5, batch=batch, I=64, H=H)
    Y, Yh, Yc, _, c_out = gpu_lstm(dev, w, "bidirectional", codes=True)
    ref = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                    direction="bidirectional")
    assert np.array_equal(Y, ref[0])
    assert np.array_equal(Yh, ref[1]) and np.array_equal(Yc, ref[2])
    for d in range(2):
        assert_codes(orc, c_out, Yh[d], d, batch)


def test_full_width_whole_sequence(orc, dev):
    """T=32 of the full-size layer (batch 64, I = H = 1024, bidirectional):
    every output of the whole sequence, bit for bit."""
    w = workloads.lstm(seed=4, T=32)
    Y, Yh, Yc, _, c_out = gpu_lstm(dev, w, "bidirectional", codes=True)
    ref = orc.dynamic_quantize_lstm(w["X"], w["W"], w["R"], w["B"], w["W_scale"], w["R_scale"],
                                    direction="bidirectional")
    assert np.array_equal(Y, ref[0])
    assert np.array_equal(Yh, ref[1]) and np.array_equal(Yc, ref[2])
    for d in range(2):
        assert_codes(orc, c_out, Yh[d], d, 64)


def test_full_size_sampled_steps(orc, dev):
    """T=512 batch=64 I=H=1024 bidirectional.  For sampled steps, the state
    the step starts from comes from the GPU: h from the whole run's Y, c
    (and the codes of h that the step read) from a GPU run over the
    preceding inputs."""
    w = workloads.lstm(seed=4)
    Y, Yh, Yc = gpu_lstm(dev, w, "bidirectional")
    assert np.all(np.isfinite(Y)) and np.abs(Y).max() < 1.0
    T = w["X"].shape[0]
    for t in (0, 1, 200, 511):
        # forward direction: state after steps 0..t-1
        if t == 0:
            h = np.zeros((64, 1024), np.float32)
            c = np.zeros((64, 1024), np.float32)
        else:
            _, hp, cp, _, c_out = gpu_lstm(dev, w, "forward", X=w["X"][:t], codes=True)
            h, c = hp[0], cp[0]
            assert np.array_equal(h, Y[t - 1, 0])
            assert_codes(orc, c_out, h, 0, 64)
        hf, _ = oracle_step(orc, w, 0, w["X"][t], h, c)
        assert np.array_equal(Y[t, 0], hf)
    for t in (511, 300):
        # reverse direction: state after steps T-1..t+1
        if t == T - 1:
            h = np.zeros((64, 1024), np.float32)
            c = np.zeros((64, 1024), np.float32)
        else:
            _, hp, cp, _, c_out = gpu_lstm(dev, w, "reverse", X=w["X"][t + 1:], codes=True)
            h, c = hp[0], cp[0]
            assert np.array_equal(h, Y[t + 1, 1])
            assert_codes(orc, c_out, h, 0, 64)
        hr, _ = oracle_step(orc, w, 1, w["X"][t], h, c)
        assert np.array_equal(Y[t, 1], hr)
