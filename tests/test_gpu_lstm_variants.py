"""DynamicQuantizeLSTM with its optional inputs and attributes on the GPU vs
the CPU oracle: sequence_lens, peepholes, clip, input_forget, uint8 weights,
nonzero W/R zero points (per direction and per channel), and the ONNX
activation functions with their alpha / beta lists.

Both sides evaluate the activations as the same fixed sequences of fp32
operations, so every output is compared bit for bit.
"""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu

DIRS = {"forward": q.LSTM_FORWARD, "reverse": q.LSTM_REVERSE, "bidirectional": q.LSTM_BIDIRECTIONAL}


@pytest.fixture(params=["persistent", "steps"], autouse=True)
def recurrence(request, monkeypatch):
    """Each case runs as the persistent recurrence (one launch, where the
    layer fits) and as one launch per step."""
    if request.param == "steps":
        monkeypatch.setenv("I8Q_LSTM_STEPS", "1")
    return request.param


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def weights(seed, T, batch, I, H, direction, wtype="s8", zp="none"):
    """Inputs of one direction setting; zp: none | dir | chan."""
    w = workloads.lstm(seed=seed, T=T, batch=batch, I=I, H=H)
    D = 2 if direction == "bidirectional" else 1
    sel = slice(1, 2) if direction == "reverse" else slice(0, D)
    W, R = w["W"][sel], w["R"][sel]
    rng = np.random.default_rng(seed)
    Wz = Rz = None
    if wtype == "u8":
        W = (W.astype(np.int16) + 128).astype(np.uint8)
        R = (R.astype(np.int16) + 128).astype(np.uint8)
    lo, hi = (0, 256) if wtype == "u8" else (-128, 128)
    if zp == "dir":
        Wz = rng.integers(lo, hi, (D,)).astype(W.dtype)
        Rz = rng.integers(lo, hi, (D,)).astype(W.dtype)
    elif zp == "chan":
        Wz = rng.integers(lo, hi, (D, 4 * H)).astype(W.dtype)
        Rz = rng.integers(lo, hi, (D, 4 * H)).astype(W.dtype)
    Ws, Rs = w["W_scale"][sel], w["R_scale"][sel]
    if zp == "dir":
        Ws, Rs = Ws[:, :1].copy(), Rs[:, :1].copy()
    return dict(X=w["X"], W=W, R=R, B=w["B"][sel], Ws=Ws, Rs=Rs, Wz=Wz, Rz=Rz, D=D, H=H)


def run_gpu(dev, p, direction, seq=None, P=None, clip=0.0, coupled=False, h0=None, c0=None, acts=None, alpha=None,
            beta=None):
    T, batch, I = p["X"].shape
    D, H = p["D"], p["H"]
    ws = torch.empty(q.dq_lstm_workspace_size(T, batch, I, H, DIRS[direction]), dtype=torch.uint8, device=dev)
    Y = torch.full((T, D, batch, H), 7.0, device=dev)  # every entry must be written
    Yh = torch.empty(D, batch, H, device=dev)
    Yc = torch.empty(D, batch, H, device=dev)
    opt = lambda a, dt=None: None if a is None else _t(a if dt is None else np.asarray(a, dt), dev)  # noqa: E731
    q.dq_lstm_forward_ex(_t(p["X"], dev), _t(p["W"], dev), _t(p["R"], dev), _t(p["Ws"], dev), _t(p["Rs"], dev), ws,
                         direction=DIRS[direction], B=_t(p["B"], dev), sequence_lens=opt(seq, np.int32),
                         h0=opt(h0), c0=opt(c0), P=opt(P), clip=clip, input_forget=coupled, Y=Y, Y_h=Yh, Y_c=Yc,
                         W_zero_point=opt(p["Wz"]), R_zero_point=opt(p["Rz"]), activations=acts,
                         activation_alpha=alpha, activation_beta=beta)
    q.sync_status()
    return Y.cpu().numpy(), Yh.cpu().numpy(), Yc.cpu().numpy()


def run_oracle(orc, p, direction, seq=None, P=None, clip=0.0, coupled=False, h0=None, c0=None, acts=None, alpha=None,
               beta=None):
    D, H = p["D"], p["H"]
    Ws = np.broadcast_to(p["Ws"], (D, 4 * H)).astype(np.float32)
    Rs = np.broadcast_to(p["Rs"], (D, 4 * H)).astype(np.float32)
    Wz = None if p["Wz"] is None else np.broadcast_to(np.asarray(p["Wz"]).reshape(D, -1), (D, 4 * H)).astype(np.int32)
    Rz = None if p["Rz"] is None else np.broadcast_to(np.asarray(p["Rz"]).reshape(D, -1), (D, 4 * H)).astype(np.int32)
    return orc.dynamic_quantize_lstm(p["X"], p["W"], p["R"], p["B"], Ws, Rs, h0=h0, c0=c0, direction=direction,
                                     W_zero_point=Wz, R_zero_point=Rz, P=P, clip=clip, input_forget=coupled,
                                     sequence_lens=seq, activations=acts, activation_alpha=alpha,
                                     activation_beta=beta)


def compare(got, ref):
    for g, r in zip(got, ref):
        assert np.array_equal(g, r), float(np.abs(g.astype(np.float64) - r).max())


FEATURES = {
    "peepholes": dict(P=True),
    "clip": dict(clip=0.4),
    "input_forget": dict(coupled=True),
    "seq_lens": dict(seq=True),
    "all": dict(P=True, clip=0.9, coupled=True, seq=True),
}


@pytest.mark.parametrize("direction", ["forward", "reverse", "bidirectional"])
@pytest.mark.parametrize("feature", sorted(FEATURES))
def test_features_short_sequence(orc, dev, direction, feature):
    p = weights(40, 7, 5, 64, 32, direction)
    f = FEATURES[feature]
    rng = np.random.default_rng(41)
    P = rng.normal(0, 0.5, (p["D"], 3 * 32)).astype(np.float32) if f.get("P") else None
    seq = np.array([7, 3, 0, 5, 1]) if f.get("seq") else None
    kw = dict(seq=seq, P=P, clip=f.get("clip", 0.0), coupled=f.get("coupled", False))
    got = run_gpu(dev, p, direction, **kw)
    ref = run_oracle(orc, p, direction, **kw)
    compare(got, ref)
    if seq is not None:
        for b, L in enumerate(seq):
            assert np.all(got[0][L:, :, b] == 0)


@pytest.mark.parametrize("wtype,zp", [("s8", "dir"), ("s8", "chan"), ("u8", "none"), ("u8", "dir"), ("u8", "chan")])
@pytest.mark.parametrize("direction", ["forward", "bidirectional"])
def test_weight_types_and_zero_points(orc, dev, wtype, zp, direction):
    p = weights(42, 6, 4, 96, 40, direction, wtype, zp)
    compare(run_gpu(dev, p, direction), run_oracle(orc, p, direction))


def test_single_step_from_given_state(orc, dev):
    """One step with every feature from a given (h, c)."""
    p = weights(43, 1, 6, 128, 48, "bidirectional", "u8", "chan")
    rng = np.random.default_rng(44)
    h0 = rng.uniform(-0.9, 0.9, (2, 6, 48)).astype(np.float32)
    c0 = rng.normal(0, 1, (2, 6, 48)).astype(np.float32)
    P = rng.normal(0, 0.5, (2, 144)).astype(np.float32)
    kw = dict(P=P, clip=1.5, coupled=True, h0=h0, c0=c0, seq=np.array([1, 1, 0, 1, 1, 0]))
    compare(run_gpu(dev, p, "bidirectional", **kw), run_oracle(orc, p, "bidirectional", **kw))


def test_all_features_wider_layer(orc, dev):
    """T=12 batch=64 I=H=256 bidirectional with every feature (several gate
    tiles, both batch tiles of the step kernel)."""
    p = weights(45, 12, 64, 256, 256, "bidirectional", "u8", "chan")
    rng = np.random.default_rng(46)
    P = rng.normal(0, 0.3, (2, 768)).astype(np.float32)
    seq = rng.integers(0, 13, 64)
    seq[:3] = [12, 0, 1]
    kw = dict(P=P, clip=2.0, coupled=False, seq=seq)
    compare(run_gpu(dev, p, "bidirectional", **kw), run_oracle(orc, p, "bidirectional", **kw))


def test_lengths_outside_range_are_clamped(orc, dev):
    p = weights(47, 5, 3, 64, 16, "reverse")
    got = run_gpu(dev, p, "reverse", seq=np.array([9, -2, 5]))
    ref = run_oracle(orc, p, "reverse", seq=np.array([5, 0, 5]))
    compare(got, ref)


ACTIVATIONS = ["Relu", "Tanh", "Sigmoid", "Affine", "LeakyRelu", "ThresholdedRelu", "ScaledTanh", "HardSigmoid",
               "Elu", "Softsign", "Softplus"]


@pytest.mark.parametrize("slot", [0, 1, 2])
@pytest.mark.parametrize("name", ACTIVATIONS)
def test_activation_functions(orc, dev, name, slot):
    """Each ONNX activation as f (the i, o, f gates), g (the candidate) or h
    (the output), with the operator's default alpha / beta, over a short
    forward sequence from a nonzero state."""
    p = weights(48, 5, 3, 32, 16, "forward")
    acts = ["Sigmoid", "Tanh", "Tanh"]
    acts[slot] = name
    rng = np.random.default_rng(49)
    h0 = rng.uniform(-0.9, 0.9, (1, 3, 16)).astype(np.float32)
    c0 = rng.normal(0, 1, (1, 3, 16)).astype(np.float32)
    kw = dict(acts=acts, h0=h0, c0=c0)
    compare(run_gpu(dev, p, "forward", **kw), run_oracle(orc, p, "forward", **kw))


def test_activation_lists_per_direction(orc, dev):
    """Six functions (three per direction) whose alpha / beta come from the
    attribute lists, consumed in the order of the functions; the last
    functions fall back to their defaults; combined with peepholes, clip
    and sequence lengths."""
    p = weights(50, 6, 5, 64, 32, "bidirectional", "u8", "chan")
    rng = np.random.default_rng(51)
    kw = dict(acts=["HardSigmoid", "Elu", "ScaledTanh", "LeakyRelu", "Affine", "Softsign"],
              alpha=[0.3, 0.8, 1.2, 0.05], beta=[0.45, 0.7],
              P=rng.normal(0, 0.5, (2, 96)).astype(np.float32), clip=3.0, seq=np.array([6, 2, 0, 5, 1]))
    compare(run_gpu(dev, p, "bidirectional", **kw), run_oracle(orc, p, "bidirectional", **kw))
    # the default functions given explicitly are the default path
    d = dict(acts=["Sigmoid", "Tanh", "Tanh"] * 2)
    compare(run_gpu(dev, p, "bidirectional", **d), run_gpu(dev, p, "bidirectional"))


def test_activation_arguments_rejected(dev):
    p = weights(52, 2, 2, 16, 8, "forward")
    for bad in (["Sigmoid", "Tanh"], ["Sigmoid", "Tanh", "Tanh"] * 2):
        with pytest.raises(q.I8QError):
            run_gpu(dev, p, "forward", acts=bad)
