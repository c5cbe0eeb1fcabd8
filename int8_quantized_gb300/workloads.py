"""Seeded synthetic inputs for the five workloads and the small usage example.

Every generator draws from a seeded CPU ``torch.Generator`` and returns numpy
arrays, so the CUDA library and the CPU oracle receive the same bytes.  This
module holds no quantization arithmetic: it only shapes random draws to the
sizes, distributions and structure the workloads name.

Workloads (sizes are the defaults; every generator takes smaller ones):
  inner_product   dynamic quantized inner product, M=64 N=128 K=256
  usage_ramp      the 4x8x16 ramp of the Simd usage example
  qdq             QuantizeLinear/DequantizeLinear x [32,1024,4096] with 1% ties
  large_gemm      dynamic quantized GEMM M=8192 K=4096 N=14336, bf16 A
  qlinearconv     u8 NCHW [32,256,56,56] with a 3x3 (or depthwise) filter
  lstm            bidirectional DynamicQuantizeLSTM, T=512 batch=64 I=H=1024
  qgemm           QGemm of 8-bit codes, M=8192 K=4096 N=14336 (the large GEMM's
                  shape), per-column B parameters, int32 C of shape (1, N)
"""
import numpy as np
import torch


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(g, shape, std, mean=0.0):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean).numpy()


def _uniform(g, shape, lo, hi):
    return (torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo).numpy()


def _randint(g, shape, lo, hi_inclusive, dtype):
    return torch.randint(lo, hi_inclusive + 1, shape, generator=g).numpy().astype(dtype)


def inner_product(seed=0, M=64, N=128, K=256):
    """A fp32 ~N(0,1) [M,K]; constant B fp32 ~N(0,0.05) [K,N]; bias ~U(-0.1,0.1)."""
    g = _gen(seed)
    A = _normal(g, (M, K), 1.0)
    B = _normal(g, (K, N), 0.05)
    bias = _uniform(g, (N,), -0.1, 0.1)
    return {"A": A, "B": B, "bias": bias}


def usage_ramp(M=4, N=8, K=16):
    """Simd usage example: A[i] = i * 0.01f, B[i] = i * 0.02f, bias 0.1 (fp32)."""
    A = (np.arange(M * K, dtype=np.float32) * np.float32(0.01)).reshape(M, K)
    B = (np.arange(K * N, dtype=np.float32) * np.float32(0.02)).reshape(K, N)
    bias = np.full(N, np.float32(0.1), dtype=np.float32)
    return {"A": A, "B": B, "bias": bias}


def qdq(seed=1, shape=(32, 1024, 4096), tie_fraction=0.01):
    """x fp32 ~N(0,2); per-axis (last axis) scales ~U(0.005,0.05) and uint8
    zero points ~U{0..255}; a `tie_fraction` of positions (drawn with
    replacement, duplicates kept once) overwritten with x = fl((k+0.5)*s[c])
    for an integer k with k+zp in [0,254], kept only where fl(x/s[c]) is
    exactly k+0.5 (a true round-half-even tie that does not saturate).
    Also returns the per-tensor int8 variant's scale 0.02 and zero point 0."""
    g = _gen(seed)
    shape = tuple(int(s) for s in shape)
    C = shape[-1]
    x = _normal(g, shape, 2.0).reshape(-1)
    scale = _uniform(g, (C,), 0.005, 0.05)
    zp = _randint(g, (C,), 0, 255, np.uint8)
    n = x.size
    n_ties = int(n * tie_fraction)
    ties = np.zeros(0, dtype=np.int64)
    if n_ties:
        pos = np.unique(torch.randint(0, n, (n_ties,), generator=g).numpy())
        ch = pos % C
        z = zp[ch].astype(np.int64)
        pending = np.ones(pos.size, dtype=bool)
        tie_val = np.zeros(pos.size, dtype=np.float32)
        for _ in range(8):
            idx = np.nonzero(pending)[0]
            if idx.size == 0:
                break
            u = torch.rand(idx.size, generator=g).numpy().astype(np.float64)
            lo, hi = -z[idx], 254 - z[idx]
            k = np.floor(lo + u * (hi - lo + 1)).astype(np.int64)
            k = np.minimum(k, hi)
            half = (k.astype(np.float32) + np.float32(0.5)).astype(np.float32)
            cand = (half * scale[ch[idx]]).astype(np.float32)
            ok = (cand / scale[ch[idx]]).astype(np.float32) == half
            tie_val[idx[ok]] = cand[ok]
            pending[idx[ok]] = False
        keep = ~pending
        ties = pos[keep]
        x[ties] = tie_val[keep]
    return {"x": x.reshape(shape), "scale": scale, "zero_point": zp, "axis": len(shape) - 1,
            "tie_positions": ties, "s8_scale": np.float32(0.02), "s8_zero_point": np.int8(0)}


def bf16_bits(a):
    """Round fp32 to bf16 (round to nearest even, torch's conversion) and
    return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def large_gemm(seed=2, M=8192, K=4096, N=14336, avoid_overflow=False):
    """A bf16 ~N(0,1) with 0.5% of elements scaled x20 (outliers), given as
    bf16 bit patterns [M,K]; bias fp32 ~N(0,0.02) [N].
    avoid_overflow=False: constant B int8 ~U{-128..127} [K,N] with per-column
    scales ~U(1e-3,1e-2).  avoid_overflow=True: B fp32 ~N(0,0.05) [K,N]."""
    g = _gen(seed)
    A = torch.randn((M, K), generator=g, dtype=torch.float32)
    n_out = max(1, int(M * K * 0.005))
    pos = torch.randint(0, M * K, (n_out,), generator=g)
    A.view(-1)[pos] *= 20.0
    A_bits = bf16_bits(A.numpy())
    bias = _normal(g, (N,), 0.02)
    out = {"A_bf16": A_bits, "bias": bias}
    if avoid_overflow:
        out["B"] = _normal(g, (K, N), 0.05)
    else:
        out["iB"] = _randint(g, (K, N), -128, 127, np.int8)
        out["scaleB"] = _uniform(g, (N,), 1e-3, 1e-2)
    return out


def qlinearconv(seed=3, N=32, C=256, H=56, W=56, M=256, k=3, depthwise=False):
    """x u8 ~U{0..255} NCHW, x_scale 0.0037, x_zero_point 132; w u8 ~U{0..255}
    [M, C/group, k, k]; per-channel w_scale ~U(0.001,0.01) and w_zero_point
    ~U{100..156}; bias int32 ~U{-5000..5000}; y_scale 0.05, y_zero_point 128;
    pad k//2, stride 1.  depthwise: group = C and M = C."""
    g = _gen(seed)
    group = C if depthwise else 1
    if depthwise:
        M = C
    x = _randint(g, (N, C, H, W), 0, 255, np.uint8)
    w = _randint(g, (M, C // group, k, k), 0, 255, np.uint8)
    w_scale = _uniform(g, (M,), 0.001, 0.01)
    w_zp = _randint(g, (M,), 100, 156, np.uint8)
    B = _randint(g, (M,), -5000, 5000, np.int32)
    p = k // 2
    return {"x": x, "x_scale": np.float32(0.0037), "x_zero_point": 132, "w": w,
            "w_scale": w_scale, "w_zero_point": w_zp, "y_scale": np.float32(0.05),
            "y_zero_point": 128, "B": B, "pads": (p, p, p, p), "strides": (1, 1), "group": group}


def lstm(seed=4, T=512, batch=64, I=1024, H=1024, D=2):
    """X fp32 ~N(0,1) [T,batch,I]; W int8 [D,I,4H] and R int8 [D,H,4H]
    ~U{-128..127}; per-channel scales ~U(1e-3,5e-3) [D,4H], zero points 0;
    B fp32 ~N(0,0.1) [D,8H]; initial h and c zero."""
    g = _gen(seed)
    X = _normal(g, (T, batch, I), 1.0)
    Wq = _randint(g, (D, I, 4 * H), -128, 127, np.int8)
    Rq = _randint(g, (D, H, 4 * H), -128, 127, np.int8)
    W_scale = _uniform(g, (D, 4 * H), 1e-3, 5e-3)
    R_scale = _uniform(g, (D, 4 * H), 1e-3, 5e-3)
    Bias = _normal(g, (D, 8 * H), 0.1)
    return {"X": X, "W": Wq, "R": Rq, "W_scale": W_scale, "R_scale": R_scale, "B": Bias,
            "W_zero_point": np.zeros((D, 4 * H), np.int8), "R_zero_point": np.zeros((D, 4 * H), np.int8)}


def qgemm(seed=5, M=8192, K=4096, N=14336, atype="u8", btype="s8", per_column=True, c_shape="1N"):
    """8-bit A (M, K) and B (K, N) codes ~U over the type's range; a_scale
    0.02, a_zero_point ~U over A's range; b_scale ~U(1e-3, 1e-2) and
    b_zero_point ~U over B's range, per column (or one of each); C int32
    ~U{-5000..5000} of shape c_shape ("MN", "1N", "N", "M1", "11" or None);
    alpha 1.5; y_scale 0.05 and y_zero_point ~U over the output type's range
    for a quantized output of A's type."""
    g = _gen(seed)
    rng = {"u8": (0, 255, np.uint8), "s8": (-128, 127, np.int8)}
    alo, ahi, adt = rng[atype]
    blo, bhi, bdt = rng[btype]
    nb = N if per_column else 1
    out = {
        "A": _randint(g, (M, K), alo, ahi, adt),
        "B": _randint(g, (K, N), blo, bhi, bdt),
        "a_scale": np.float32(0.02),
        "a_zero_point": int(_randint(g, (1,), alo, ahi, np.int64)[0]),
        "b_scale": _uniform(g, (nb,), 1e-3, 1e-2),
        "b_zero_point": _randint(g, (nb,), blo, bhi, bdt),
        "alpha": np.float32(1.5),
        "y_scale": np.float32(0.05),
        "y_zero_point": int(_randint(g, (1,), alo, ahi, np.int64)[0]),
    }
    shapes = {"MN": (M, N), "1N": (1, N), "N": (N,), "M1": (M, 1), "11": (1, 1), None: None}
    out["C"] = None if c_shape is None else _randint(g, shapes[c_shape], -5000, 5000, np.int32)
    return out
