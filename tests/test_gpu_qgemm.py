"""Dynamic quantized inner product on the GPU vs the CPU oracle.

Bit-exact: the uint8 codes of A with their scales and zero points, the int8
codes of B with scales and column sums, and the int32 accumulators.  Float
outputs: max relative error <= 1e-6 for fp32 (expected exactly 0: the
epilogue is one fixed sequence of fp32 operations), <= 1 bf16 ulp for bf16
(GELU's erff may differ by an fp32 ulp between the two libraries, which can
move a bf16 rounding by one step).
"""
import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from conftest import bf16_ulp_distance, max_rel_err
from int8_quantized_gb300 import workloads

pytestmark = pytest.mark.gpu

ACT = {"identity": q.ACT_IDENTITY, "relu": q.ACT_RELU, "gelu": q.ACT_GELU}
CORE_INFO = {"imma": "mma.sync", "tc1": "tcgen05", "tc2": "tcgen05", "small": "dp4a"}


@pytest.fixture(params=["imma", "tc1", "tc2", "small"], autouse=True)
def core(request, monkeypatch):
    """Every case runs on each integer core, forced regardless of the shape:
    the int8 mma.sync core, the exact-integer tcgen05 core with single-CTA
    128 x 256 tiles and with CTA-pair 256 x 256 tiles, and the fused
    small-product dp4a kernel."""
    monkeypatch.setenv("I8Q_FORCE_CORE", request.param)
    return request.param


def _t(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _bits(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def run_case(orc, dev, A, B=None, iB=None, scaleB=None, bias=None, act="identity", avoid=False, typeA="f32",
             typeC="f32", constB=True, rows=None, check_codes=True):
    """Run one configuration through the C ABI and compare with the oracle.
    A: fp32 array, or bf16 bit patterns (uint16) when typeA == 'bf16'."""
    M, K = A.shape
    N = (iB if iB is not None else B).shape[1]
    tA = q.BF16 if typeA == "bf16" else q.F32
    tC = q.BF16 if typeC == "bf16" else q.F32
    if iB is not None:
        tB = q.S8
    else:
        tB = q.BF16 if B.dtype == np.uint16 else q.F32
    ctx = q.QGemmDyn(M, N, K, tA, tB, tC, constB=constB, bias=bias is not None, activation=ACT[act],
                     avoidOverflow=avoid)
    import os
    assert CORE_INFO[os.environ["I8Q_FORCE_CORE"]] in ctx.info()
    Ad = _t(A.view(np.int16) if typeA == "bf16" else A, dev)
    if typeA == "bf16":
        Ad = Ad.view(torch.bfloat16)
    bias_d = None if bias is None else _t(bias, dev)
    Bd = None
    if constB:
        if iB is not None:
            ctx.set_params(_t(iB, dev), _t(scaleB, dev), bias_d)
        else:
            ctx.set_params(_t(B, dev), None, bias_d)
    else:
        ctx.set_params(None, None, bias_d)
        Bd = _t(B.view(np.int16), dev).view(torch.bfloat16) if B.dtype == np.uint16 else _t(B, dev)
    assert ctx.enabled()
    buf = torch.empty(ctx.external_buffer_size(), dtype=torch.uint8, device=dev)
    C = torch.empty(M, N, dtype=torch.bfloat16 if typeC == "bf16" else torch.float32, device=dev)
    ctx.forward(Ad, C, B=Bd, buf=buf)
    acc = torch.empty(M, N, dtype=torch.int32, device=dev)
    ctx.forward_s32(Ad, acc, B=Bd, buf=buf)
    q.sync_status()

    A_rows = A if rows is None else A[rows]
    ref = orc.dynamic_quantized_inner_product(A_rows, B, iB=iB, scaleB=scaleB, bias=bias, act=orc.__dict__[
        "ACT_" + act.upper()], avoid_overflow=avoid, typeC="bf16" if typeC == "bf16" else "f32")
    sel = slice(None) if rows is None else rows
    if check_codes:
        uA, sA, zA, lda = ctx.buf_views(buf)
        assert np.array_equal(uA.cpu().numpy()[sel, :K], ref["uA"])
        assert np.all(uA.cpu().numpy()[sel, K:] == 0)
        assert np.array_equal(sA.cpu().numpy()[sel], ref["scaleA"])
        assert np.array_equal(zA.cpu().numpy()[sel], ref["zeroA"])
        # B's codes, scales and column sums: stored by SetParams (constant B)
        # or written by this Forward into buf (B quantized per call)
        iBt, sB, cs, ldb = ctx.weight_views(None if constB else buf)
        assert np.array_equal(iBt.cpu().numpy()[:, :K], ref["iB"].T)
        assert np.all(iBt.cpu().numpy()[:, K:] == 0)
        assert np.array_equal(sB.cpu().numpy(), ref["scaleB"])
        assert np.array_equal(cs.cpu().numpy(), ref["iB"].astype(np.int64).sum(0))
    assert np.array_equal(acc.cpu().numpy()[sel], ref["acc"])
    if typeC == "bf16":
        d = bf16_ulp_distance(_bits(C)[sel], ref["C"])
        assert d.max() <= 1, f"bf16 ulp distance {d.max()}"
    else:
        err = max_rel_err(C.cpu().numpy()[sel], ref["C"])
        if act == "gelu":
            # erfcf of the two libraries may differ by a few ulps; below the
            # fp32 normal range that is an absolute difference
            got = C.cpu().numpy()[sel].astype(np.float64)
            r = ref["C"].astype(np.float64)
            assert np.all(np.abs(got - r) <= 1e-6 * np.abs(r) + 1e-37), f"max rel err {err}"
        else:
            assert err <= 1e-6, f"max rel err {err}"
    ctx.clear()
    return ref


def test_inner_product_workload(orc, dev):
    """M=64 N=128 K=256, fp32, constant fp32 B quantized by SetParams."""
    w = workloads.inner_product(seed=0)
    run_case(orc, dev, w["A"], w["B"], bias=w["bias"])


@pytest.mark.parametrize("avoid", [True, False])
def test_usage_ramp_example(orc, dev, avoid):
    w = workloads.usage_ramp()
    run_case(orc, dev, w["A"], w["B"], bias=w["bias"], avoid=avoid)


SHAPES = [(1, 1, 1), (1, 7, 3), (7, 13, 63), (63, 65, 64), (129, 130, 129), (200, 300, 1000), (256, 256, 512),
          (33, 520, 4100)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_ragged_shapes_fp32_constB(orc, dev, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    B = rng.normal(0, 0.05, (K, N)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, N).astype(np.float32)
    run_case(orc, dev, A, B, bias=bias)


@pytest.mark.parametrize("act", ["identity", "relu", "gelu"])
@pytest.mark.parametrize("typeA,typeC", [("bf16", "bf16"), ("f32", "bf16"), ("bf16", "f32")])
def test_types_and_activations_int8_B(orc, dev, act, typeA, typeC):
    rng = np.random.default_rng(11)
    M, N, K = 150, 200, 320
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    if typeA == "bf16":
        A = workloads.bf16_bits(A)
    iB = rng.integers(-128, 128, (K, N)).astype(np.int8)
    sB = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = rng.normal(0, 0.02, N).astype(np.float32)
    run_case(orc, dev, A, iB=iB, scaleB=sB, bias=bias, act=act, typeA=typeA, typeC=typeC)


@pytest.mark.parametrize("typeC", ["bf16", "f32"])
def test_gelu_over_its_whole_range(orc, dev, typeC):
    """With every B code zero the sum is 0 and each output is GELU(bias[j])
    exactly, so the bias sweeps the activation's input: [-20, 20] densely,
    the negative tail where GELU falls through the bf16 subnormals to zero,
    tiny and subnormal magnitudes of both signs, and huge ones."""
    rng = np.random.default_rng(21)
    xs = np.concatenate([np.linspace(-20, 20, 8001), -np.geomspace(12.5, 14.5, 2001),
                         np.geomspace(1e-44, 1e-3, 401), -np.geomspace(1e-44, 1e-3, 401),
                         [0.0, -0.0, 1e30, -1e30, 3e38, -3e38]]).astype(np.float32)
    M, K, N = 256, 64, xs.size
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    iB = np.zeros((K, N), np.int8)
    sB = np.ones(N, np.float32)
    run_case(orc, dev, A, iB=iB, scaleB=sB, bias=xs, act="gelu", typeC=typeC, check_codes=False)


@pytest.mark.parametrize("path", ["strip", "two_pass"])
@pytest.mark.parametrize("Btype", ["f32", "bf16"])
@pytest.mark.parametrize("K,N", [(300, 104), (1000, 200), (520, 64)])
def test_column_quantization_paths(orc, dev, monkeypatch, path, Btype, K, N):
    """B quantized per column inside Forward by the one-read strip kernel
    (TMA boxes past K and strips past N read as zero) and by the two-pass
    kernels, with K not a multiple of the 256-row box and N not a multiple
    of the strip width."""
    if path == "two_pass":
        monkeypatch.setenv("I8Q_COLS_TWO_PASS", "1")
    rng = np.random.default_rng(K + N)
    A = rng.normal(0, 1, (40, K)).astype(np.float32)
    B = rng.normal(0, 0.05, (K, N)).astype(np.float32)
    B[:, 3] = 0.0  # a zero column: scale 1
    if Btype == "bf16":
        B = workloads.bf16_bits(B)
    run_case(orc, dev, A, B, bias=None, avoid=True, constB=False)


@pytest.mark.parametrize("Btype", ["f32", "bf16"])
@pytest.mark.parametrize("avoid", [False, True])
def test_non_constant_B(orc, dev, Btype, avoid):
    rng = np.random.default_rng(5)
    M, N, K = 96, 160, 200
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    B = rng.normal(0, 0.05, (K, N)).astype(np.float32)
    if Btype == "bf16":
        B = workloads.bf16_bits(B)
    run_case(orc, dev, A, B, bias=None, avoid=avoid, constB=False)


def test_edge_rows_and_columns(orc, dev):
    rng = np.random.default_rng(9)
    M, N, K = 40, 70, 130
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    A[0] = 0.0                        # degenerate row
    A[1] = 3.0                        # constant positive row
    A[2] = -2.5                       # constant negative row
    A[3] = np.abs(A[3])               # zero point 0
    A[4] = -np.abs(A[4])              # zero point 255
    A[5, 7] = 1e4                     # one huge outlier
    A[6] = 1e-30                      # tiny values
    B = rng.normal(0, 0.05, (K, N)).astype(np.float32)
    B[:, 0] = 0.0                     # degenerate column
    B[:, 1] = -0.3                    # constant column
    run_case(orc, dev, A, B, bias=rng.uniform(-1, 1, N).astype(np.float32), act="relu")


def test_worst_case_accumulator_magnitude(orc, dev):
    """Every product at its extreme: uA - zeroA = 255 or -255 with iB = -128,
    K = 4096 (|sum| close to 2^27)."""
    M, N, K = 16, 64, 4096
    A = np.zeros((M, K), np.float32)
    A[0::2] = 1.0                     # all max: zero point 0, codes 255
    A[1::2] = -1.0                    # all min: zero point 255, codes 0
    iB = np.full((K, N), -128, np.int8)
    iB[:, 1::2] = 127
    run_case(orc, dev, A, iB=iB, scaleB=np.full(N, 1e-3, np.float32), bias=None)


def test_worst_case_accumulator_narrow_range(orc, dev):
    """avoidOverflow with non-constant B: codes 255 x +-63 in every product,
    K = 3000 (the tensor-core core sums 1024 of them in fp32 per chunk,
    reaching 1024 * 16065 < 2^24)."""
    M, N, K = 8, 300, 3000
    A = np.ones((M, K), np.float32)
    A[1::2] = -np.ones(K, np.float32)
    B = np.full((K, N), 0.7, np.float32)
    B[:, ::3] = -0.7
    run_case(orc, dev, A, B, bias=None, avoid=True, constB=False)


@pytest.mark.parametrize("K", [511, 512, 513, 1025, 2048 + 64])
def test_chunk_boundaries(orc, dev, K):
    rng = np.random.default_rng(K)
    M, N = 130, 260
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    iB = rng.integers(-128, 128, (K, N)).astype(np.int8)
    run_case(orc, dev, A, iB=iB, scaleB=rng.uniform(1e-3, 1e-2, N).astype(np.float32), bias=None)


@pytest.mark.parametrize("register", [False, True])
@pytest.mark.parametrize("typeA,K,M", [("f32", 2056, 1237), ("f32", 3200, 1300), ("bf16", 4104, 1237),
                                       ("f32", 4104, 701), ("bf16", 2048, 1300), ("f32", 1024, 1237),
                                       ("f32", 6408, 640)])
def test_row_quantization_forms(orc, dev, core, monkeypatch, register, typeA, K, M):
    """Rows of A long enough for the shared-memory staged form (more than
    2048 elements, at least 152 groups of 4 rows, a ragged last group),
    shorter ones that take the register form, fp32 rows of 6408 too long for
    either (CTA per row), each also forced to the register form or its
    fallback: codes, scales and zero points of sampled rows."""
    if core != "tc2":
        pytest.skip("row quantization does not depend on the integer core")
    if register:
        monkeypatch.setenv("I8Q_ROWS_REGISTER", "1")
    rng = np.random.default_rng(K + M)
    A = rng.normal(0, 1, (M, K)).astype(np.float32)
    A[::5, ::7] *= 40.0
    A[3] = 0.0
    if typeA == "bf16":
        A = (A.view(np.uint32) >> 16).astype(np.uint16)
    iB = rng.integers(-128, 128, (K, 32)).astype(np.int8)
    run_case(orc, dev, A, iB=iB, scaleB=rng.uniform(1e-3, 1e-2, 32).astype(np.float32), bias=None, typeA=typeA,
             rows=np.array([0, 3, 5, 600, M - 2, M - 1]))


@pytest.mark.parametrize("register", [False, True])
@pytest.mark.parametrize("typeA", ["f32", "bf16"])
def test_row_quantization_ties(orc, dev, core, monkeypatch, register, typeA):
    """Rows spanning exactly [0, 255 * s] (scale s, zero point 0) with inputs
    at (j + 1/2) * s: every quotient a tie (round half to even decides), a
    third of the rows just beside one; rows long enough for the staged form
    and enough of them for a full wave, or forced to the register form."""
    if core != "tc2":
        pytest.skip("row quantization does not depend on the integer core")
    if register:
        monkeypatch.setenv("I8Q_ROWS_REGISTER", "1")
    rng = np.random.default_rng(31)
    M, K = 700, 2056
    s = np.where(np.arange(M) % 2 == 0, 1.0, 0.5).astype(np.float32)[:, None]
    j = rng.integers(0, 255, (M, K)).astype(np.float32)
    A = ((j + 0.5) * s).astype(np.float32)
    A[1::3] = np.nextafter(A[1::3], np.float32(0))
    A[:, 0], A[:, 1] = 0.0, (255.0 * s[:, 0]).astype(np.float32)
    if typeA == "bf16":
        # bf16 holds j + 1/2 exactly only below 128: keep those rows' codes small
        A = np.where(j < 127, A, (0.5 * s).astype(np.float32))
        A[:, 0], A[:, 1] = 0.0, (255.0 * s[:, 0]).astype(np.float32)
        A = (A.view(np.uint32) >> 16).astype(np.uint16)
    iB = rng.integers(-128, 128, (K, 32)).astype(np.int8)
    run_case(orc, dev, A, iB=iB, scaleB=rng.uniform(1e-3, 1e-2, 32).astype(np.float32), bias=None, typeA=typeA,
             rows=np.array([0, 1, 2, 3, 350, M - 2, M - 1]))


@pytest.mark.parametrize("M,N,K,expect", [(64, 128, 256, "dp4a"), (1, 7, 3, "dp4a"), (8192, 14336, 4096, "tcgen05"),
                                          (64, 1024, 4096, "tcgen05"), (64, 128, 10000, "tcgen05")])
def test_default_core_choice(monkeypatch, core, M, N, K, expect):
    """Without the override, small products take the fused dp4a kernel and
    the rest the tensor-core path."""
    if core != "tc1":
        pytest.skip("the default choice does not depend on the forced core")
    monkeypatch.delenv("I8Q_FORCE_CORE")
    ctx = q.QGemmDyn(M, N, K, constB=True, bias=False)
    assert expect in ctx.info()
    ctx.clear()


def test_context_reinit_and_errors(orc, dev):
    ctx = q.QGemmDyn(8, 16, 32, constB=True, bias=False)
    first = ctx._ctx.value
    ctx.init(8, 16, 32, constB=True, bias=False)           # unchanged: kept
    assert ctx._ctx.value == first
    assert not ctx.enabled()                                # SetParams not called
    C = torch.empty(8, 16, device=dev)
    with pytest.raises(q.I8QError) as e:
        ctx.forward(torch.zeros(8, 32, device=dev), C)
    assert e.value.code == -3
    ctx.init(8, 16, 64, constB=True, bias=False)           # changed: recreated
    assert ctx.internal_buffer_size() > 0 and ctx.external_buffer_size() > 0
    ctx.clear()


def test_forward_host_buffers(orc, dev):
    w = workloads.inner_product(seed=0)
    ctx = q.QGemmDyn(64, 128, 256, constB=True, bias=True)
    ctx.set_params(_t(w["B"], dev), None, _t(w["bias"], dev))
    A = torch.from_numpy(w["A"]).pin_memory()
    C = torch.empty(64, 128, dtype=torch.float32).pin_memory()
    ctx.forward_host(A, C)
    ref = orc.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"])
    assert max_rel_err(C.numpy(), ref["C"]) <= 1e-6
    ctx.clear()


@pytest.mark.parametrize("M", [2048, 5000])
def test_forward_host_pipelined_rows(orc, dev, M):
    """Large host-buffer calls run as a pipeline over row chunks (the last
    one ragged at M=5000): the result equals the device-buffer Forward bit
    for bit, and the oracle on sampled rows."""
    rng = np.random.default_rng(M)
    K, N = 384, 520
    A = workloads.bf16_bits(rng.normal(0, 1, (M, K)).astype(np.float32))
    iB = rng.integers(-128, 128, (K, N)).astype(np.int8)
    sB = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
    bias = rng.normal(0, 0.02, N).astype(np.float32)
    ctx = q.QGemmDyn(M, N, K, q.BF16, q.S8, q.BF16, constB=True, bias=True, activation=q.ACT_GELU)
    ctx.set_params(_t(iB, dev), _t(sB, dev), _t(bias, dev))
    Ah = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).pin_memory()
    Ch = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    Cd = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    # calls 1 (direct), 2 (captured as a graph) and 3, 4 (graph replays)
    # with the same host buffers; A changes before each of the later calls,
    # so every replay must read the buffer's current contents
    for call in range(4):
        if call:
            Ah.copy_(torch.from_numpy(np.roll(A, 37 * call, axis=0).view(np.int16)).view(torch.bfloat16))
        Ch.fill_(0)
        ctx.forward_host(Ah, Ch)
        ctx.forward(Ah.to(dev), Cd)
        q.sync_status()
        assert torch.equal(Ch.view(torch.int16), Cd.cpu().view(torch.int16)), f"call {call}"
    rows = np.array([0, 1, 1023, 1024, M // 2, M - 2, M - 1])
    A_last = np.roll(A, 37 * 3, axis=0)
    ref = orc.dynamic_quantized_inner_product(A_last[rows], iB=iB, scaleB=sB, bias=bias, act=orc.ACT_GELU,
                                              typeC="bf16")
    d = bf16_ulp_distance(Ch.view(torch.int16).numpy().view(np.uint16)[rows], ref["C"])
    assert d.max() <= 1
    # new parameters invalidate the captured pipeline
    ctx.set_params(_t(-iB, dev), _t(sB, dev), _t(bias, dev))
    ctx.forward_host(Ah, Ch)
    ctx.forward(Ah.to(dev), Cd)
    q.sync_status()
    assert torch.equal(Ch.view(torch.int16), Cd.cpu().view(torch.int16)), "after SetParams"
    ctx.clear()


SAMPLE_ROWS = np.array([0, 1, 2, 777, 1024, 3000, 4095, 4096, 5001, 6666, 8190, 8191])


def test_large_gemm_constant_int8_B(orc, dev):
    """M=8192 K=4096 N=14336, bf16 A with outliers, constant int8 B, GELU,
    bf16 C: all codes of A compared, output rows sampled."""
    w = workloads.large_gemm(seed=2)
    run_case(orc, dev, w["A_bf16"], iB=w["iB"], scaleB=w["scaleB"], bias=w["bias"], act="gelu", typeA="bf16",
             typeC="bf16", rows=SAMPLE_ROWS, check_codes=True)


def test_large_gemm_avoid_overflow(orc, dev):
    """Same shape with non-constant fp32 B quantized in Forward to [-64,63]."""
    w = workloads.large_gemm(seed=2, avoid_overflow=True)
    run_case(orc, dev, w["A_bf16"], w["B"], bias=w["bias"], act="gelu", typeA="bf16", typeC="bf16", avoid=True,
             constB=False, rows=SAMPLE_ROWS[::2], check_codes=True)
