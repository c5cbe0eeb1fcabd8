"""Failure detection on the GPU without a fault: a bounded device wait that
runs out.

The library's waits (mbarrier phases in the tcgen05 pipelines, the grid
barriers of the persistent LSTM recurrence) give up after a time limit,
record a code in the device status word and let the kernel return, so the
host learns of the failure from i8q_sync_status and the context stays
usable.  i8q_debug_wait_timeout runs one such wait, with a limit of a few
milliseconds, on an event that never comes (no TMA copy or MMA is in flight
while it waits).
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import int8_quantized_gb300 as q
from int8_quantized_gb300 import _lib, workloads

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("kind", [0, 1], ids=["mbarrier", "grid_barrier"])
def test_bounded_wait_gives_up_and_reports(orc, dev, kind):
    lib = _lib.load()
    assert lib.i8q_sync_status(_stream()) == 0          # nothing pending before
    t0 = time.perf_counter()
    assert lib.i8q_debug_wait_timeout(kind, 3_000_000, _stream()) == 0, lib.i8q_last_error()
    assert lib.i8q_sync_status(_stream()) == _lib.ERR_DEVICE_TIMEOUT
    assert time.perf_counter() - t0 < 2.0               # gave up after its limit, not the 4 s default
    assert b"bounded wait" in lib.i8q_last_error()
    assert lib.i8q_sync_status(_stream()) == 0          # the report clears the status word
    # the context is still usable: the next product matches the oracle
    w = workloads.inner_product(seed=0)
    ctx = q.QGemmDyn(64, 128, 256, q.F32, q.F32, q.F32, constB=True, bias=True)
    ctx.set_params(torch.from_numpy(w["B"]).to(dev), None, torch.from_numpy(w["bias"]).to(dev))
    C = torch.empty(64, 128, device=dev)
    ctx.forward(torch.from_numpy(w["A"]).to(dev), C)
    q.sync_status()
    ref = orc.dynamic_quantized_inner_product(w["A"], w["B"], bias=w["bias"])["C"]
    assert np.max(np.abs(C.cpu().numpy() - ref) / np.maximum(np.abs(ref), 1e-30)) <= 1e-6
    ctx.clear()


def test_probe_rejects_bad_arguments(dev):
    lib = _lib.load()
    assert lib.i8q_debug_wait_timeout(2, 3_000_000, _stream()) == _lib.ERR_INVALID_ARG
    assert lib.i8q_debug_wait_timeout(0, 10, _stream()) == _lib.ERR_INVALID_ARG
    assert lib.i8q_debug_wait_timeout(0, 5_000_000_000, _stream()) == _lib.ERR_INVALID_ARG
