"""bench.py's multi-rank host logic on CPU with two gloo ranks: the step time
is the max over ranks, the value counts every rank's work (weak scaling),
and only rank 0 of the reference arm does any work."""
import os
import socket

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = 1.0 + rank                          # rank 1 is the slow one
    m = bench.reduce_max(secs, world)
    bench.barrier(world)
    value = bench.weak_scaling_value(100.0, 4, world, m)
    out.put((rank, m, value))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, value in res:
        assert m == 2.0                          # max of 1.0 and 2.0 on every rank
        assert value == pytest.approx(100.0 * 4 * 2 / 2.0)


def test_reference_arm_only_rank0_works(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_rows_selection(monkeypatch):
    """--rows times only the named hot-path workloads (the row functions are
    stubbed: no GPU work)."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    called = []
    for name in ("_row_avoid_overflow", "_row_inner_product", "_row_qgemm_family", "_row_qlinear_ew", "_row_lstm"):
        monkeypatch.setattr(bench, name, lambda *a, _n=name, **k: called.append(_n))
    monkeypatch.setattr(bench, "_row_qlinearconv", lambda *a, **k: called.append("conv_dw" if a[-1] else "conv_dense"))
    args = bench.parse_args(["--rows", "qlinearconv_depthwise,dq_lstm_bidirectional"])
    bench.measure_rows(args, None, None, 1)
    assert called == ["conv_dw", "_row_lstm"]
    called.clear()
    bench.measure_rows(bench.parse_args([]), None, None, 1)
    assert called == ["_row_avoid_overflow", "_row_inner_product", "conv_dense", "conv_dw", "_row_qgemm_family",
                      "_row_qlinear_ew", "_row_lstm"]
    called.clear()
    bench.measure_rows(bench.parse_args(["--rows", "matmul_integer_to_float"]), None, None, 1)
    assert called == ["_row_qgemm_family"]
