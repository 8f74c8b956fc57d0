"""The N > 1 host logic of bench.py on CPU: two ranks over gloo, no GPU.

Each rank times its own batch (weak scaling, no collective on the data path);
the reported time is the maximum over ranks and the rate counts every rank's
bytes. Under torchrun the reference arm runs on rank 0 only and the other ranks
exit without work.
"""
import os
import socket
import sys
import types

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, elapsed, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        dist.barrier()
        out[rank] = bench.aggregate_over_ranks(elapsed[rank], 1000, 10, ws, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    ws, port = 2, _free_port()
    elapsed = [10.0, 12.5]  # ms over 10 steps
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(ws, port, elapsed, out), nprocs=ws, start_method="spawn", join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for r in range(ws):
        e, ms_step, gbs = res[r]
        assert e == 12.5 and ms_step == 1.25
        # 1000 bytes per step on each of two ranks, 10 steps, in 12.5 ms
        assert abs(gbs - 2 * 1000 * 10 / 12.5e-3 / 1e9) < 1e-15


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.aggregate_over_ranks(4.0, 500, 2, 1, "cpu") == (4.0, 2.0, 500 * 2 / 4e-3 / 1e9)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    def no_oracle(*a, **k):
        raise AssertionError("a rank other than 0 ran the oracle")

    monkeypatch.setattr(bench, "oracle_step_sample", no_oracle)
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(gpus=2, steps=1, warmup=0, ref_seconds=1.0, workload="softmax_T8192_E2304_k36")
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
