"""The N > 1 path of bench.py on the CPU: two gloo ranks, each timing its own
replica, combine into one whole-job throughput (max time over ranks)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, _ = bench.dist_info()
    seconds = 1.0 + rank  # rank 1 is the slow one
    value, t = bench.aggregate(seconds, 100.0, w, device=None)
    bench.barrier(w)
    q.put((r, w, value, t))
    dist.destroy_process_group()


def test_two_rank_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    for _, _, value, t in out:
        assert t == pytest.approx(2.0)          # max over ranks
        assert value == pytest.approx(100.0)    # 2 ranks x 100 units / 2 s


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--workload", "tiny", "--steps", "3",
                                          "--warmup", "3"]))
    assert capsys.readouterr().out == ""
