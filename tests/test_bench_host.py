"""Host-side logic of bench.py without a GPU: the max/sum over ranks used for multi-GPU runs
(world size 2 over gloo on 127.0.0.1), and the reference arm's JSON line."""
import dataclasses
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mx = bench.reduce_max(float(rank + 1) * 1.5, world)
    sm = bench.reduce_sum(float(rank + 1), world)
    bench.barrier(world)
    out[rank] = (mx, sm)
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == (3.0, 3.0) and out[1] == (3.0, 3.0)


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.5, 1) == 2.5 and bench.reduce_sum(4.0, 1) == 4.0


def test_reference_arm_line(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    import synth
    small = dataclasses.replace(synth.WORKLOADS["gdn4k"], B=1, T=128, H=2)
    monkeypatch.setitem(synth.WORKLOADS, "gdn4k", small)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                                      "--ref-chains", "2"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["higher_is_better"] is True and line["metric"] == bench.METRIC


def test_reference_arm_other_ranks_are_silent(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference"])
    bench.main()
    assert capsys.readouterr().out.strip() == ""


def test_warmup_below_three_is_rejected(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py", "--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.main()
