"""The multi-GPU host path of bench.py on CPU: two replica processes joined over gloo
(world size 2, 127.0.0.1). The decode step does not shard, so N GPUs run N independent
replicas; what crosses ranks is only the timing: the slowest replica's elapsed time
(max over ranks), the whole-job value (all ranks' tokens over that time), and one JSON
line from rank 0 alone. The reference arm does its work on rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    r, w, local, dist = bench.init_replicas(backend="gloo")
    res = {"rank": r, "world": w, "local": local, "joined": dist is not None}
    # each replica reports its own elapsed time; the job is as slow as the slowest
    elapsed = 100.0 + 50.0 * rank
    res["max_elapsed"] = bench.max_over_ranks(elapsed, dist)
    res["value"] = bench.whole_job_value(w, 8, 64, res["max_elapsed"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.emit({"metric": "m", "value": res["value"], "n_gpus": w}, r)
        if r != 0:
            # the reference arm returns at once on ranks other than 0
            bench.reference_arm(None, r, w)
    res["stdout"] = buf.getvalue()
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_replicas_time_max_value_and_single_line(tmp_path):
    world = 2
    tmp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert x["rank"] == r and x["world"] == world and x["local"] == r and x["joined"]
        assert x["max_elapsed"] == 150.0  # the slower replica's time, on every rank
        assert x["value"] == pytest.approx(world * 8 * 64 / 0.150)
    line = json.loads(res[0]["stdout"])
    assert line["n_gpus"] == world and line["value"] == pytest.approx(res[0]["value"])
    assert res[1]["stdout"] == ""


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    rank, world, local, dist = bench.init_replicas()
    assert (rank, world, local, dist) == (0, 1, 0, None)
    assert bench.max_over_ranks(12.5, None) == 12.5
    assert bench.whole_job_value(1, 1, 100, 250.0) == pytest.approx(400.0)
