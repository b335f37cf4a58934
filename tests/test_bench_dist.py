"""bench.py's multi-rank path on CPU: two gloo ranks, max-over-ranks timing, and the
reference arm printing one line from rank 0 only."""
import contextlib
import io
import json
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, outdir: str):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        w, r, _ = bench.dist_init()
        assert (w, r) == (world, rank)
        got = bench.max_over_ranks(float(rank + 1), w, "cpu")
        bench.barrier(w)
        bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3"])
    with open(os.path.join(outdir, f"rank{rank}.txt"), "w") as f:
        f.write(json.dumps({"max": got, "stdout": buf.getvalue()}))


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.loads(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert res[0]["max"] == res[1]["max"] == 2.0
    lines = [l for l in res[0]["stdout"].splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    # the same workload, data and metric as the library's arm prints by default
    assert line["config"]["workload"] == bench.WORKLOAD and line["data"] == bench.DATA
    assert line["metric"] == bench.METRIC and line["unit"] == "steps/s"
    assert line["e2e"]["h2d_bytes_per_step"] == line["e2e"]["d2h_bytes_per_step"] == 0
    assert not [l for l in res[1]["stdout"].splitlines() if l.startswith("{")]
