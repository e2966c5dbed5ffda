"""The multi-process side of bench.py on CPU: two gloo ranks (spawned
processes, rendezvous on 127.0.0.1).  The path shards by batch with no data
exchange, so what there is to check is the harness: the barrier, the max over
ranks of the timed region, each rank's own inputs, the whole-job rate, and
that only rank 0 of the reference arm prints its line."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    from vision_transformer_shifted_gb300.inputs import WORKLOADS, generate
    r, wsize, local, dist = bench.dist_setup(world)
    assert (r, wsize, local) == (rank, world, rank) and dist.get_backend() == "gloo"
    bench.barrier(dist)
    # the timed region's time is the slowest rank's
    assert bench.max_over_ranks(10.0 + 5.0 * rank, dist) == 10.0 + 5.0 * (world - 1)
    # each rank draws its own inputs of the same shapes
    w = bench.rank_workload(WORKLOADS["tiny"], rank)
    x = generate(w)["x"]
    xs = [torch.zeros_like(x) for _ in range(world)]
    dist.all_gather(xs, x)
    assert all(xs[i].shape == x.shape for i in range(world))
    assert not torch.equal(xs[0], xs[1])
    # whole-job rate: all ranks' tokens over the slowest time
    assert bench.job_rate(w.tokens, world, 2.0) == w.tokens * world / 2.0
    # the reference arm: rank 0 alone prints its line (the others return at once)
    import contextlib
    import io

    class Args:
        gpus, steps, warmup, ref_seconds = world, 1, 0, 0.2

    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args, WORKLOADS["tiny"])
    with open(os.path.join(outdir, "rank%d.txt" % rank), "w") as f:
        f.write(buf.getvalue())
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    if sys.platform != "linux":
        pytest.skip("spawned gloo ranks are tested on Linux")
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    lines = [open(tmp_path / ("rank%d.txt" % r)).read().strip() for r in range(world)]
    assert lines[1] == ""
    d = json.loads(lines[0].splitlines()[-1])
    assert d["impl"] == "reference" and d["n_gpus"] == world and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_stored_traffic_is_reported_only_for_the_source_it_was_taken_on(monkeypatch):
    """bench.py's roofline.traffic comes from ncu counters stored with the sha1
    prefix of the kernel source they were taken on: it is reported while that
    source is unchanged and null once it has changed (or the file is gone),
    and every stored entry names an existing source file."""
    import hashlib
    sys.path.insert(0, ROOT)
    import bench
    csrc = os.path.join(ROOT, "vision_transformer_shifted_gb300", "csrc")
    for (_wl, _k), (traffic, fname, _sha) in bench.PROFILED_TRAFFIC.items():
        assert traffic > 0 and os.path.exists(os.path.join(csrc, fname)), fname
    sha = hashlib.sha1(open(os.path.join(csrc, "attn_window.cu"), "rb").read()).hexdigest()[:12]
    monkeypatch.setattr(bench, "PROFILED_TRAFFIC", {
        ("w", "same"): (1.0e6, "attn_window.cu", sha),
        ("w", "changed"): (1.0e6, "attn_window.cu", "000000000000"),
        ("w", "gone"): (1.0e6, "no_such_file.cu", sha),
    })
    assert bench.profiled_traffic("w", "same") == 1.0e6
    assert bench.profiled_traffic("w", "changed") is None
    assert bench.profiled_traffic("w", "gone") is None
    assert bench.profiled_traffic("w", "absent") is None
