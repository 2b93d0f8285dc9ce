"""The bench's multi-rank path on the CPU: two `gloo` processes reduce their
timings with `bench.max_over_ranks` (each rank's step time is the slowest
rank's), and the whole-job throughput counts every rank's tokens."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (1 + r) ms per step and (10 - r) ms end to end
        ms, e2e = bench.max_over_ranks([1.0 + rank, 10.0 - rank], torch.device("cpu"))
        out[rank] = (ms, e2e, bench.headline_config(bench.synth.SINGLE_4K, world)["parallelism"])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_processes():
    world = 2
    with mp.Manager() as manager:
        out = manager.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
        got = dict(out)
    assert set(got) == {0, 1}
    for rank in range(world):
        ms, e2e, par = got[rank]
        assert ms == 2.0 and e2e == 10.0  # the slowest rank's time, on every rank
        assert par == "replicas x2"


def test_max_over_ranks_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.5, 1.25], torch.device("cpu")) == [3.5, 1.25]


def test_reference_arm_prints_one_line():
    """`bench.py --impl reference` runs the oracle on the host cores (no GPU)
    and prints one JSON line with the keys the bench's contract names."""
    import json
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["config"]["workload"] == "prefill_long_T131072"
    assert d["ms_per_step"] > 0 and "chains" in d["cpu_baseline"]["sample"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("name", ["LONG_128K", "VARLEN_32K", "SINGLE_4K"])
def test_dram_summaries_match_the_sources(name):
    """Each committed DRAM-traffic summary the bench reports from was taken on
    the chunked prefill's current sources (its sha256 over them matches), its
    kernels add up to the call and the traffic is at least the algorithmic
    bytes; a change to those sources without a new capture fails here."""
    sys.path.insert(0, ROOT)
    import bench
    cfg = getattr(bench.synth, name)
    tr = bench.profiled_traffic(cfg)
    assert tr is not None, f"profiles/dram_{cfg.name}.md is missing or was taken on other sources"
    assert sum(tr["kernels"].values()) == tr["call"]
    nbytes, _ = bench.prefill_work(cfg)
    assert tr["call"] >= nbytes
