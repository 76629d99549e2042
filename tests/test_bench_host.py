"""Host-side logic of bench.py (no GPU): multi-rank aggregation over two
gloo ranks, per-rank sharding, clock-sample parsing, and the reference arm
(the fp64 oracle) end to end on the tiny workload."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t, u = bench.aggregate(elapsed_s=1.0 + rank, units=10 * (rank + 1), world=world)
    q.put((rank, t, u, bench.shard_seed(0, rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, u, seed in res:
        assert t == 2.0            # slowest rank's time
        assert u == 30.0           # all ranks' units
    assert res[0][3] != res[1][3]  # each rank verifies its own batch


def test_aggregate_single_rank_identity():
    assert bench.aggregate(1.5, 7, world=1) == (1.5, 7)


def test_clock_summary_parsing():
    s = bench.ClockSampler(0)
    s.samples = [(1.0, "0, 1900, 2070, 800.5, 0x0, Not Active, Not Active, Not Active, Not Active"),
                 (2.0, "0, 1950, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active"),
                 (9.0, "0, 500, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active")]
    s.mark(0.5, 2.5)
    out = s.summary()
    assert out["sm_mhz"] == 1925.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "0", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "calls/s"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_greedy_and_tree_modes():
    for extra in (["--workload", "3", "--greedy"], ["--workload", "4"]):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--steps", "2", "--warmup", "3"] + extra,
                           capture_output=True, text=True, timeout=600, cwd=ROOT)
        assert r.returncode == 0, r.stderr
        d = json.loads(r.stdout.strip().splitlines()[-1])
        assert d["value"] > 0 and d["config"]["mode"] in ("greedy", "tree")


def test_profiled_traffic_follows_its_kernel_sources(tmp_path, monkeypatch):
    """A profile's DRAM bytes (profiles/traffic.json) are reported only while
    the code of the kernel it was taken on is unchanged (each profiled kernel
    has its own source list; comments do not count); the committed entries
    name kernels the bench knows and summaries that exist."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        committed = json.load(f)
    for (workload, mode), name in bench.PROFILE_NAMES.items():
        assert name in committed
    for name, entry in committed.items():
        assert entry["kernel"] in bench.KERNEL_SOURCES
        assert os.path.exists(os.path.join(ROOT, entry["summary"])), name
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for kind, files in bench.KERNEL_SOURCES.items():
        for rel in files:
            src = tmp_path / rel
            src.parent.mkdir(parents=True, exist_ok=True)
            src.write_text("// %s\nint f_%d;\n" % (rel, len(rel)))
    h = bench.kernel_source_hash("filter")
    assert h != bench.kernel_source_hash("stream")
    # an edit to comments alone keeps the hash; an edit to code changes it
    src = tmp_path / bench.KERNEL_SOURCES["filter"][0]
    src.write_text("// reworded\n" + src.read_text() + "   // and more\n\n")
    assert bench.kernel_source_hash("filter") == h
    (prof / "traffic.json").write_text(json.dumps(
        {"p": {"kernel": "filter", "kernel_source_hash": h, "dram_bytes_per_launch": 1234},
         "q": {"kernel": "stream", "kernel_source_hash": h, "dram_bytes_per_launch": 99}}))
    assert bench.profiled_traffic("p") == 1234
    assert bench.profiled_traffic("q") is None  # another kernel's sources
    (tmp_path / bench.KERNEL_SOURCES["filter"][0]).write_text("int changed;\n")
    assert bench.profiled_traffic("p") is None  # the kernel changed since
    assert bench.profiled_traffic(None) is None and bench.profiled_traffic("nope") is None


def test_input_sets_exceed_l2():
    """Rotating input sets: a set comes back only after more than twice the
    L2 of other inputs (2 sets when one is larger than L2, else at least 4)."""
    for nbytes in (114688, 99 * 2**20, 115 * 2**20, 124928000, 467140608):
        n = bench.n_input_sets(nbytes)
        assert n >= 2 and (nbytes > bench.L2_BYTES or n >= 4)
        assert (n - 1) * nbytes >= (2 * bench.L2_BYTES if nbytes <= bench.L2_BYTES else nbytes)
    assert bench.per_graph_for(20, 100) == 20 and bench.per_graph_for(20000, 100) == 100
    assert bench.per_graph_for(7, 100) == 7 and bench.per_graph_for(101, 100) == 1
