"""Host-side logic of bench.py (CPU only): the multi-rank plumbing over world_size-2 gloo
process groups, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist(world)
    d.barrier()
    mx = d.max(float(10 + rank))
    q.put((rank, d.world, mx))
    d.close()


def test_two_rank_gloo_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2, 11.0), (1, 2, 11.0)]


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-tokens", "8"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["metric"].startswith("TP-sharded MLP fwd+bwd")


def test_reference_arm_takes_every_core_when_launched_with_one_thread():
    # torchrun hands every rank OMP_NUM_THREADS=1; rank 0 of the reference arm runs the oracle alone
    # and must report (and use) every usable core.
    env = dict(os.environ, OMP_NUM_THREADS="1", RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--cpu-tokens", "8"], capture_output=True, text=True, timeout=600,
                       env=env)
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][0])
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))


def test_cpu_cores_honours_omp_num_threads(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("OMP_NUM_THREADS", "1")
    assert bench.cpu_cores() == 1
    monkeypatch.delenv("OMP_NUM_THREADS")
    assert bench.cpu_cores() == len(os.sched_getaffinity(0))


def test_peak_follows_the_clocks_of_the_window():
    sys.path.insert(0, ROOT)
    import bench
    pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1950.0, "bf16_tflops_sustained": 1718.0, "sm_max_mhz": 2070.0,
          "source": "measured"}
    assert bench.tensor_peak(pk, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})[0] == 1950.0
    assert bench.tensor_peak(pk, {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0})[0] == 1950.0
    assert bench.tensor_peak(pk, {"sm_mhz": 1460.0, "sm_max_mhz": 2070.0})[0] == 1718.0
    assert bench.tensor_peak(pk, {"sm_mhz": None, "sm_max_mhz": None})[0] == 1718.0
    r = bench.roofline("tensor", "k", 1500.0, pk, {"sm_mhz": 1800.0, "sm_max_mhz": 2070.0})
    assert r["peak"] == 1718.0 and r["frac"] == round(1500.0 / 1718.0, 4)
    assert r["achieved_at_max_clock"] == round(1500.0 * 2070.0 / 1800.0, 1)
    comp = {"a": bench.pending("hbm", "x", 3400.0), "b": {"c": bench.pending("tensor", "y", 975.0)}}
    bench.finish_rooflines(comp, pk, {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0})
    assert comp["a"]["frac"] == 0.5 and comp["a"]["unit"] == "GB/s"
    assert comp["b"]["c"]["frac"] == 0.5 and comp["b"]["c"]["unit"] == "TFLOP/s"


def test_clock_windows_select_samples_by_time():
    sys.path.insert(0, ROOT)
    import bench
    c = bench.Clocks(0)
    c.p = object()          # as if nvidia-smi had run
    c.samples = [(10.0, 2070.0, 2070.0, set()), (10.1, 2070.0, 2070.0, set()),
                 (20.0, 1500.0, 2070.0, {"sw_power_cap"}), (20.1, 1400.0, 2070.0, {"sw_power_cap"})]
    w = c.window(9.9, 10.2)
    assert w["sm_mhz"] == 2070.0 and w["samples"] == 2 and w["reasons"] == []
    w = c.window(19.0, 21.0)
    assert w["sm_mhz"] == 1450.0 and w["reasons"] == ["sw_power_cap"]
    import os as _os
    _os.unlink(c.f.name)
