"""Host-side logic of bench.py on CPU: the N > 1 replica path over gloo with
world size 2, and the CPU reference arm (the fp64 oracle) end to end."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    t = bench.barrier_max(10.0 + 5.0 * rank, w, torch.device("cpu"))
    v = bench.replica_throughput(8192, 20, w, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, r, w, lr, t, v))


def test_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, r, w, lr, t, v in out:
        assert (r, w, lr) == (rank, 2, rank)
        assert t == 15.0                                   # max over ranks, in ms
        assert v == pytest.approx(8192 * 2 * 20 / 0.015)   # both replicas' tokens / slowest time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.barrier_max(3.0, 1, torch.device("cpu")) == 3.0
    assert bench.replica_throughput(10, 5, 1, 1000.0) == 50.0


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       capture_output=True, text=True, timeout=120, env=env, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_profiled_traffic_matches_the_summaries_and_is_dropped_after_an_edit():
    sys.path.insert(0, ROOT)
    import bench
    for kernel, e in bench.PROFILED_TRAFFIC.items():
        text = open(os.path.join(ROOT, e["profile"])).read()
        for mb in (e["read_mb"], e["write_mb"]):
            assert f"{mb:.1f} MB" in text, (kernel, mb)           # the figure the summary shows
        assert kernel.split("_kernel")[0] in text
    # a source that no longer hashes to the recorded prefix voids the entry
    e = dict(bench.PROFILED_TRAFFIC["kda_tc_prep"])
    e["sources"] = dict(e["sources"], **{"csrc/prefill_tc.cu": "0000000000000000"})
    traffic, why = bench.profiled_traffic("kda_tc_prep", {"kda_tc_prep": e})
    assert traffic is None and "prefill_tc.cu" in why
    assert bench.profiled_traffic("no_such_kernel") == (None, "no capture")


def test_bench_line_assembly_without_a_gpu(monkeypatch, capsys):
    """bench.run_gpu with every device call faked: the JSON line carries the
    contract's keys and derives its figures from the timings it was given."""
    sys.path.insert(0, ROOT)
    import types
    import bench
    from kimi_delta_attention_chunked_gb300 import build, inputs
    import kimi_delta_attention_chunked_gb300 as kda

    class Clocks:
        def __init__(self, gpu):
            pass

        def __enter__(self):
            return self

        def __exit__(self, *exc):
            return False

        def summary(self):
            return {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5}

    T, H = 8192, 32

    def fake_prefill(w, device=None, seed=0, lengths=None):
        small = lambda *s: torch.zeros(*s)
        return {"T": T, "q": small(4, 2), "k": small(4, 2), "v": small(4, 2), "log_alpha": small(4, 2),
                "beta": small(4), "S0": None}

    monkeypatch.setattr(bench, "ClockSampler", Clocks)
    monkeypatch.setattr(bench, "time_prefill", lambda *a, **k: (9.0, 0.25, 0.2, 40))
    monkeypatch.setattr(bench, "time_decode", lambda *a, **k: (168.0, 1000))
    monkeypatch.setattr(bench, "time_verify", lambda *a, **k: (0.368, 1_100_000_000))
    monkeypatch.setattr(bench, "time_few_heads", lambda *a, **k: {"value": 1.0})
    monkeypatch.setattr(bench, "time_e2e", lambda *a, **k: (20.0, 336_592_896, 69_206_016))
    monkeypatch.setattr(bench, "link_bandwidth", lambda *a, **k: {"h2d_gbs": 400.0, "d2h_gbs": 400.0})
    big = {}

    def fake_workload(kda_, inputs_, name, steps, warmup, stream, dev, seed=0):
        big[name] = steps
        return {"workload": name, "ms_per_step": 1.0, "roofline": bench.step_roofline(6.8e9 * 1e-3 / 2, 1.0)}
    monkeypatch.setattr(bench, "time_prefill_workload", fake_workload)
    monkeypatch.setattr(build, "build", lambda *a, **k: None)
    monkeypatch.setattr(kda, "load", lambda *a, **k: None)
    monkeypatch.setattr(inputs, "make_prefill", fake_prefill)
    monkeypatch.setattr(torch.cuda, "set_device", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a: None)
    monkeypatch.setattr(torch.cuda, "Stream", lambda *a, **k: None)
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    args = types.SimpleNamespace(steps=20, warmup=3, decode_steps=1000, no_cpu_baseline=True, oracle_tokens=8192,
                                 oracle_seconds=10.0, long_steps=3, parts=None)
    assert bench.run_gpu(args) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "clocks", "gpu_launches"):
        assert key in line, key
    assert line["value"] == pytest.approx(T * 20 / 9.0e-3)
    assert line["ms_per_step"] == pytest.approx(9.0 / 20)
    r = line["roofline"]
    assert r["achieved"] == pytest.approx(r["bytes_per_launch"] / 0.25e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert set(r) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert line["step_roofline"]["tflops_with_inverse"] > line["step_roofline"]["tflops"]
    dec = line["decode"]
    assert dec["value"] == pytest.approx(1000 / 0.168)
    assert dec["roofline"]["frac_of_nominal_8tbs"] < dec["roofline"]["frac"]
    assert line["e2e"]["h2d_bytes_per_step"] == 336_592_896
    assert line["gpu_launches"] == 40 and line["config"]["workload"] == bench.PREFILL
    # the two larger prefill workloads carry their own rooflines
    assert set(big) == {"varlen_bf16_8seq_1K_32K_H32_D128", "long_bf16_T1M_H32_D128"}
    assert line["varlen"]["roofline"]["frac"] == pytest.approx(0.5 * 6.8e9 / 1e9 / bench.peaks()[0])
    assert line["long_1M"]["workload"] == "long_bf16_T1M_H32_D128"
    e = line["e2e"]
    assert e["roofline"]["copy_floor_ms"] == pytest.approx(336_592_896 / 400e9 * 1e3)
    assert e["roofline"]["frac"] == pytest.approx(e["roofline"]["copy_floor_ms"] / e["ms_per_step"])
