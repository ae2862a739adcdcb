"""The multi-process path of bench.py (replicas only: no collective in the data
path), on CPU with gloo: the timing reduction over ranks and the reference arm's
rank filter."""
import os
import pathlib
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = pathlib.Path(__file__).resolve().parents[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, str(ROOT))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r timed 10 (r + 1) ms for 100 steps: the job's time is the slowest rank's
        ms, value = bench.replica_timing(10.0 * (rank + 1), 100, world, "cpu")
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_replica_timing_takes_the_slowest_rank(world):
    port = 29500 + 17 * world + os.getpid() % 1000
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn")
        res = dict(out)
    assert sorted(res) == list(range(world))
    for ms, value in res.values():
        assert ms == 10.0 * world
        assert abs(value - world * 100 / (10.0 * world / 1e3)) < 1e-9


def test_single_replica_needs_no_process_group():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.replica_timing(5.0, 50, 1) == (5.0, 50 / 0.005)


def test_reference_arm_other_ranks_exit_silently():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--gpus", "2"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_both_arms_share_the_config_object():
    sys.path.insert(0, str(ROOT))
    import bench
    from block_diffusion_drafter_fc_gb300.synth import get_config, make_workload
    cfg = get_config("tiny_f32")
    c = bench.workload_config(cfg, make_workload(cfg), 1)
    assert c["workload"].startswith("tiny_f32: 1 layers") and c["parallelism"] == "replicas x1"
    assert set(c) == {"workload", "sequences", "rows_per_step", "l2", "timing", "parallelism"}


@pytest.mark.parametrize("config", ["tiny_f32", "small_fp4"])
def test_reference_arm_prints_the_contract_line(config):
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--config", config,
                        "--steps", "2", "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    out = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in out, key
    assert out["impl"] == "reference" and out["steps"] == 2 and out["warmup"] == 1
    assert out["value"] > 0 and abs(out["ms_per_step"] - 1e3 / out["value"]) < 1e-3 * out["ms_per_step"] + 1e-3
    assert out["config"]["workload"].startswith(config + ":")
    cb = out["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == out["value"] and cb["cores"] >= 1
    assert out["e2e"] == {"value": out["value"], "unit": out["unit"], "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("config", ["tiny_f32", "small_fp8"])
def test_class_rates_cover_every_class(config):
    sys.path.insert(0, str(ROOT))
    import bench
    from block_diffusion_drafter_fc_gb300.synth import get_config, make_workload
    cfg = get_config(config)
    wl = make_workload(cfg)
    cb = bench.class_bytes(cfg, wl)
    # every class took 10 us per launch over 3 launches; the embedding is not rated
    prof = {k: (0.03, 3) for k in list(cb) + ["attention", "embed"]}
    r = bench.class_rates(cfg, wl, prof)
    assert set(r) == set(cb) | {"attention"}
    for k, nbytes in cb.items():
        assert abs(r[k] - round(nbytes / 1e-5 / 1e9, 1)) < 0.051
    ring = bench.step_bytes(cfg, wl) - wl.weight_bytes() - cfg.n_seq * 16 * cfg.n_vocab * 4
    assert ring > 0 and abs(r["attention"] - round(ring / cfg.n_layer / 1e-5 / 1e9, 1)) < 0.051
    # classes that did not run are left out
    assert bench.class_rates(cfg, wl, {k: (0.0, 0) for k in prof}) == {}


def test_reference_arm_times_whole_steps_when_they_fit():
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--config",
                        "tiny_f32", "--steps", "3", "--warmup", "2"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["cpu_baseline"]["sample"].startswith("3 whole fp64 oracle block steps of tiny_f32")


def test_graph_breakdown_charges_the_critical_path():
    """Each launch is charged from the previous launch's end to its own end
    (launches overlap under programmatic dependent launch), so the classes sum
    to the last end; spans are each launch's own start-to-end."""
    sys.path.insert(0, str(ROOT))
    import bench

    class FakeDrafter:
        def dflash_replay(self, stream):
            pass

        def dflash_profile_stamps(self, stream):
            return [("embed", 0.0, 5.0), ("qkv", 3.0, 30.0), ("attention", 25.0, 40.0),
                    ("qkv", 38.0, 61.0), ("accept", 60.0, 62.0)]

    class FakeTraffic:
        def run(self):
            pass

    crit, span, launches, total = bench.graph_breakdown(FakeDrafter(), None, FakeTraffic(), 3)
    assert crit == {"embed": 5.0, "qkv": 25.0 + 21.0, "attention": 10.0, "accept": 1.0}
    assert abs(sum(crit.values()) - 62.0) < 1e-9 and total == 62.0
    assert span == {"embed": 5.0, "qkv": 25.0, "attention": 15.0, "accept": 2.0}
    assert launches == {"embed": 1, "qkv": 2, "attention": 1, "accept": 1}
