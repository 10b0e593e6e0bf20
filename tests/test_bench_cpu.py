"""CPU check of the benchmark's output contract on its reference arm (the fp64 oracle on
the host cores): one JSON line with the fields the driver reads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "1", "--ref-seconds", "1", "--workload", "tiny_fp32"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 1
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"]
    assert line["config"]["workload"] == "tiny_fp32"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert "single-request copies" in cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_multi_rank_sets_are_shards_of_one_global_batch():
    """Under torchrun each rank's input set is its longest-prompt-first shard of one global
    batch of world x batch requests: together the shards hold every request's prompt length
    and step labels once, and each set's workload has the shard's batch size."""
    import argparse
    import sys as _sys
    _sys.path.insert(0, ROOT)
    import bench
    import workloads
    w = workloads.WORKLOADS["ragged_bf16"].with_(batch=6, Hq=4, Hkv=1, V=64)
    args = argparse.Namespace(cache_layout="NHD")
    world = 2
    glay = workloads.make_layout_inputs(w.with_(batch=w.batch * world), seed=w.seed)
    plens, taus = [], []
    for rank in range(world):
        (s,) = bench._make_sets(w, args, "cpu", 1, rank, world=world)
        assert s["_w"].batch == s["prompt_len"].numel() == s["q"].shape[0]
        assert int(s["k_cache"].shape[0]) == int(s["prompt_len"].sum())
        plens += s["prompt_len"].tolist()
        taus += [tuple(t) for t in s["tau"].tolist()]
    assert sorted(plens) == sorted(glay["prompt_len"].tolist())
    assert sorted(taus) == sorted(tuple(t) for t in glay["tau"].tolist())
