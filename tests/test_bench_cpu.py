"""bench.py pieces that need no GPU: the algorithmic byte accounting against
the per-step definition (index row, C row, one weight row per (beam, legal
slot), survivor pairs, outputs), and the reference arm's JSON line."""
import importlib.util
import json
import os
import subprocess
import sys

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_step_bytes_definition():
    b = _bench()
    cfg = synth.CONFIGS["mid_sparse"]
    # step 2 of a batch: 1,024 live beams, sparse rows with 52,525 legal slots in all
    st = {"live_beams": 1024, "legal_slots": 52525, "index_bytes": 8 * 1024 + 2 * 52525, "unique_tokens": 2048}
    want = (8 * 1024 + 2 * 52525) + 1024 * cfg.d * 4 + 52525 * cfg.d * 4 + 1024 * cfg.beam * 8
    assert b.step_bytes(st, cfg, 2) == want
    # the last step adds the outputs: B * K * (4L + 4)
    last = b.step_bytes(st, cfg, cfg.L)
    assert last == want + cfg.batch * cfg.topk * (4 * cfg.L + 4)
    # step 1 has no gather-add row; half weights count 2 bytes an element
    half = synth.CONFIGS["large"]
    st1 = {"live_beams": 64, "legal_slots": 64 * 8192, "index_bytes": 64 * (8 + 4 * 256), "unique_tokens": 8192}
    assert b.step_bytes(st1, half, 1) == 64 * (8 + 4 * 256) + 64 * 8192 * half.d * 2 + 64 * half.beam * 8
    # the distinct-row bound reads each touched weight row once
    assert b.step_unique_bytes(st, cfg, 2) == (8 * 1024 + 2 * 52525) + 2048 * cfg.d * 4 + 1024 * cfg.d * 4 + 1024 * cfg.beam * 8


def test_full_flops():
    b = _bench()
    cfg = synth.CONFIGS["dense_early"]
    assert b.full_flops({}, cfg, 2) == 2 * cfg.batch * cfg.beam * cfg.V * cfg.d
    assert b.full_flops({}, cfg, 1) == 2 * cfg.batch * cfg.V * cfg.d


def test_launches_per_decode():
    """Kernel launches of one decode, counted from the plan as the engine issues them."""
    b = _bench()
    # large catalogue plan: step 1 full (hidden split, tensor cores, select), steps 2-4 stand-alone selective
    assert b.launches_per_decode([1, 0, 0, 0], 5, 4, "bf16") == 3 + 3 * 3
    # every step in the fused cluster kernel: one launch
    assert b.launches_per_decode([0, 0, 0], 1, 3, "f32") == 1
    # two full steps (the second with its gather-add), then the fused rest
    assert b.launches_per_decode([1, 1, 0, 0], 3, 4, "f16") == 3 + 4 + 1
    # fp32 weights: no hidden split
    assert b.launches_per_decode([1, 0], 3, 2, "f32") == 2 + 3


def test_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "requests/s" and line["value"] > 0
    for key in ("metric", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line
    assert line["config"]["global_batch"] == synth.CONFIGS["tiny"].batch
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
