"""bench.py's reference arm runs the oracle on the host cores: on CPU it must print the contract's one
JSON line (the same keys as the GPU arm's line, plus impl, cpu_baseline and e2e describing this run),
and under a multi-rank launch only rank 0 does any work."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra, *args):
    env = dict(os.environ, OMP_NUM_THREADS="2", **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


@pytest.fixture(scope="module")
def oracle_built():
    import oracle
    oracle.build_lib()  # the plain C oracle (gcc), as the oracle pins build it


def test_reference_arm_prints_the_contract_line(oracle_built):
    r = _run({}, "--steps", "2", "--warmup", "1", "--workload", "tiny-moe-4e2r")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["unit"] == "tokens/s" and d["dtype"] == "f64" and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith("tiny-moe-4e2r")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # ms_per_step and value describe the same sampled tokens
    per_step = d["config"]["sample_tokens_per_step"]
    assert abs(per_step / (d["ms_per_step"] / 1e3) - d["value"]) <= 1e-6 * d["value"]


def test_reference_arm_other_ranks_exit_without_work(oracle_built):
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--steps", "2", "--warmup", "1",
             "--workload", "tiny-moe-4e2r", "--gpus", "2")
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_roofline_counts_follow_the_layer_shape():
    """The roofline's algorithmic FLOPs and bytes, written out by hand from the layer's shape: the up
    projection's two (SwiGLU) or one matrices over every routed row, the down projection's one, the
    router's logits; bytes = the active experts' three (or two) matrices + x in + fp32 out + W_r."""
    sys.path.insert(0, ROOT)
    import bench
    import testgen
    s = testgen.CONFIGS["mixtral-prefill"]          # T=8192, d=4096, f=14336, E=8, top-2, SwiGLU, bf16
    a = bench.algorithmic(s, s.T)
    rows = 2 * 8192
    assert a["flops_up"] == 2.0 * rows * 4096 * 14336 * 2 == 3848290697216.0
    assert a["flops_down"] == 2.0 * rows * 4096 * 14336
    assert a["flops"] == a["flops_up"] + a["flops_down"] + 2.0 * 8192 * 8 * 4096
    assert a["bytes"] == 8 * 3 * 4096 * 14336 * 2 + 8192 * 4096 * 2 + 8192 * 4096 * 4 + 8 * 4096 * 2
    # decode-sized: only the distinct active experts' weights are streamed
    d1 = bench.algorithmic(s, 1, active_experts=2)
    assert d1["w_bytes_up"] == 2 * 2 * 4096 * 14336 * 2 and d1["w_bytes_expert"] == 3 * 4096 * 14336 * 2
    r = testgen.CONFIGS["tiny-moe-4e2r"]            # ReLU+bias: one up matrix, fp32
    t = bench.algorithmic(r, r.T)
    assert t["flops_up"] == t["flops_down"] == 2.0 * 2 * r.T * r.d_model * r.d_ff
    assert t["w_bytes_expert"] == 2 * r.d_model * r.d_ff * 4
