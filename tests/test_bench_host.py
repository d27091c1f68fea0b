"""The benchmark's CPU restatement of the pages' method (gather + einsum
attention in fp32) computes the same attention as the oracle."""
import numpy as np
import pytest

import bench
import oracle
from gpu_step import raw
from workloads import draw_plan, make_layer


@pytest.mark.parametrize("name", ["toy", "smollm2-135m"])
def test_pages_method_matches_oracle(name):
    plan = draw_plan(name)
    layer = make_layer(plan, 0)
    nd = plan.n_decode
    outs = []
    bench.pages_method_sample(plan, layer, range(nd), outputs=outs)
    r = {n: raw(layer[n]) for n in ("q", "k_pool", "v_pool")}
    ref = oracle.paged_attention_decode(r["q"][:nd], r["k_pool"], r["v_pool"], plan.block_tables[:nd],
                                        plan.seq_lens[:nd], plan.shape.scale, plan.shape.dtype)
    got = np.stack([o.double().numpy() for o in outs])
    assert np.max(np.abs(got - ref)) < 1e-5


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the float64 oracle on the host cores)
    prints one JSON line with the contract's keys, its own e2e with no
    copies, and a cpu_baseline describing the sample it timed."""
    import json
    import subprocess
    import sys
    root = __import__("os").path.dirname(__import__("os").path.dirname(__file__))
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "smollm2-135m", "--steps", "2", "--warmup", "1"], cwd=root,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert "smollm2-135m" in cb["sample"] and "0 prefill queries" in cb["sample"]
    assert d["config"]["workload"] == "smollm2-135m" and "launch" not in d["config"]
    assert cb["host_cores"] >= 1


def test_decode_traffic_ratios_match_current_kernel_sources():
    """Every DRAM-traffic ratio the benchmark reports was captured on the
    decode kernel sources as they are now: a ratio recorded with another
    source hash is stale (recapture it, or drop the entry)."""
    h = bench.decode_source_hash()
    for key, rec in bench.DECODE_TRAFFIC.items():
        assert rec["source_sha256"] == h, (
            f"traffic ratio for {key} was captured on decode sources {rec['source_sha256']}, "
            f"now {h}")
        assert 0.9 < rec["ratio"] < 2.0 and rec["capture"]


def test_config_has_workload_keys_only():
    """Both arms describe the workload with the same keys; how the GPU arm
    launches its kernels is reported outside `config`."""
    from workloads import draw_plan
    cfg = bench.workload_config(draw_plan("llama2-70b-mixed"))
    assert "launch" not in cfg
    assert cfg["workload"] == bench.WORKLOAD_LABEL and cfg["layers_timed"] == 1
