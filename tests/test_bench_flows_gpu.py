"""Every flow bench.py times runs and prints one well-formed JSON line (small
param slices, a few steps)."""
import json
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

from gpu_cases import ensure_built  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


FLOWS = [
    [], ["--clip", "1.0"], ["--writeback"], ["--no-gather"], ["--unshard"], ["--fp32-gather"],
    ["--fp32-gather", "--unshard"], ["--per-param"], ["--per-param", "--unshard"], ["--graph"],
    ["--workload", "5"], ["--workload", "4"], ["--n-d", "9"], ["--workload", "0", "--layers", "3"],
    ["--workload", "0", "--layers", "3", "--unshard"], ["--workload", "0", "--layers", "3", "--no-gather"],
]


@pytest.mark.parametrize("flow", FLOWS, ids=[" ".join(f) or "step" for f in FLOWS])
def test_bench_flow_prints_one_line(flow, capsys):
    args = ["--param-slice", "1:6", "--steps", "3", "--warmup", "3", "--no-e2e", "--no-cpu-baseline"] + flow
    bench.main(args)
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "roofline", "clocks",
              "gpu_launches", "config"):
        assert k in d, k
    assert d["value"] > 0 and d["roofline"]["achieved"] > 0
    assert "l2" in d["config"]
    layers = int(flow[flow.index("--layers") + 1]) if "--layers" in flow else 1
    assert d["gpu_launches"] == 3 * layers * (4 if "--clip" in flow else 1)
    import fsdp_sharded_mixed_pass_gb300 as fsp
    assert fsp.device_error() == 0


def test_workloads_block_times_each_workload():
    """The default run's block of the other workloads: one entry each, with
    its own time, bandwidth and roofline fraction (small slices here)."""
    dev = torch.device("cuda", 0)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    dist = bench.Dist(1)
    try:
        out = bench.time_workloads(["qwen3_layer", "ragged_500", "dense_1p5b_bf16grad", ("qwen3_layer", 3),
                                    ("qwen3_0p6b_fsdp2", 2, "1:3")], 3, 3,
                                   dist, None, dev, l2, 6698.2, param_slice="1:6")
    finally:
        dist.close()
    assert [e["workload"] for e in out] == ["qwen3_layer[1:6]", "ragged_500[1:6]", "dense_1p5b_bf16grad[1:6]",
                                            "qwen3_layer[1:6] x3 (one plan per layer, stepped back to back)",
                                            "qwen3_0p6b_fsdp2[1:3] x2 (one plan per layer, stepped back to back)"]
    assert out[3]["layers"] == 3 and out[3]["params"] == 3 * out[0]["params"]
    assert out[3]["ms_per_layer"] == out[3]["ms_per_step"] / 3
    for e in out:
        assert "error" not in e, e
        assert e["ms_per_step"] > 0 and e["params_per_s"] > 0
        assert abs(e["hbm_gbs"] - e["bytes_per_param"] * e["params"] / (e["ms_per_step"] / 1e3) / 1e9) < 1e-6 * e["hbm_gbs"]
        assert e["frac_of_measured"] == e["hbm_gbs"] / 6698.2
    assert out[0]["bytes_per_param"] == 48 and out[2]["bytes_per_param"] == 88
    assert "graph_ms_per_step" in out[0]          # small enough for an L2 flush: also a CUDA-graph time
