"""Pins of the oracle's byte ledger, collective volumes and parameter count."""
import json
import os
from fractions import Fraction

import pytest

from oracle import ledger as L
from oracle import plan as P
from synth_inputs import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("n_d", [1, 2, 4, 6, 8, 16, 64])
def test_bytes_per_param_tables(n_d):
    g = _golden("bytes_per_param.json")
    for scheme, (a, b) in g["fp32_grad"].items():
        assert L.bytes_per_param(scheme, n_d, grad_bytes=4) == a + Fraction(b, n_d)
    for scheme, (a, b) in g["bf16_grad"].items():
        assert L.bytes_per_param(scheme, n_d, grad_bytes=2) == a + Fraction(b, n_d)


def test_7b_parameter_count_and_ledger():
    g = _golden("memory_ledger_7b.json")
    m = g["model"]
    total = L.dense_param_count(m["h"], m["L"], m["a"], m["g"], m["d"], m["ffn"], m["V"], final_norm=True)
    assert total == g["P_total"]
    # the pieces printed beside the total
    no_vocab = L.dense_param_count(m["h"], 1, m["a"], m["g"], m["d"], m["ffn"], 0, final_norm=False)
    assert no_vocab == g["per_layer_total"]
    assert L.dense_param_count(m["h"], m["L"], m["a"], m["g"], m["d"], m["ffn"], 0) == g["block_total_with_final_ln"]
    assert m["V"] * m["h"] == g["embedding"]
    # most loaded (first) stage: TP-split matrices / PP / TP, embedding / TP, replicated norms / PP
    tp, pp, dp = g["parallel"]["TP"], g["parallel"]["PP"], g["parallel"]["DP"]
    split = (g["per_layer_total"] - g["ln_per_layer"]) * m["L"]
    assert split // pp // tp == g["tp_split_first_stage"]
    assert g["embedding"] // tp == g["embedding_per_tp"]
    assert (g["ln_per_layer"] * m["L"] + m["h"]) // pp == g["replicated_per_pp"]
    p_shard = g["tp_split_first_stage"] + g["embedding_per_tp"] + g["replicated_per_pp"]
    assert float(f"{p_shard:.4g}") == g["P_shard_approx"]

    def gb(x):
        return round(float(x) / 1e9, g["GB_decimals"])

    assert L.bytes_per_param("distopt", dp) == Fraction(g["distopt_bytes_per_param"])
    parts = L.resident_breakdown_distopt(p_shard, dp)
    assert gb(parts["param"]) == g["distopt_param_GB"]
    assert gb(parts["grad"]) == g["distopt_grad_GB"]
    assert gb(parts["optimizer"]) == g["distopt_optimizer_GB"]
    assert gb(L.resident_bytes("distopt", p_shard, dp)) == g["distopt_resident_GB"]
    assert gb(L.resident_bytes("ddp", p_shard, dp)) == g["no_distopt_resident_GB"]
    assert gb(L.resident_bytes("fsdp", p_shard, dp)) == g["fsdp_resident_GB"]


def test_qwen3_layer_comm_volume():
    g = _golden("comm_volume_qwen3_layer.json")
    w = workload(0)
    payload = w.numel * 2
    assert round(payload / 1e6, 2) == g["layer_MB_2byte"]
    ag = L.coll_bytes("all_gather", g["n_d"], payload)
    rs = L.coll_bytes("reduce_scatter", g["n_d"], payload)
    assert round(float(ag) / 1e6, 2) == g["all_gather_MB_per_rank"]
    assert round(float(rs) / 1e6, 2) == g["reduce_scatter_MB_per_rank"]
    # forward all-gather + backward all-gather + backward reduce-scatter
    assert round(float(2 * ag + rs) / 1e6, 1) == g["per_layer_step_MB_per_rank"]


def test_all_reduce_is_reduce_scatter_plus_all_gather_in_volume():
    for n in (1, 2, 3, 4, 8, 64):
        s = 1000
        assert L.coll_bytes("all_reduce", n, s) == L.coll_bytes("reduce_scatter", n, s) + L.coll_bytes("all_gather", n, s)
    assert L.coll_bytes("send_recv", 1, 7) == 7
    with pytest.raises(ValueError):
        L.coll_bytes("broadcast", 2, 1)


def test_workload_param_counts_follow_the_formula():
    # one walkthrough layer: d=512, 8/4 heads of 64, ffn 1024, q/k-norm, no vocab
    assert L.dense_param_count(512, 1, 8, 4, 64, 1024, 0, final_norm=False, qk_norm=True) == workload(0).numel
    # Qwen3-0.6B shape: 28 layers, d=1024, 16/8 heads of 128, ffn 3072, tied vocab 151936
    assert L.dense_param_count(1024, 28, 16, 8, 128, 3072, 151936, final_norm=True, qk_norm=True) == workload(1).numel
    # 24 layers, d=2048, 16/4 heads of 128, ffn 5632
    assert L.dense_param_count(2048, 24, 16, 4, 128, 5632, 0, final_norm=False) == workload(4).numel


@pytest.mark.parametrize("idx,per_param", [(0, 48), (1, 72), (2, 72), (3, 60), (4, 88)])
def test_algorithmic_bytes_per_element(idx, per_param):
    w = workload(idx)
    assert L.sharded_step_bytes(w.n_d, w.grad_bytes) == per_param


def test_ledger_from_a_plan():
    """FSDP2 rank holds 18/N_d bytes per param of the model when nothing is padded."""
    w = workload(1)
    plan = P.plan_fsdp2(w.shapes, w.n_d)
    per_rank = sum(s.padded_len for s in plan.segments if s.rank == 0)
    assert per_rank * 8 == w.numel
    assert L.resident_bytes("fsdp", w.numel, w.n_d) == 18 * per_rank
