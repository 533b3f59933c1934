"""Pins of the oracle's distributed-optimizer flow: reduce-scatter with
write-back into the owner's grad slice, global-norm clipping."""
import json
import os

import numpy as np
import pytest

import synth_inputs as S
from oracle import plan as P
from oracle import step as O

from test_oracle_step import HP, _inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_write_back_fills_only_the_owners_slice():
    g = json.load(open(os.path.join(GOLDEN, "zero1_toy.json")))
    n = g["n_ranks"]
    plan = P.plan_fsdp2([(8,)], n)
    grads = [np.float32(10 * r) + np.arange(8, dtype=np.float32) for r in range(n)]
    O.reduce_scatter_write_back(plan, grads)
    avg = [x / n for x in g["all_reduce"]]          # [15, 16, ..., 22]
    for r in range(n):
        own = slice(2 * r, 2 * r + 2)
        want = 10 * r + np.arange(8, dtype=np.float32)
        want[own] = avg[own]
        assert grads[r].tolist() == want.tolist()


def test_global_norm_and_coefficient_by_hand():
    assert O.global_grad_norm([np.array([3.0], np.float32), np.array([4.0], np.float32)]) == 5.0
    assert O.clip_coefficient(5.0, 1.0) == np.float32(1.0 / (5.0 + 1e-6))
    assert O.clip_coefficient(5.0, 10.0) == np.float32(1.0)
    assert O.clip_coefficient(0.0, 1.0) == np.float32(1.0)


def test_no_clipping_equals_the_plain_step():
    shapes = [(13, 5), (7,), (40, 3)]
    a = P.plan_fsdp2(shapes, 4)
    ga, sa, pa = _inputs(a, "f32", 4)
    gb, sb, pb = _inputs(a, "f32", 4)
    norm, coef = O.sharded_step_clipped(a, ga, *sa, pa, HP, 10, max_norm=1e30)
    O.sharded_step(a, gb, "f32", *sb, pb, HP, 10)
    assert coef == 1.0 and norm > 0
    for x, y in zip(sa + pa, sb + pb):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_clipping_scales_the_gradient_not_the_update():
    # t=1, m=v=0, wd=0, eps=0: Adam's first step is lr * sign(G), whatever the
    # scale of G, so a clipped step moves theta exactly as an unclipped one,
    # while m' = (1 - b1) * coef * G shows the scaled gradient.
    plan = P.plan_fsdp2([(64,)], 2)
    grads, (master, m, v), params = _inputs(plan, "f32", 6)
    m[:] = 0
    v[:] = 0
    hp = dict(HP, weight_decay=0.0, eps=0.0)
    th0 = master.copy()
    g_ref = [g.copy() for g in grads]
    norm, coef = O.sharded_step_clipped(plan, grads, master, m, v, params, hp, 1, max_norm=1e-4)
    assert coef < 0.5
    G = O.average(O.rank_ordered_sum(g_ref), 2)
    fi, si = P.owned_indices(plan)
    step = (th0[si] - master[si]).astype(np.float64)
    # exact up to the fp32 rounding of theta itself (|theta| < 0.13: ulp < 1.5e-8)
    assert np.allclose(step, np.float32(hp["lr"]) * np.sign(G[fi]), rtol=0, atol=2e-8)
    want_m = (1 - np.float64(np.float32(0.9))) * (G[fi] * coef).astype(np.float32)
    assert np.allclose(m[si], want_m, rtol=1e-6, atol=0)
    assert np.isclose(norm, np.sqrt(np.sum(G.astype(np.float64) ** 2)), rtol=1e-12)


def test_clipped_step_distopt_matches_fsdp2_per_element():
    shapes = [(9, 4), (3,), (17,), (40, 3)]
    out = {}
    for mode in ("fsdp2", "distopt"):
        plan = P.plan_layout(shapes, 4, mode)
        grads, (master, m, v), params = _inputs(plan, "f32", 5)
        norm, coef = O.sharded_step_clipped(plan, grads, master, m, v, params, HP, 10, max_norm=1e-3)
        fi, si = P.owned_indices(plan)
        o = np.argsort(fi)
        out[mode] = (norm, coef, master[si][o], params[0][:plan.valid_elems])
    assert out["fsdp2"][1] == out["distopt"][1] < 1
    assert np.isclose(out["fsdp2"][0], out["distopt"][0], rtol=1e-12)
    assert np.array_equal(out["fsdp2"][2], out["distopt"][2])
    assert np.array_equal(out["fsdp2"][3], out["distopt"][3])


def test_clipping_rejects_bf16():
    plan = P.plan_hsdp([(8,)], 2, 2)
    grads, _, _ = _inputs(plan, "f32", 1)
    with pytest.raises(ValueError):
        O.reduce_scatter_write_back(P.plan_fsdp2([(8,)], 2), grads[:2], "bf16")


@pytest.mark.parametrize("n_rep,n_shard", [(2, 2), (2, 3), (3, 2), (4, 1)])
@pytest.mark.parametrize("max_norm", [1e-4, 1e30])
def test_hsdp_clipped_step_equals_the_unsharded_definition(n_rep, n_shard, max_norm):
    """HSDP with clipping against the plain definition over the full buffer:
    the grouped all-reduce average, its fp64 norm over every element once, the
    clipped AdamW; every replica group's state copy and parameters, and every
    group's owner slices written back with the averaged gradient."""
    shapes = [(9, 5), (13,), (1,), (2 * n_shard + 1, 3)]
    plan = P.plan_hsdp(shapes, n_rep, n_shard)
    grads, (master, m, v), params = _inputs(plan, "f32", 21)
    n = plan.full_len_padded
    G = O.all_reduce(grads, "f32", n_rep=n_rep)
    want_norm = float(np.sqrt(np.sum(G[:plan.valid_elems].astype(np.float64) ** 2)))
    fi, si = P.owned_indices(plan)
    th0, m0, v0 = master[si].copy(), m[si].copy(), v[si].copy()
    norm, coef = O.sharded_step_clipped(plan, grads, master, m, v, params, HP, 7, max_norm)
    assert norm == pytest.approx(want_norm, rel=1e-12)
    assert abs(float(coef) - float(O.clip_coefficient(want_norm, max_norm))) <= 2.0 ** -23 * float(coef)
    assert (coef < 1) == (max_norm < 1)
    th, mm, vv = O.adamw(th0, m0, v0, (G[fi] * coef).astype(np.float32), HP, 7)
    assert np.array_equal(master[si], th) and np.array_equal(m[si], mm) and np.array_equal(v[si], vv)
    for s in plan.segments:   # every group's owner holds the averaged slice
        assert np.array_equal(grads[s.rank][s.full_off:s.full_off + s.length], G[s.full_off:s.full_off + s.length])
    cast = np.zeros(n, np.uint16)
    cast[fi] = O.bf16_rne(th)
    for q in range(plan.n_d):
        assert np.array_equal(params[q][:plan.valid_elems], cast[:plan.valid_elems])


def test_hsdp_clipped_with_one_group_is_the_fsdp2_flow():
    shapes = [(9, 5), (13,), (1,)]
    outs = []
    for plan in (P.plan_fsdp2(shapes, 3), P.plan_hsdp(shapes, 1, 3)):
        grads, (master, m, v), params = _inputs(plan, "f32", 22)
        norm, coef = O.sharded_step_clipped(plan, grads, master, m, v, params, HP, 4, 1e-3)
        outs.append((norm, coef, master, m, v, params, grads))
    a, b = outs
    assert a[0] == b[0] and a[1] == b[1]
    for x, y in zip(a[2:5], b[2:5]):       # (NaN sentinels in the padding: compare bits)
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    for x, y in zip(a[5] + a[6], b[5] + b[6]):
        assert np.array_equal(x.view(np.uint16 if x.dtype == np.uint16 else np.uint32),
                              y.view(np.uint16 if y.dtype == np.uint16 else np.uint32))
