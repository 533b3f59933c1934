"""Pins of the oracle's HSDP extension (shard group x replicate group)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import synth_inputs as S
from oracle import ledger as L
from oracle import plan as P
from oracle import step as O

from test_oracle_step import HP, SENTINEL_PARAM, SENTINEL_STATE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_hybrid_sum_is_group_then_across_groups():
    # ranks (r, j) = (0,0) 1e8, (0,1) 1, (1,0) -1e8, (1,1) 1 in fp32:
    # inside group 0: 1e8 + 1 = 1e8; group 1: -1e8 + 1 = -1e8; across: 0.
    # The flat rank-ordered fold of the same four numbers gives 1.
    g = [np.array([v], np.float32) for v in (1e8, 1.0, -1e8, 1.0)]
    assert O.hybrid_sum(g, 2).tolist() == [0.0]
    assert O.hybrid_sum(g, 1).tolist() == [1.0] == O.rank_ordered_sum(g).tolist()
    assert O.hybrid_sum(g, 4).tolist() == [1.0]


def test_hsdp_plan_is_replicated_fsdp2():
    shapes = [(9, 4), (3,), (17,)]
    h = P.plan_hsdp(shapes, 3, 2)
    f = P.plan_fsdp2(shapes, 2)
    assert h.n_d == 6 and h.n_rep == 3 and h.n_shard == 2
    assert h.state_len_total == 3 * f.state_len_total
    for r in range(3):
        mine = [s for s in h.segments if s.rank // 2 == r]
        assert [(s.param, s.rank - 2 * r, s.full_off, s.state_off - r * f.state_len_total, s.length)
                for s in mine] == [(s.param, s.rank, s.full_off, s.state_off, s.length) for s in f.segments]


def _inputs(plan, grad_dtype, seed):
    idx = np.arange(plan.full_len_padded)
    if grad_dtype == "f32":
        grads = [S.grad_f32(seed, q, idx) for q in range(plan.n_d)]
    else:
        grads = [S.grad_bf16_bits(seed, q, idx) for q in range(plan.n_d)]
    fi, si = P.owned_indices(plan)
    states = []
    for fn in (S.master_f32, S.adam_m_f32, S.adam_v_f32):
        buf = np.full(plan.state_len_total, SENTINEL_STATE, np.uint32).view(np.float32)
        buf[si] = fn(seed, fi)
        states.append(buf)
    params = [np.full(plan.full_len_padded, SENTINEL_PARAM, np.uint16) for _ in range(plan.n_d)]
    return grads, states, params


@pytest.mark.parametrize("n_rep,n_shard", [(1, 4), (2, 1), (2, 2), (2, 3), (4, 2), (3, 5)])
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
def test_hsdp_sharded_equals_unsharded(n_rep, n_shard, grad_dtype):
    rng = np.random.default_rng(n_rep * 10 + n_shard)
    shapes = [(int(rng.integers(1, 2 * n_shard + 5)), int(rng.choice([1, 3, 64]))) for _ in range(5)]
    plan = P.plan_hsdp(shapes, n_rep, n_shard)
    grads, (master, m, v), params = _inputs(plan, grad_dtype, 3)
    fi, si = P.owned_indices(plan)
    n = plan.valid_elems
    th0 = np.empty(n, np.float32); m0 = np.empty(n, np.float32); v0 = np.empty(n, np.float32)
    th0[fi] = master[si]; m0[fi] = m[si]; v0[fi] = v[si]
    O.sharded_step(plan, grads, grad_dtype, master, m, v, params, HP, 10)
    th_u, m_u, v_u, b_u = O.unsharded_step(grads, grad_dtype, th0, m0, v0, n, HP, 10, n_rep=n_rep)
    per = n  # every replica's copy of every element
    for r in range(n_rep):
        sl = slice(r * per, (r + 1) * per)
        order = np.argsort(fi[sl])
        assert np.array_equal(master[si[sl]][order].view(np.uint32), th_u.view(np.uint32))
        assert np.array_equal(m[si[sl]][order].view(np.uint32), m_u.view(np.uint32))
        assert np.array_equal(v[si[sl]][order].view(np.uint32), v_u.view(np.uint32))
    for q in range(plan.n_d):
        assert np.array_equal(params[q][:n], b_u)


def test_hsdp_with_one_replica_is_fsdp2_bit_for_bit():
    shapes = [(13, 5), (7,), (40, 3)]
    a = P.plan_hsdp(shapes, 1, 4)
    b = P.plan_fsdp2(shapes, 4)
    ga, sa, pa = _inputs(a, "f32", 8)
    gb, sb, pb = _inputs(b, "f32", 8)
    O.sharded_step(a, ga, "f32", *sa, pa, HP, 10)
    O.sharded_step(b, gb, "f32", *sb, pb, HP, 10)
    for x, y in zip(sa + pa, sb + pb):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_hsdp_with_unit_shard_groups_is_flat_data_parallel():
    # N_s = 1: no sharding inside a group, N_r replicas: the flat rank-ordered
    # all-reduce of plain data parallelism, element for element
    shapes = [(13, 5), (7,)]
    a = P.plan_hsdp(shapes, 4, 1)
    ga, (ma, m_a, va), pa = _inputs(a, "f32", 9)
    b = P.plan_fsdp2(shapes, 4)
    gb, (mb, m_b, vb), pb = _inputs(b, "f32", 9)
    O.sharded_step(a, ga, "f32", ma, m_a, va, pa, HP, 10)
    O.sharded_step(b, gb, "f32", mb, m_b, vb, pb, HP, 10)
    fa, sa = P.owned_indices(a)
    fb, sb = P.owned_indices(b)
    n = a.valid_elems
    oa = np.argsort(fa[:n]); ob = np.argsort(fb)
    assert np.array_equal(ma[sa[:n]][oa], mb[sb][ob])
    for q in range(4):
        assert np.array_equal(pa[q], pb[q])


def test_hsdp_memory_and_traffic_pins():
    g = json.load(open(os.path.join(GOLDEN, "hsdp_70b.json")))
    for ns, want in g["per_card_GB"].items():
        per = L.hsdp_bytes_per_param(int(ns), grad_bytes=2)
        assert per == Fraction(g["bytes_per_param_unsharded"], int(ns))
        assert round(float(per) * g["params"] / 1e9, g["per_card_GB_decimals"][ns]) == want
    # cross-group traffic 2(N_r-1)/N_r * S/N_s -> 2S/N_s as N_r grows
    S_ = 1_000_000
    for n_rep, n_shard in ((2, 8), (16, 8), (1024, 64)):
        sent = L.hsdp_step_sent(n_rep, n_shard, S_, S_)
        assert sent["cross_group_all_reduce"] == Fraction(2 * (n_rep - 1), n_rep) * Fraction(S_, n_shard)
        assert sent["cross_group_all_reduce"] < Fraction(2 * S_, n_shard)
        assert sent["reduce_scatter"] == Fraction(n_shard - 1, n_shard) * S_
    # one replica: no cross-group traffic; HSDP memory = FSDP memory over N_s
    assert L.hsdp_step_sent(1, 8, S_, S_)["cross_group_all_reduce"] == 0
    assert L.hsdp_bytes_per_param(8) == L.bytes_per_param("fsdp", 8)
    assert L.sharded_step_bytes(8, 4, n_rep=2) == 8 * 4 + 48 + 16
