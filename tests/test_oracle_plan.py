"""Pins of the oracle's layout planner (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import plan as P
from synth_inputs import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_qwen3_layer_shard_table_matches_walkthrough():
    """The per-rank shard shapes of the walkthrough's N=4 table."""
    g = _golden("qwen3_layer_shard_table.json")
    shapes = [tuple(p["shape"]) for p in g["params"]]
    assert tuple(shapes) == workload(0).shapes
    plan = P.plan_fsdp2(shapes, g["n_d"])
    for i, p in enumerate(g["params"]):
        assert P.numel(p["shape"]) == p["numel"]
        assert list(P.shard_shape(p["shape"], g["n_d"])) == p["shard"]
        segs = [s for s in plan.segments if s.param == i]
        assert len(segs) == g["n_d"]
        for s in segs:  # every rank owns a full, unpadded shard here
            assert s.length == p["shard_numel"] == s.padded_len
    per_rank = [sum(s.length for s in plan.segments if s.rank == r) for r in range(4)]
    assert per_rank == [590112] * 4
    assert round(per_rank[0] / 1000) == g["per_rank_total_approx_K"]
    assert round(per_rank[0] * 2 / 1e6, 2) == g["per_rank_MB_2byte"]
    assert round(plan.valid_elems / 1e6, 2) == g["layer_total_approx_M"]
    assert round(plan.valid_elems * 2 / 1e6, 2) == g["layer_MB_2byte"]


def _random_shapes(rng, n, n_d):
    shapes = []
    for _ in range(n):
        rows = int(rng.integers(0, 2 * n_d + 4))
        cols = int(rng.choice([1, 3, 5, 64]))
        if cols == 1 and rng.random() < 0.5:
            shapes.append((rows,))
        elif rng.random() < 0.3:
            shapes.append((rows, cols, 2))
        else:
            shapes.append((rows, cols))
    return shapes


@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 5, 6, 7, 8, 16])
def test_fsdp2_shards_equal_torch_chunk(n_d):
    """Rank r's rows are torch.chunk(param, N_d, dim=0)[r] (empty when chunk runs out)."""
    rng = np.random.default_rng(100 + n_d)
    shapes = _random_shapes(rng, 40, n_d)
    plan = P.plan_fsdp2(shapes, n_d)
    total = plan.valid_elems
    flat = torch.arange(total, dtype=torch.int64)
    for i, shape in enumerate(shapes):
        n = P.numel(shape)
        t = flat[plan.param_offsets[i]:plan.param_offsets[i] + n].reshape(shape)
        chunks = torch.chunk(t, n_d, dim=0) if shape[0] > 0 else ()
        for r in range(n_d):
            seg = [s for s in plan.segments if s.param == i and s.rank == r]
            assert len(seg) == 1
            seg = seg[0]
            want = chunks[r].reshape(-1) if r < len(chunks) else torch.zeros(0, dtype=torch.int64)
            got = torch.arange(seg.full_off, seg.full_off + seg.length)
            assert torch.equal(got, want)
            c = math.ceil(shape[0] / n_d)
            assert seg.padded_len == c * (n // shape[0] if shape[0] else 0)


@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
@pytest.mark.parametrize("n_d", [1, 2, 3, 5, 6, 8, 16])
def test_every_element_owned_once_and_state_disjoint(mode, n_d):
    rng = np.random.default_rng(7 * n_d)
    shapes = _random_shapes(rng, 30, n_d)
    plan = P.plan_layout(shapes, n_d, mode)
    owner = np.zeros(plan.full_len_padded, dtype=np.int64)
    slot = np.zeros(plan.state_len_total, dtype=np.int64)
    for s in plan.segments:
        owner[s.full_off:s.full_off + s.length] += 1
        slot[s.state_off:s.state_off + s.padded_len] += 1
        assert s.length <= s.padded_len
        # a rank's segments stay inside its own shard of the state buffers
        base = s.rank * plan.state_len_per_rank
        assert base <= s.state_off and s.state_off + s.padded_len <= base + plan.state_len_per_rank
    assert np.all(owner[:plan.valid_elems] == 1)
    assert np.all(owner[plan.valid_elems:] == 0)
    assert np.all(slot <= 1)


def test_fsdp2_state_alignment_and_rank_major_order():
    shapes = [(7,), (5, 3), (1,), (13, 64), (2, 5)]
    n_d = 3
    plan = P.plan_fsdp2(shapes, n_d)
    assert plan.state_len_per_rank % 16 == 0
    for r in range(n_d):
        segs = [s for s in plan.segments if s.rank == r]
        assert [s.param for s in segs] == list(range(len(shapes)))
        prev_end = r * plan.state_len_per_rank
        for s in segs:
            assert (s.state_off - s.full_off) % 16 == 0
            assert prev_end <= s.state_off < prev_end + 16   # the first congruent slot
            prev_end = s.state_off + s.padded_len


def test_rows_fewer_than_ranks():
    """rows=1 on 6 ranks: rank 0 owns the row, the others own padding only."""
    plan = P.plan_fsdp2([(1,)], 6)
    assert [s.length for s in plan.segments] == [1, 0, 0, 0, 0, 0]
    assert [s.padded_len for s in plan.segments] == [1] * 6
    plan = P.plan_fsdp2([(4, 3)], 6)
    assert [s.length for s in plan.segments] == [3, 3, 3, 3, 0, 0]


@pytest.mark.parametrize("total,n_d,padded", [
    (1000, 8, 1024), (1000, 6, 1152), (1000, 1, 1024), (128, 4, 128), (129, 4, 256),
    (1, 16, 128), (0, 8, 0), (384, 6, 384), (385, 6, 768), (1000, 3, 1152), (1000, 256, 1024),
])
def test_distopt_lcm_padding(total, n_d, padded):
    plan = P.plan_distopt([(total,)] if total else [], n_d)
    lcm = n_d * 128 // math.gcd(n_d, 128)
    assert plan.full_len_padded == padded and padded % lcm == 0 and padded - total < lcm
    shard = padded // n_d
    assert [s.full_off for s in plan.segments] == [r * shard for r in range(n_d)]
    assert all(s.padded_len == shard and s.state_off == s.full_off for s in plan.segments)
    assert sum(s.length for s in plan.segments) == total


def test_distopt_shards_ignore_param_boundaries():
    w = workload(2)
    plan = P.plan_distopt(w.shapes, w.n_d)
    assert plan.valid_elems == 596_049_920 == plan.full_len_padded
    assert plan.state_len_per_rank == 74_506_240
    # at least one shard boundary falls strictly inside a parameter
    starts = set(plan.param_offsets)
    assert any(s.full_off not in starts for s in plan.segments[1:])


def test_fsdp2_and_distopt_cover_same_elements():
    shapes = [(9, 4), (3,), (17,), (2, 2, 2)]
    a = P.plan_fsdp2(shapes, 4)
    b = P.plan_distopt(shapes, 4)
    fa, _ = P.owned_indices(a)
    fb, _ = P.owned_indices(b)
    assert np.array_equal(np.sort(fa), np.arange(a.valid_elems))
    assert np.array_equal(np.sort(fb), np.arange(b.valid_elems))


def test_workload_layouts():
    w1 = workload(1)
    p1 = P.plan_fsdp2(w1.shapes, w1.n_d)
    assert len(w1.shapes) == 310 and p1.valid_elems == 596_049_920
    # every row count of the 0.6B stack divides by 8: no FSDP2 padding
    assert all(s.length == s.padded_len for s in p1.segments)
    w3 = workload(3)
    assert len(w3.shapes) == 500
    assert all(s[0] % 6 != 0 and 1 <= s[0] <= 4099 for s in w3.shapes)
    assert {1 if len(s) == 1 else s[1] for s in w3.shapes} <= {1, 64, 1024, 4096}
    w4 = workload(4)
    assert len(w4.shapes) == 216 and w4.numel == 1_082_228_736


# --- per-parameter buffers: parameters at 16-element-aligned virtual offsets ---

def test_per_param_layout_worked_by_hand():
    """shapes (3,), (5, 2), (17,) on 2 ranks: offsets 0, 16, 32 (extent 49);
    dim-0 shards of 2, 3 and 9 rows; state slots by the residue rule."""
    p = P.plan_layout([(3,), (5, 2), (17,)], 2, "fsdp2", param_align=16)
    assert p.param_offsets == (0, 16, 32)
    assert (p.valid_elems, p.full_len_padded) == (3 + 10 + 17, 49)
    got = [(s.param, s.rank, s.full_off, s.state_off, s.length, s.padded_len) for s in p.segments]
    assert got == [
        (0, 0, 0, 0, 2, 2), (0, 1, 2, 48 + 2, 1, 2),
        (1, 0, 16, 16, 6, 6), (1, 1, 22, 48 + 6, 4, 6),
        (2, 0, 32, 32, 9, 9), (2, 1, 41, 48 + 25, 8, 9),
    ]
    assert p.state_len_per_rank == 48


@pytest.mark.parametrize("n_d", [1, 3, 4, 8])
def test_per_param_layout_properties(n_d):
    shapes = [(7, 3), (1,), (33,), (16, 2), (5,), (129, 7)]
    p = P.plan_layout(shapes, n_d, "fsdp2", param_align=16)
    flat = P.plan_layout(shapes, n_d, "fsdp2")
    at = 0
    for off, s in zip(p.param_offsets, shapes):
        assert off % 16 == 0 and at <= off < at + 16
        at = off + P.numel(s)
    assert p.full_len_padded == at and p.valid_elems == flat.valid_elems
    fi, si = P.owned_indices(p)
    want = np.concatenate([np.arange(o, o + P.numel(s)) for o, s in zip(p.param_offsets, shapes)])
    assert np.array_equal(np.sort(fi), want)                     # every element once, gaps nobody's
    assert len(set(si.tolist())) == si.size
    for s in p.segments:
        assert (s.state_off - s.full_off) % 16 == 0
    # shard heights and lengths are the flat plan's, element for element
    assert [(s.param, s.rank, s.length, s.padded_len) for s in p.segments] == \
        [(s.param, s.rank, s.length, s.padded_len) for s in flat.segments]


def test_per_param_layout_equals_flat_when_sizes_are_multiples_of_16():
    shapes = [(16, 3), (32,), (4, 4)]
    assert P.plan_layout(shapes, 4, "fsdp2", param_align=16) == P.plan_layout(shapes, 4, "fsdp2")


def test_per_param_layout_hsdp_and_rejections():
    p = P.plan_layout([(3,), (5, 2)], 4, "hsdp", n_rep=2, param_align=16)
    assert p.param_offsets == (0, 16) and p.n_rep == 2
    with pytest.raises(ValueError):
        P.plan_layout([(3,)], 2, "distopt", param_align=16)
    with pytest.raises(ValueError):
        P.plan_layout([(3,)], 2, "fsdp2", param_align=8)
