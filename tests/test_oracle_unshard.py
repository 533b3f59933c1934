"""Pins of the oracle's FSDP2 unshard."""
import numpy as np
import pytest
import torch

from oracle import plan as P
from oracle import step as O

from test_oracle_step import HP, _inputs


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 4, 1), ("distopt", 4, 1), ("hsdp", 6, 2), ("fsdp2", 1, 1)])
def test_unshard_after_step_reproduces_the_steps_params(mode, n_d, n_rep):
    shapes = [(13, 5), (7,), (40, 3), (1,)]
    plan = P.plan_layout(shapes, n_d, mode, n_rep=n_rep)
    grads, (master, m, v), params = _inputs(plan, "f32", 2)
    O.sharded_step(plan, grads, "f32", master, m, v, params, HP, 10)
    fresh = [np.full_like(p, 0xFFFF) for p in params]
    O.unshard(plan, master, fresh)
    for a, b in zip(params, fresh):
        assert np.array_equal(a, b)


def test_unshard_equals_torch_cat_of_chunks():
    """Unsharding = torch.chunk's pieces, cast to bf16, concatenated back in rank order."""
    shapes = [(10, 3), (5,)]
    plan = P.plan_fsdp2(shapes, 3)
    rng = np.random.default_rng(0)
    master = np.full(plan.state_len_total, np.nan, np.float32)
    fi, si = P.owned_indices(plan)
    full = rng.standard_normal(plan.valid_elems).astype(np.float32)
    master[si] = full[fi]
    params = [np.zeros(plan.full_len_padded, np.uint16) for _ in range(3)]
    O.unshard(plan, master, params)
    want = torch.from_numpy(full).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for p in params:
        assert np.array_equal(p, want)


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 4, 1), ("fsdp2", 6, 1), ("distopt", 3, 1), ("hsdp", 8, 2)])
def test_shard_then_unshard_gives_the_cast_of_every_element(mode, n_d, n_rep):
    """shard is the inverse of the unshard's gather: going full -> shards ->
    every rank's full buffer gives back each element (cast to bf16) on every
    rank, and leaves shard padding alone."""
    shapes = [(7, 3), (1,), (13,), (5, 4, 2)]
    plan = P.plan_layout(shapes, n_d, mode, n_rep=n_rep)
    rng = np.random.default_rng(3)
    full = rng.standard_normal(plan.full_len_padded).astype(np.float32)
    master = np.full(plan.state_len_total, np.nan, np.float32)
    O.shard(plan, full, master)
    params = [np.zeros(plan.full_len_padded, np.uint16) for _ in range(n_d)]
    O.unshard(plan, master, params)
    want = O.bf16_rne(full[:plan.valid_elems])
    for q in range(n_d):
        assert np.array_equal(params[q][:plan.valid_elems], want)
    fi, si = P.owned_indices(plan)
    owned = np.zeros(plan.state_len_total, bool)
    owned[si] = True
    assert np.isnan(master[~owned]).all() and not np.isnan(master[owned]).any()
