"""GPU parity of the fused step against the oracle, element by element, on
sizes the oracle finishes in seconds (several tiles, ragged tails, every
specialised and the generic N_d)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from synth_inputs import workload

from gpu_cases import HP, DeviceCase, Guarded, OracleCase, compare, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _tiny_shapes(rng, n_d):
    shapes = []
    for _ in range(int(rng.integers(2, 10))):
        rows = int(rng.integers(1, 2 * n_d + 6))
        cols = int(rng.choice([1, 3, 5, 64, 67]))
        shapes.append((rows,) if cols == 1 else (rows, cols))
    return shapes


def _run(shapes, n_d, mode, grad_dtype, seed, steps=(10, 11), n_rep=1):
    dev = DeviceCase(shapes, n_d, mode, grad_dtype, seed, n_rep)
    ora = OracleCase(shapes, n_d, mode, grad_dtype, seed, n_rep)
    stats = None
    for t in steps:
        dev.step(t)
        ora.step(t)
        torch.cuda.synchronize()
        stats = compare(dev, ora)
    return stats


@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 5, 6, 7, 8, 12, 16])
def test_tiny_cases(n_d, mode, grad_dtype):
    rng = np.random.default_rng(n_d * 100 + (mode == "distopt") * 7 + (grad_dtype == "bf16"))
    _run(_tiny_shapes(rng, n_d), n_d, mode, grad_dtype, seed=1000 + n_d)


@pytest.mark.parametrize("n_d", [9, 13, 33, 64])
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
def test_generic_rank_count(n_d, grad_dtype):
    """N_d without a specialised kernel, up to the maximum of 64."""
    rng = np.random.default_rng(n_d)
    _run(_tiny_shapes(rng, n_d) + [(3 * n_d + 1, 17)], n_d, "fsdp2", grad_dtype, seed=2000 + n_d)


@pytest.mark.parametrize("n_rep,n_shard", [(2, 2), (2, 4), (2, 8), (4, 2), (4, 4),   # bulk-copy kernels
                                           (2, 3), (3, 2), (2, 1), (4, 1), (8, 8)])  # generic kernel
@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
def test_hsdp_cases(n_rep, n_shard, grad_dtype):
    """HSDP: reduce-scatter inside each replica group, all-reduce across groups,
    each group's own copy of the state, gather within the group."""
    rng = np.random.default_rng(n_rep * 31 + n_shard)
    shapes = _tiny_shapes(rng, n_shard) + [(4097,), (3 * n_shard + 1, 67)]
    _run(shapes, n_rep * n_shard, "hsdp", grad_dtype, seed=3000 + n_rep * n_shard, n_rep=n_rep)


@pytest.mark.parametrize("n_d,mode", [(3, "fsdp2"), (6, "fsdp2"), (6, "distopt"), (8, "fsdp2")])
def test_several_tiles_ragged(n_d, mode):
    """Segments spanning many 4096-element tiles, starting and ending off
    vector boundaries, with rows not divisible by N_d."""
    shapes = [(3001, 7), (5, 4099), (1,), (12289,), (777, 64), (2, 3, 5), (4097,), (64, 129)]
    stats = _run(shapes, n_d, mode, "f32", seed=31)
    assert stats["param_max_ulp"] <= 1


def test_qwen3_layer_workload_both_entries():
    w = workload(0)
    stats = _run(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed)
    assert stats["master_max_scaled_err"] <= 16 and stats["exp_avg_sq_max_scaled_err"] <= 16
    # the production entry writes the same bits as the debug entry
    a = DeviceCase(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed)
    b = DeviceCase(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed)
    a.step(w.step, debug=False)
    b.step(w.step, debug=True)
    torch.cuda.synchronize()
    for x, y in zip(a.state + a.params, b.state + b.params):
        assert np.array_equal(x.bits(), y.bits())


def test_deterministic_and_stream_ordered():
    w = workload(0)
    outs = []
    for _ in range(2):
        c = DeviceCase(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            c.step(w.step, debug=False)
            c.step(w.step + 1, debug=False)
        s.synchronize()
        outs.append([x.bits() for x in c.state + c.params])
    for x, y in zip(*outs):
        assert np.array_equal(x, y)


def test_zero_learning_rate_only_moves_adam_state():
    shapes = [(40, 9), (7,)]
    hp = dict(HP, lr=0.0)
    dev = DeviceCase(shapes, 4, "fsdp2", "f32", 5)
    ora = OracleCase(shapes, 4, "fsdp2", "f32", 5)
    before = dev.state[0].bits().copy()
    dev.step(3, hp=hp)
    ora.step(3, hp=hp)
    torch.cuda.synchronize()
    compare(dev, ora)
    assert np.array_equal(dev.state[0].bits(), before)


def test_empty_and_all_padding_plans():
    # no parameters, a zero-row parameter, and rows=1 over 8 ranks (7 pad-only shards)
    for shapes in ([], [(0, 4)], [(1,)], [(1, 3), (0,), (2,)]):
        _run(shapes, 8, "fsdp2", "f32", seed=3, steps=(1,))
    _run([(1,)], 8, "distopt", "f32", seed=3, steps=(1,))


def test_exact_size_torch_buffers_pass_the_allocation_check():
    """Buffers of exactly the planned size (fresh torch allocations) are accepted
    by the driver range check and give the oracle's result."""
    shapes = [(1000, 4), (3,)]
    plan = fsp.plan_layout(shapes, 2)
    n = plan.full_len_padded
    grads = [torch.zeros(n, device="cuda") for _ in range(2)]
    state = [torch.zeros(plan.state_len_total, device="cuda") for _ in range(3)]
    params = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    fsp.sharded_step(plan, grads, *state, params, HP, 1)
    torch.cuda.synchronize()
    # zero grads and state: only weight decay acts, and 0 * (1 - lr wd) = 0
    assert not any(bool(t.any()) for t in state + params)


def test_guarded_buffers_catch_writes():
    """The guard-band helper itself notices a write just outside a buffer."""
    g = Guarded(100, torch.float32, 0)
    assert g.guards_intact()
    g.raw[g.g + 100] = 7
    assert not g.guards_intact()
