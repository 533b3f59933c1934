"""GPU parity of the fused step on hand-placed edge values, against the oracle:
signed zeros, subnormal and smallest-normal gradients, gradients near 1e17,
exact cancellation across ranks, sums whose value depends on the rank order,
masters at 1e30 and at bf16 rounding ties, subnormal and huge Adam moments -
in fp32 and bf16 gradients, on specialised and generic rank counts, FSDP2,
DistOpt and HSDP.  The generator's inputs never reach these corners."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from oracle import step as OS

from gpu_cases import HP, STATE_SENTINEL, DeviceCase, OracleCase, compare, ensure_built

pytestmark = pytest.mark.gpu

SHAPES = [(37, 129), (4099,), (3, 5), (1,), (700, 9)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _upload(buf, bits: np.ndarray) -> None:
    """Bit patterns into a guarded device buffer (its guard bands untouched)."""
    view = bits.view(np.int32 if bits.dtype.itemsize == 4 else np.int16)
    buf.raw[buf.g:buf.g + buf.n].copy_(torch.from_numpy(view.copy()).cuda())


def _grads_f32(n_d: int, n: int, rng) -> np.ndarray:
    """Every rank's fp32 gradient; element f takes pattern f % 9."""
    g = rng.normal(0.0, 1e-3, size=(n_d, n)).astype(np.float32)
    k = np.arange(n) % 9
    q = np.arange(n_d, dtype=np.float64)[:, None]
    alt = np.where(np.arange(n_d)[:, None] % 2 == 0, 1.0, -1.0)
    g[:, k == 0] = 0.0
    g[:, k == 1] = np.where(alt > 0, 0.0, -0.0).astype(np.float32)                 # +0 and -0
    g[:, k == 2] = (alt * (q + 1) * 1e-41).astype(np.float32)                        # subnormal
    g[:, k == 3] = (1e17 * (q + 1) * np.where((q // 2) % 2 == 0, 1.0, -1.0)).astype(np.float32)
    cancel = np.zeros((n_d, 1), np.float32)
    if n_d >= 2:
        cancel[0], cancel[1] = 3.0, -3.0                                             # sums to exactly 0
    g[:, k == 4] = cancel
    order = np.array([[1e8, 1.0, -1e8, 1.0][r % 4] for r in range(n_d)], np.float32)[:, None]
    g[:, k == 5] = order                                                             # value set by the fold order
    g[:, k == 6] = (alt * np.float32(2.0 ** -126)).astype(np.float32)               # smallest normal
    g[:, k == 7] = (alt * 10.0 ** (q % 6 * 6 - 15)).astype(np.float32)              # 1e-15 .. 1e15 mixed
    return g


def _grads_bf16(n_d: int, n: int, rng) -> np.ndarray:
    """Every rank's bf16 gradient bits; element f takes pattern f % 6."""
    g = (rng.normal(0.0, 1e-3, size=(n_d, n)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    k = np.arange(n) % 6
    r = np.arange(n_d)[:, None]
    g[:, k == 0] = np.where(r % 2 == 0, 0x0000, 0x8000).astype(np.uint16)         # signed zeros
    g[:, k == 1] = ((1 + (0x15 * r) % 0x7E) | np.where(r % 2 == 0, 0, 0x8000)).astype(np.uint16)  # subnormals
    g[:, k == 2] = np.where(r % 2 == 0, 0x5C31, 0xDC30).astype(np.uint16)          # about +-2e17
    g[:, k == 3] = np.where(r == 0, 0x4040, np.where(r == 1, 0xC040, 0x0000)).astype(np.uint16)  # 3, -3, 0...
    g[:, k == 4] = np.array([[0x4CBF, 0x3F80, 0xCCBF, 0x3F80][x % 4] for x in range(n_d)],
                            np.uint16)[:, None]                                      # 1e8-ish, 1, -1e8-ish, 1
    return g


def _state(n: int, rng):
    """master, m, v by full index; element f takes pattern f % 7, f % 5, f % 4."""
    f = np.arange(n)
    th = rng.normal(0.0, 0.02, n).astype(np.float32)
    k = f % 7
    th[k == 1] = 0.0
    th[k == 2] = -0.0
    th[k == 3] = np.where(f[k == 3] % 2 == 0, 1e30, -1e30).astype(np.float32)
    th[k == 4] = 1e-30
    th[k == 5] = np.float32(3e-40)
    ties = (rng.integers(0x3C00, 0x4400, n).astype(np.uint32) << 16) | 0x8000        # bf16 halfway points
    th[k == 6] = ties[k == 6].view(np.float32)
    m = rng.normal(0.0, 1e-4, n).astype(np.float32)
    j = f % 5
    m[j == 0] = 0.0
    m[j == 2] = 1e10
    m[j == 3] = -1e-30
    m[j == 4] = np.float32(-5e-41)
    v = rng.uniform(0.0, 1e-6, n).astype(np.float32)
    i = f % 4
    v[i == 0] = 0.0
    v[i == 2] = 1e30
    v[i == 3] = np.float32(1e-40)
    return th, m, v


def _case(n_d, mode, grad_dtype, n_rep=1, seed=3):
    rng = np.random.default_rng(seed + 31 * n_d)
    dev = DeviceCase(SHAPES, n_d, mode, grad_dtype, seed, n_rep)
    ora = OracleCase(SHAPES, n_d, mode, grad_dtype, seed, n_rep)
    n = dev.plan.full_len_padded
    grads = _grads_f32(n_d, n, rng) if grad_dtype == "f32" else _grads_bf16(n_d, n, rng)
    for q in range(n_d):
        _upload(dev.grads[q], grads[q])
        ora.grads[q] = grads[q].copy()
    for k, full in enumerate(_state(n, rng)):
        slots = np.full(dev.plan.state_len_total, STATE_SENTINEL, np.uint32).view(np.float32)
        slots[ora.si] = full[ora.fi]
        _upload(dev.state[k], slots.view(np.uint32))
        ora.state[k] = slots.copy()
    torch.cuda.synchronize()
    return dev, ora


@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_d,mode,n_rep", [(4, "fsdp2", 1), (8, "distopt", 1), (9, "fsdp2", 1), (16, "fsdp2", 1),
                                            (8, "hsdp", 2)])
def test_edge_values_match_oracle(n_d, mode, n_rep, grad_dtype):
    dev, ora = _case(n_d, mode, grad_dtype, n_rep)
    for t in (1, 10):
        dev.step(t)
        ora.step(t)
        torch.cuda.synchronize()
        compare(dev, ora)      # reduced gradient bit-exact, state within the bars, params within 1 bf16 ulp
        # the next step starts both sides from the device's state: where
        # theta' = theta (1 - lr wd) - u cancels (v = 0 makes u ~ lr m / eps),
        # the few ulps by which two fp32-accurate states differ would
        # otherwise exceed the bar on the much smaller result
        ora.state = [d.bits().view(np.float32).copy() for d in dev.state]


def test_rank_order_decides_the_sum():
    """The pattern 1e8, 1, -1e8, 1, ... sums to 1 in rank order and to other
    values in other orders; the device's reduced gradient is the rank-order one."""
    dev, ora = _case(8, "fsdp2", "f32")
    dev.step(1)
    ora.step(1)
    torch.cuda.synchronize()
    red = dev.reduced.bits()[ora.si].view(np.float32)
    f = ora.fi
    assert np.all(red[f % 9 == 5] == np.float32(1.0) / np.float32(8))
    assert np.all(red[f % 9 == 4] == 0.0)
    compare(dev, ora)


def test_zero_learning_rate_rounds_ties_to_even():
    """lr = 0 keeps every master as it is, so the gathered params are the
    round-to-nearest-even bf16 of hand-placed halfway points, exactly."""
    hp = dict(HP, lr=0.0)
    dev, ora = _case(4, "fsdp2", "f32")
    before = dev.state[0].bits()[ora.si].view(np.float32).copy()
    dev.step(5, hp=hp)
    ora.step(5, hp=hp)
    torch.cuda.synchronize()
    after = dev.state[0].bits()[ora.si].view(np.float32)
    assert np.array_equal(after, before)                       # values (signed zeros compare equal)
    p = dev.params[0].bits()[ora.fi]
    want = OS.bf16_rne(before)
    nz = before != 0                                           # a zero's sign is not pinned
    assert np.array_equal(p[nz], want[nz]) and np.all(p[~nz] & 0x7FFF == 0)
    ties = ora.fi % 7 == 6
    assert ties.sum() > 100
    tb = before[ties].view(np.uint32)
    assert np.all(tb & 0xFFFF == 0x8000)
    assert np.array_equal(p[ties], ((tb >> 16) + ((tb >> 16) & 1)).astype(np.uint16))   # up only from odd
    compare(dev, ora)


@pytest.mark.parametrize("max_norm", [1.0, 1e30])
@pytest.mark.parametrize("n_d,mode", [(4, "fsdp2"), (8, "distopt"), (9, "fsdp2")])
def test_clipped_flow_on_edge_values(n_d, mode, max_norm):
    """Write-back, global norm (squares from 1e-82 to 1e34 in one sum) and the
    clipped update on the same hand-placed values."""
    from test_clip_gpu import _check, _clipped
    dev, ora = _case(n_d, mode, "f32")
    norm, coef = _clipped(dev, 10, max_norm)
    ora.prev = [a.copy() for a in ora.state]
    ora.hp = HP
    o_norm, o_coef = OS.sharded_step_clipped(ora.plan, ora.grads, *ora.state, ora.params, HP, 10, max_norm)
    _check(dev, ora, norm, coef, o_norm, o_coef)
    assert (coef < 1.0) == (max_norm < 1e20)


@pytest.mark.parametrize("n_d,mode,n_rep", [(4, "fsdp2", 1), (8, "distopt", 1), (8, "hsdp", 2)])
def test_unshard_of_edge_masters_is_the_exact_cast(n_d, mode, n_rep):
    """The unshard casts ties, subnormals, signed zeros and 1e30 exactly as
    the oracle's round-to-nearest-even (and the fp32 unshard copies them)."""
    dev, ora = _case(n_d, mode, "f32", n_rep)
    n = dev.plan.full_len_padded
    bf = [torch.full((n,), -1, dtype=torch.int16, device="cuda") for _ in range(n_d)]
    f32 = [torch.full((n,), -1, dtype=torch.int32, device="cuda") for _ in range(n_d)]
    fsp.unshard(dev.plan, dev.state[0].t, [b.view(torch.bfloat16) for b in bf])
    fsp.unshard(dev.plan, dev.state[0].t, [b.view(torch.float32) for b in f32], fp32=True)
    o_params = [np.full(n, 0xFFFF, np.uint16) for _ in range(n_d)]
    OS.unshard(ora.plan, ora.state[0], o_params)
    torch.cuda.synchronize()
    fi = ora.fi
    want32 = np.full(n, 0xFFFFFFFF, np.uint32)
    want32[fi] = ora.state[0][ora.si].view(np.uint32)
    for q in range(n_d):
        assert np.array_equal(bf[q].cpu().numpy().view(np.uint16), o_params[q])   # padding included
        assert np.array_equal(f32[q].cpu().numpy().view(np.uint32), want32)
    assert fsp.device_error() == 0


@pytest.mark.parametrize("n_d,mode", [(4, "fsdp2"), (8, "distopt"), (9, "fsdp2")])
def test_writeback_step_on_edge_values(n_d, mode):
    """The fused step with the write-back: the owners' grad slices hold the
    oracle's averaged gradient bit for bit, the rest of every grad buffer is
    unchanged, and state and params match the oracle as the plain step's do."""
    dev, ora = _case(n_d, mode, "f32")
    fsp.sharded_step_writeback(dev.plan, [g.t for g in dev.grads], *[s.t for s in dev.state],
                               [p.t for p in dev.params], HP, 10)
    written = [g.copy() for g in ora.grads]
    OS.reduce_scatter_write_back(ora.plan, written)
    ora.step(10)                                   # on the gradients as they were before the step
    torch.cuda.synchronize()
    for q in range(n_d):
        assert np.array_equal(dev.grads[q].bits(), written[q].view(np.uint32)), f"grad buffer {q}"
    compare(dev, ora, check_reduced=False)


@pytest.mark.parametrize("n_d,mode,n_rep,gd", [(4, "fsdp2", 1, "f32"), (8, "hsdp", 2, "bf16"), (9, "fsdp2", 1, "f32")])
def test_per_parameter_tensors_on_edge_values(n_d, mode, n_rep, gd):
    """The step on per-parameter tensors equals the flat step element for
    element on the same hand-placed values (state copied slot by slot)."""
    from test_params_gpu import ParamCase
    dev, _ = _case(n_d, mode, gd, n_rep)
    pc = ParamCase(dev, n_rep)
    flat_seg = {(s.param, s.rank): s for s in dev.plan.segments}
    for s in pc.plan.segments:
        f = flat_seg[(s.param, s.rank)]
        for dst, src in zip(pc.state, dev.state):
            dst.t[s.state_off:s.state_off + s.length] = src.t[f.state_off:f.state_off + f.length]
    for t in (1, 10):
        dev.step(t, debug=False)
        pc.step(t)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    pc.params_match_flat()
    assert pc.guards_intact() and dev.all_guards_intact() and fsp.device_error() == 0


@pytest.mark.parametrize("n_d,mode,n_rep", [(4, "fsdp2", 1), (8, "hsdp", 2), (9, "fsdp2", 1)])
def test_fp32_gather_and_zero3_steps_on_edge_values(n_d, mode, n_rep):
    """The same state as the plain step on the hand-placed values; the fp32
    all-gather writes the new master itself, bit for bit, into every rank's
    buffer (group's for HSDP); the ZeRO-3 step writes no parameter."""
    plain, ora = _case(n_d, mode, "f32", n_rep)
    f32, _ = _case(n_d, mode, "f32", n_rep)
    z3, _ = _case(n_d, mode, "f32", n_rep)
    n = plain.plan.full_len_padded
    bufs = [torch.full((n,), -1, dtype=torch.int32, device="cuda") for _ in range(n_d)]
    plain.step(10, debug=False)
    fsp.sharded_step_fp32_gather(f32.plan, [g.t for g in f32.grads], *[s.t for s in f32.state],
                                 [b.view(torch.float32) for b in bufs], HP, 10)
    fsp.sharded_step(z3.plan, [g.t for g in z3.grads], *[s.t for s in z3.state], None, HP, 10)
    torch.cuda.synchronize()
    for a, b, c in zip(plain.state, f32.state, z3.state):
        assert np.array_equal(a.bits(), b.bits()) and np.array_equal(a.bits(), c.bits())
    master = plain.state[0].bits()
    want = np.full(n, 0xFFFFFFFF, np.uint32)
    want[ora.fi] = master[ora.si]
    for q in range(n_d):      # (HSDP: each group gathers its own state copy; the copies are equal)
        assert np.array_equal(bufs[q].cpu().numpy().view(np.uint32), want)
    for p in z3.params:
        assert np.all(p.bits() == 0xFFFF)       # untouched: still the sentinel
    assert fsp.device_error() == 0
