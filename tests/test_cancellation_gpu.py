"""GPU parity where the master update cancels: theta (1 - lr wd) placed next
to the step u, at depths from 2^-1 to 2^-30 of theta, so that most elements
take the kernel's float-pair evaluation and the rest its fp32 one.  Against
the oracle: state within the bars, params within one bf16 ulp on every
element.  Inputs are built on the host from the oracle's own update (with the
weight decay off, theta - theta' is u)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
import synth_inputs as S
from oracle import step as OS

from gpu_cases import HP, STATE_SENTINEL, DeviceCase, OracleCase, compare, ensure_built

pytestmark = pytest.mark.gpu

SHAPES = [(1000, 64), (4099,), (17, 3)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _upload(buf, bits: np.ndarray) -> None:
    view = bits.view(np.int32 if bits.dtype.itemsize == 4 else np.int16)
    buf.raw[buf.g:buf.g + buf.n].copy_(torch.from_numpy(view.copy()).cuda())


def _cancelling_case(n_d, t, seed, mode="fsdp2", n_rep=1, grad_dtype="f32"):
    dev = DeviceCase(SHAPES, n_d, mode, grad_dtype, seed, n_rep)
    ora = OracleCase(SHAPES, n_d, mode, grad_dtype, seed, n_rep)
    n = dev.plan.full_len_padded
    rng = np.random.default_rng(seed)
    # every rank holds the same gradient; G is its (grouped) rank-ordered sum / N_d
    if grad_dtype == "f32":
        g = S.grad_f32(seed, 0, np.arange(n))
        gw = g
    else:
        g = S.grad_bf16_bits(seed, 0, np.arange(n))
        gw = OS.bf16_bits_to_f32(g)
    G = OS.average(OS.hybrid_sum([gw] * n_d, n_rep), n_d)
    th, m, v = S.master_f32(seed, np.arange(n)), S.adam_m_f32(seed, np.arange(n)), S.adam_v_f32(seed, np.arange(n))
    # u from the oracle's update without weight decay, then theta such that
    # theta (1 - lr wd) = u (1 + e), e of either sign and 2^-1 .. 2^-30 in size
    th0, _, _ = OS.adamw(th, m, v, G, dict(HP, weight_decay=0.0), t)
    u = th.astype(np.float64) - th0.astype(np.float64)
    decay = 1.0 - float(np.float32(HP["lr"])) * float(np.float32(HP["weight_decay"]))
    e = rng.choice([-1.0, 1.0], n) * 2.0 ** -rng.uniform(1, 30, n)
    theta = (u / decay * (1.0 + e)).astype(np.float32)
    keep = rng.random(n) < 0.1            # a tenth keep their ordinary masters
    theta[keep] = th[keep]
    for q in range(n_d):
        _upload(dev.grads[q], g.view(np.uint32) if grad_dtype == "f32" else g)
        ora.grads[q] = g.copy()
    for k, full in enumerate((theta, m, v)):
        slots = np.full(dev.plan.state_len_total, STATE_SENTINEL, np.uint32).view(np.float32)
        slots[ora.si] = full[ora.fi]
        _upload(dev.state[k], slots.view(np.uint32))
        ora.state[k] = slots.copy()
    torch.cuda.synchronize()
    return dev, ora


@pytest.mark.parametrize("n_d,t,mode,n_rep,gd", [(4, 10, "fsdp2", 1, "f32"), (8, 1, "fsdp2", 1, "f32"),
                                                 (4, 1000, "fsdp2", 1, "f32"), (9, 10, "fsdp2", 1, "f32"),
                                                 (8, 10, "hsdp", 2, "f32"), (6, 3, "distopt", 1, "f32"),
                                                 (16, 10, "fsdp2", 1, "bf16")])
def test_cancelling_updates_match_the_oracle(n_d, t, mode, n_rep, gd):
    """The bulk kernel (N_d 4, 8, 6, 16 with bf16 gradients and the HSDP 4 x 2
    mesh) and the per-thread kernel (N_d 9)."""
    dev, ora = _cancelling_case(n_d, t, 70 + n_d + t, mode, n_rep, gd)
    before = ora.state[0][ora.si].astype(np.float64)
    dev.step(t)
    ora.step(t)
    torch.cuda.synchronize()
    after = ora.state[0][ora.si].astype(np.float64)
    # most elements cancel below 2^-10 of theta: the float-pair path is taken
    deep = np.abs(after) < 2.0 ** -10 * np.abs(before)
    assert deep.mean() > 0.5
    compare(dev, ora)
    assert fsp.device_error() == 0


def test_device_resident_t_gives_the_same_bits_on_cancelling_updates():
    """The bias-correction scalars (float pairs) computed on the device from a
    device-resident t equal the host's bit for bit: the float-pair path, which
    uses their low parts, gives the same state and params."""
    ref, _ = _cancelling_case(8, 10, 91)
    dev, _ = _cancelling_case(8, 10, 91)
    t = torch.tensor([10], dtype=torch.int64, device="cuda")
    ref.step(10, debug=False)
    fsp.sharded_step_device_t(dev.plan, [g.t for g in dev.grads], *[s.t for s in dev.state],
                              [p.t for p in dev.params], HP, t, advance=False)
    torch.cuda.synchronize()
    for x, y in zip(ref.state + ref.params, dev.state + dev.params):
        assert np.array_equal(x.bits(), y.bits())
    assert fsp.device_error() == 0
