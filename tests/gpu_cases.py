"""Shared machinery of the GPU parity tests: device buffers with guard bands,
inputs from the seeded generator, and comparison with the oracle."""
from __future__ import annotations

import os

import numpy as np
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
import synth_inputs as S
from oracle import plan as OP
from oracle import step as OS
from synth_inputs import device as D

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
GUARD_BYTES = 4096
STATE_SENTINEL = 0x7FC0DEAD          # a NaN pattern no computation produces
PARAM_SENTINEL = 0xFFFF              # bf16 NaN pattern
GUARD_WORD = 0x5A5A5A5A


def ensure_built():
    from fsdp_sharded_mixed_pass_gb300 import build
    from fsdp_sharded_mixed_pass_gb300 import fsp as B
    if not os.path.exists(B.LIB_PATH):
        build.build()
    if not os.path.exists(D.LIB):
        D.build()


class Guarded:
    """A device buffer of ``n`` elements with a guard band on both sides."""

    def __init__(self, n: int, dtype: torch.dtype, fill_bits: int, device="cuda"):
        esz = torch.tensor([], dtype=dtype).element_size()
        g = GUARD_BYTES // esz
        self.g, self.n = g, n
        int_dtype = {4: torch.int32, 2: torch.int16}[esz]
        self.raw = torch.empty(n + 2 * g, dtype=int_dtype, device=device)
        guard = np.array([GUARD_WORD], np.uint32).view(np.int32)[0] if esz == 4 else np.int16(0x5A5A)
        self.raw.fill_(int(guard))
        fill = np.array([fill_bits], np.uint32 if esz == 4 else np.uint16).view(
            np.int32 if esz == 4 else np.int16)[0]
        self.raw[g:g + n].fill_(int(fill))
        self.t = self.raw[g:g + n].view(dtype)
        self._guard = int(guard)

    def guards_intact(self) -> bool:
        return bool((self.raw[:self.g] == self._guard).all() and (self.raw[self.g + self.n:] == self._guard).all())

    def bits(self) -> np.ndarray:
        a = self.raw[self.g:self.g + self.n].cpu().numpy()
        return a.view(np.uint32 if a.dtype == np.int32 else np.uint16)


def ordered(bits: np.ndarray) -> np.ndarray:
    """Bit patterns mapped to integers that order like the float values."""
    if bits.dtype == np.uint32:
        i = bits.view(np.int32).astype(np.int64)
        return np.where(i < 0, -(2 ** 31) - i, i)
    i = bits.view(np.int16).astype(np.int64)
    return np.where(i < 0, -(2 ** 15) - i, i)


def ulp_dist(a_bits, b_bits) -> np.ndarray:
    return np.abs(ordered(a_bits) - ordered(b_bits))


def within_tol(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """|got - ref| <= 1e-6 * max(1, |ref|) elementwise (the stated bar)."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    return np.abs(g - r) <= 1e-6 * np.maximum(1.0, np.abs(r))


# fp32 arithmetic against the fp64 oracle.  Each of m', v' and theta' is a
# short sum of terms (m' = b1 m + (1 - b1) G, v' = b2 v + (1 - b2) G^2,
# theta' = theta (1 - lr wd) - u), and a few fp32 roundings stay far below
# 2^-20 of the terms' scale:
#   m', v':  |old| + |new| bounds every term;
#   theta':  |theta| + |theta'| bounds theta (1 - lr wd) and u, and u inherits
#            m''s error: u is proportional to m', and m' can cancel, so u's
#            error scale is |u| (2|m| + |m'| + 2^-125) / |m'| - the last term
#            because below 2^-126 the fp32 grid that m' is rounded to is
#            evenly spaced at 2^-149 (subnormals), so each of its two
#            roundings may be off by 2^-150 = 2^-24 * 2^-126 whatever |m'| is;
#            where m' itself rounds to 0 the whole of u is allowed (such a u
#            is at most lr / (bc1 eps) times 2^-150: about 2^-132 with the
#            tests' hyper-parameters at t = 1).
# Near-cancellation makes ulp distance meaningless (a result can be tiny
# while its terms are not), and the absolute bar above sees a dropped
# weight-decay term (lr wd theta) only where |theta| > 0.033, so parity also
# requires this.
SCALED_BOUND = 2.0 ** -20


def scaled_err(got: np.ndarray, ref: np.ndarray, old: np.ndarray, extra=0.0) -> np.ndarray:
    """|got - ref| in units of 2^-24 (|old| + |ref| + extra)."""
    g = got.astype(np.float64)
    r = ref.astype(np.float64)
    scale = np.abs(old.astype(np.float64)) + np.abs(r) + extra
    return np.abs(g - r) / np.maximum(scale * 2.0 ** -24, 1e-45)


def master_extra_scale(th_old, th_ref, m_old, m_ref, hp=HP) -> np.ndarray:
    """|u| (2|m| + |m'| + 2^-125) / |m'|: the part of theta''s error scale
    carried in from m' (the last term: m''s two roundings on the subnormal
    grid); where the reference m' is 0 it lets theta' miss all of u."""
    decay = 1.0 - float(np.float32(hp["lr"])) * float(np.float32(hp["weight_decay"]))
    u = np.abs(th_old.astype(np.float64) * decay - th_ref.astype(np.float64))
    mo = np.abs(m_old.astype(np.float64))
    mr = np.abs(m_ref.astype(np.float64))
    with np.errstate(divide="ignore", invalid="ignore"):
        return np.where(mr > 0, u * (2 * mo + mr + 2.0 ** -125) / mr, u * 2.0 ** 20)


def state_errors(got, ref, old, hp=HP):
    """Scaled errors of (master, m, v) given (got, ref, old) triples of arrays."""
    extra = master_extra_scale(old[0], ref[0], old[1], ref[1], hp)
    return [scaled_err(got[0], ref[0], old[0], extra), scaled_err(got[1], ref[1], old[1]),
            scaled_err(got[2], ref[2], old[2])]


# The bf16 params: within one bf16 ulp of the oracle's cast, everywhere (the
# stated bar), and exactly bf16_rne of the device's own fp32 master.
PARAM_ULP_BAR = 1


def check_params(param_bits, ref_bits, fi, what="param copy"):
    """Owned elements within PARAM_ULP_BAR bf16 ulps of the oracle; all others
    (padding) identical to the oracle's buffer (the sentinel)."""
    d = ulp_dist(param_bits[fi], ref_bits[fi])
    bad = d > PARAM_ULP_BAR
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements more than {PARAM_ULP_BAR} bf16 ulp from the oracle "
                           f"(worst {int(d.max())})")
    rest = np.ones(param_bits.size, bool)
    rest[fi] = False
    assert np.array_equal(param_bits[rest], ref_bits[rest]), f"{what}: a padding element was written"


class DeviceCase:
    """A plan plus guarded device buffers filled from the seeded generator."""

    def __init__(self, shapes, n_d, mode, grad_dtype, seed, n_rep=1):
        self.shapes, self.n_d, self.mode, self.grad_dtype, self.seed = shapes, n_d, mode, grad_dtype, seed
        self.plan = fsp.plan_layout(shapes, n_d, mode, n_replicate=n_rep)
        p = self.plan
        gdt = torch.float32 if grad_dtype == "f32" else torch.bfloat16
        self.grads = [Guarded(p.full_len_padded, gdt, 0) for _ in range(n_d)]
        for q, g in enumerate(self.grads):
            D.fill_grad(g.t, seed, q, grad_dtype)
        self.state = [Guarded(p.state_len_total, torch.float32, STATE_SENTINEL) for _ in range(3)]
        self.reduced = Guarded(p.state_len_total, torch.float32, STATE_SENTINEL)
        D.fill_state_segments(self.state[0].t, self.state[1].t, self.state[2].t, seed,
                              [(s.full_off, s.state_off, s.length) for s in p.segments])
        self.params = [Guarded(p.full_len_padded, torch.bfloat16, PARAM_SENTINEL) for _ in range(n_d)]
        torch.cuda.synchronize()

    def step(self, t, debug=True, hp=HP):
        st = [s.t for s in self.state]
        if debug:
            fsp.sharded_step_debug(self.plan, [g.t for g in self.grads], *st, [q.t for q in self.params], hp, t,
                                   self.reduced.t)
        else:
            fsp.sharded_step(self.plan, [g.t for g in self.grads], *st, [q.t for q in self.params], hp, t)

    def all_guards_intact(self):
        return all(b.guards_intact() for b in self.grads + self.state + self.params + [self.reduced])


class OracleCase:
    """The same inputs on the host, from the oracle's planner and the host generator."""

    def __init__(self, shapes, n_d, mode, grad_dtype, seed, n_rep=1):
        self.plan = OP.plan_layout(shapes, n_d, mode, n_rep=n_rep)
        self.grad_dtype = grad_dtype
        p = self.plan
        idx = np.arange(p.full_len_padded)
        if grad_dtype == "f32":
            self.grads = [S.grad_f32(seed, q, idx) for q in range(n_d)]
        else:
            self.grads = [S.grad_bf16_bits(seed, q, idx) for q in range(n_d)]
        self.fi, self.si = OP.owned_indices(p)
        self.state = []
        for fn in (S.master_f32, S.adam_m_f32, S.adam_v_f32):
            a = np.full(p.state_len_total, STATE_SENTINEL, np.uint32).view(np.float32)
            a[self.si] = fn(seed, self.fi)
            self.state.append(a)
        self.params = [np.full(p.full_len_padded, PARAM_SENTINEL, np.uint16) for _ in range(n_d)]
        self.reduced = np.full(p.state_len_total, STATE_SENTINEL, np.uint32).view(np.float32)

    def step(self, t, hp=HP):
        self.prev = [a.copy() for a in self.state]
        self.hp = hp
        OS.sharded_step(self.plan, self.grads, self.grad_dtype, *self.state, self.params, hp, t,
                        reduced_out=self.reduced)


def compare(dev: DeviceCase, ora: OracleCase, check_reduced=True) -> dict:
    """Asserts parity; returns error statistics."""
    si = ora.si
    stats = {}
    names = ("master", "exp_avg", "exp_avg_sq")
    gots = [d.bits() for d in dev.state]
    errs = state_errors([g[si].view(np.float32) for g in gots], [o[si] for o in ora.state],
                        [o[si] for o in ora.prev], ora.hp)
    for name, got, o, se in zip(names, gots, ora.state, errs):
        want = o.view(np.uint32)
        g32, r32 = got[si].view(np.float32), want[si].view(np.float32)
        ok = within_tol(g32, r32)
        assert ok.all(), f"{name}: {int((~ok).sum())} of {ok.size} outside 1e-6*max(1,|ref|)"
        stats[name + "_max_scaled_err"] = float(se.max()) if si.size else 0.0
        assert np.all(se <= SCALED_BOUND * 2 ** 24), f"{name}: error {se.max():.1f} x 2^-24 of the terms' scale"
        stats[name + "_max_ulp"] = int(ulp_dist(got[si], want[si]).max()) if si.size else 0
        # slots nobody owns keep their sentinel
        untouched = np.ones(got.size, bool)
        untouched[si] = False
        assert np.all(got[untouched] == STATE_SENTINEL), f"{name}: padding slot written"
    if check_reduced:
        got = dev.reduced.bits()
        assert np.array_equal(got[si], ora.reduced.view(np.uint32)[si]), "reduced gradient not bit-exact"
    master_bits = dev.state[0].bits()
    th_dev = master_bits[si].view(np.float32)
    cast = OS.bf16_rne(th_dev)
    p0 = dev.params[0].bits()
    assert np.array_equal(p0[ora.fi], cast), "params != bf16_rne(device master)"
    for q, prm in enumerate(dev.params):
        got = prm.bits() if q else p0
        assert np.array_equal(got, p0), f"param copy {q} differs from copy 0"
        check_params(got, ora.params[q], ora.fi, f"param copy {q}")
    stats["param_max_ulp"] = int(ulp_dist(p0, ora.params[0]).max(initial=0))
    assert dev.all_guards_intact(), "guard band overwritten"
    assert fsp.device_error() == 0, "a bounded wait in the step kernel ran out"
    return stats
