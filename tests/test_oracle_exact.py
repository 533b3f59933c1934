"""The oracle's AdamW against exact arithmetic (CPU only).

The oracle evaluates the update in fp64 and rounds the results to fp32; the
GPU parity bar (bf16 params within one ulp of the oracle's cast) is only as
good as that rounding where theta' = theta (1 - lr wd) - u cancels.  Here the
same update is evaluated with 60 significant decimal digits (Python's decimal
module: the fp32 inputs and hyper-parameters are exact binary fractions, the
bias corrections b^t are exact products, and only the square root and the
divisions round, far below fp32's precision), rounded correctly to fp32, and
the oracle's fp32 results must equal it - on random elements and on elements
placed at cancellation depths down to 2^-30 of theta.
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest

import synth_inputs as S
from oracle import step as O

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
getcontext().prec = 60


def _dec(x) -> Decimal:
    """The exact value of a float (fp32 values widen to fp64 exactly)."""
    return Decimal(float(x))


def _round_f32(x: Decimal) -> np.float32:
    """x rounded to the nearest fp32, ties to even (exact: the candidates are
    compared against x itself, not against a double-rounded value)."""
    f = np.float32(float(x))                      # within one fp32 ulp of x
    lo, hi = (np.nextafter(f, np.float32(-np.inf)), f) if _dec(f) > x else (f, np.nextafter(f, np.float32(np.inf)))
    dl, dh = x - _dec(lo), _dec(hi) - x
    if dl < dh:
        return lo
    if dh < dl:
        return hi
    return lo if (lo.view(np.uint32) & 1) == 0 else hi


def _exact_adamw(theta, m, v, g, t):
    """theta', m', v' of the decoupled, bias-corrected AdamW, to 60 digits."""
    h = O.hparams_f32(HP)
    lr, b1, b2, eps, wd = (_dec(h[k]) for k in ("lr", "beta1", "beta2", "eps", "weight_decay"))
    th, mm, vv, gg = _dec(theta), _dec(m), _dec(v), _dec(g)
    m1 = b1 * mm + (1 - b1) * gg
    v1 = b2 * vv + (1 - b2) * gg * gg
    bc1 = 1 - b1 ** t
    bc2 = 1 - b2 ** t
    th1 = th - lr * wd * th - lr * (m1 / bc1) / ((v1 / bc2).sqrt() + eps)
    return th1, m1, v1


def _elements(n, seed, t):
    idx = np.arange(n)
    g = O.average(O.rank_ordered_sum([S.grad_f32(seed, q, idx) for q in range(4)]), 4)
    th, m, v = S.master_f32(seed, idx), S.adam_m_f32(seed, idx), S.adam_v_f32(seed, idx)
    # half of them: theta (1 - lr wd) placed next to u, 2^-1 .. 2^-30 of theta away
    rng = np.random.default_rng(seed)
    th0, _, _ = O.adamw(th, m, v, g, dict(HP, weight_decay=0.0), t)
    u = th.astype(np.float64) - th0.astype(np.float64)
    decay = 1.0 - float(np.float32(HP["lr"])) * float(np.float32(HP["weight_decay"]))
    e = rng.choice([-1.0, 1.0], n) * 2.0 ** -rng.uniform(1, 30, n)
    near = (u / decay * (1.0 + e)).astype(np.float32)
    pick = rng.random(n) < 0.5
    th = np.where(pick, near, th).astype(np.float32)
    return th, m, v, g


@pytest.mark.parametrize("t", [1, 10, 1000])
def test_oracle_rounds_the_exact_update(t):
    """Each fp32 result is the exact value rounded to nearest, up to the fp64
    evaluation's own error: a few fp64 roundings, each at most 2^-53 of a
    term, bound it by 2^-50 of the terms' size for m' and v' and by 2^-48 for
    theta' (|theta| + |u| with u = theta (1 - lr wd) - theta'), so the result
    must lie between the roundings of exact -/+ that bound.  Away from fp32
    midpoints and deep cancellation the two coincide and the result is the
    correctly rounded exact value; where theta' cancels to 2^-28 of theta the
    bound spans several fp32 ulps of theta' but still far less than one bf16
    ulp."""
    n = 3000
    th, m, v, g = _elements(n, 51 + t, t)
    got_th, got_m, got_v = O.adamw(th, m, v, g, HP, t)
    h = O.hparams_f32(HP)
    b1, b2, lr, wd = (_dec(h[k]) for k in ("beta1", "beta2", "lr", "weight_decay"))
    deep = ambiguous = rounded = 0
    for i in range(n):
        th1, m1, v1 = _exact_adamw(th[i], m[i], v[i], g[i], t)
        tt, mm, vv, gg = _dec(th[i]), _dec(m[i]), _dec(v[i]), _dec(g[i])
        u = tt * (1 - lr * wd) - th1
        bounds = (Decimal(2) ** -48 * (abs(tt) + abs(u)),
                  Decimal(2) ** -50 * (abs(b1 * mm) + abs((1 - b1) * gg)),
                  Decimal(2) ** -50 * (b2 * vv + (1 - b2) * gg * gg))
        for name, got, want, eps in (("theta", got_th[i], th1, bounds[0]), ("m", got_m[i], m1, bounds[1]),
                                     ("v", got_v[i], v1, bounds[2])):
            lo, hi = _round_f32(want - eps), _round_f32(want + eps)
            assert lo <= got <= hi, (name, i, float(got), str(want))
            ambiguous += lo != hi
            if name == "theta":
                # the bf16 parameter the GPU must come within one ulp of: the cast of a value in that range
                b = O.bf16_rne(np.array([got, lo, hi], np.float32)).view(np.int16).astype(np.int64)
                assert min(b[1], b[2]) <= b[0] <= max(b[1], b[2])
        deep += abs(th1) < Decimal(2) ** -10 * abs(tt)
        rounded += got_th[i] == _round_f32(th1)
    assert deep > n // 4                # the cancellation regime is well represented
    assert ambiguous < n // 10          # the exact rounding alone decides most results
    assert rounded >= n - n // 100      # theta' is the correctly rounded exact value almost everywhere


def test_exact_rounding_helper():
    # ties to even, and values next to fp32 midpoints
    one = Decimal(1)
    ulp = Decimal(2) ** -23
    assert _round_f32(one + ulp / 2) == np.float32(1.0)                  # tie: even neighbour
    assert _round_f32(one + 3 * ulp / 2) == np.float32(1.0) + np.float32(2.0 ** -22)
    assert _round_f32(one + ulp / 2 + Decimal(10) ** -40) == np.float32(1.0) + np.float32(2.0 ** -23)
    assert _round_f32(-(one + ulp / 2 - Decimal(10) ** -40)) == np.float32(-1.0)
