"""Oracle of the sharded mixed-precision step (test infrastructure only).

The step, as the pages describe it ("Parallelism strategies: which state to
shard", section 二.2 "ZeRO-1 / ZeRO-2"; "FSDP2 Qwen3 Decoder Layer
Walkthrough", section "Backward 简述"; "07 · 显存模型", section 2.1):

1. reduce-scatter: every rank ends with the sum over all ranks of its own 1/N_d
   slice of the gradient, averaged.  The sum is an fp32 left fold in rank
   order 0..N_d-1 (the grad buffer is fp32 - Megatron's grad_reduce_in_fp32 -
   and bf16 gradients are widened exactly to fp32 before the fold), followed by
   an IEEE fp32 division by N_d;
2. an optimizer update of the rank's fp32 master / Adam m / Adam v shard, with
   no communication;
3. the updated master is cast to bf16 and all-gathered so every rank's full
   bf16 param buffer holds it.

Because all-reduce = reduce-scatter + all-gather and ZeRO-1 only puts the
optimizer between the two halves, the result must equal the unsharded
definition: all-reduce-average the full gradient, run the optimizer over the
full buffer, cast, and copy to every rank (``unsharded_step``).

AdamW (the pages never print it; this is the reading taken): with t the 1-based
index of this update,
    m' = b1 m + (1 - b1) G
    v' = b2 v + (1 - b2) G^2
    theta' = theta - lr wd theta - lr (m' / (1 - b1^t)) / (sqrt(v' / (1 - b2^t)) + eps)
i.e. bias-corrected Adam with eps outside the square root and weight decay
decoupled and applied to the old master.  It is evaluated in fp64 from the fp32
inputs; the hyper-parameters are first rounded to fp32 (the width they have at
the library boundary); the stored master/m/v are the fp64 results rounded to
fp32 and the bf16 param is the round-to-nearest-even of the stored fp32 master.
"""
from __future__ import annotations

import numpy as np

from .plan import Plan


# ---------------------------------------------------------------------------
# Element types
# ---------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit pattern, round to nearest, ties to even (finite inputs).

    Adds 0x7FFF plus the lowest kept bit to the 32-bit pattern and keeps the
    high half: below the halfway point the carry does not reach bit 16, above
    it it does, and exactly at halfway it does only when the kept part is odd.
    """
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def grads_as_f32(g: np.ndarray, grad_dtype: str) -> np.ndarray:
    if grad_dtype == "f32":
        return np.asarray(g, dtype=np.float32)
    if grad_dtype == "bf16":
        return bf16_bits_to_f32(g)
    raise ValueError(grad_dtype)


# ---------------------------------------------------------------------------
# Stage 1: reduce-scatter (and its all-reduce counterpart)
# ---------------------------------------------------------------------------

def rank_ordered_sum(slices) -> np.ndarray:
    """fp32 left fold ((g_0 + g_1) + g_2) + ... over the ranks' slices."""
    acc = np.zeros(np.shape(slices[0]), dtype=np.float32)
    for s in slices:
        acc = (acc + np.asarray(s, dtype=np.float32)).astype(np.float32)
    return acc


def average(summed: np.ndarray, n_d: int) -> np.ndarray:
    """IEEE fp32 division of the rank-ordered sum by N_d."""
    return (summed / np.float32(n_d)).astype(np.float32)


def hybrid_sum(slices, n_rep: int):
    """HSDP reduction ("Parallelism strategies: which state to shard", section
    二.6): a reduce-scatter inside each replica group - the rank-ordered fold of
    that group's N_s slices - then an all-reduce across the N_r groups - the
    fold of the groups' partial sums in group order.  Global rank = r*N_s + j.
    With N_r = 1 or N_s = 1 it is the plain rank-ordered fold."""
    n_shard = len(slices) // n_rep
    partials = [rank_ordered_sum(slices[r * n_shard:(r + 1) * n_shard]) for r in range(n_rep)]
    return rank_ordered_sum(partials)


def reduce_scatter(plan: Plan, grads, grad_dtype: str = "f32", mean: bool = True):
    """Per segment (in plan order), the owner's reduced slice of the gradient."""
    out = []
    for seg in plan.segments:
        sl = slice(seg.full_off, seg.full_off + seg.length)
        s = hybrid_sum([grads_as_f32(g[sl], grad_dtype) for g in grads], plan.n_rep)
        out.append(average(s, plan.n_d) if mean else s)
    return out


def all_reduce(grads, grad_dtype: str = "f32", length: int | None = None, mean: bool = True, n_rep: int = 1):
    """Unsharded counterpart: every element reduced, nobody owns anything
    (with the HSDP grouping when n_rep > 1)."""
    n = len(grads)
    sl = slice(0, length)
    s = hybrid_sum([grads_as_f32(g[sl], grad_dtype) for g in grads], n_rep)
    return average(s, n) if mean else s


# ---------------------------------------------------------------------------
# Stage 2: AdamW on a shard
# ---------------------------------------------------------------------------

def hparams_f32(hp: dict) -> dict:
    """Hyper-parameters as the fp32 numbers the library boundary carries."""
    return {k: float(np.float32(hp[k])) for k in ("lr", "beta1", "beta2", "eps", "weight_decay")}


def adamw(theta, m, v, g, hp: dict, t: int):
    """Decoupled, bias-corrected AdamW in fp64; returns fp32 (theta', m', v')."""
    h = hparams_f32(hp)
    lr, b1, b2, eps, wd = h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"]
    theta = np.asarray(theta, dtype=np.float32).astype(np.float64)
    m = np.asarray(m, dtype=np.float32).astype(np.float64)
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    g = np.asarray(g, dtype=np.float32).astype(np.float64)

    m_new = b1 * m + (1.0 - b1) * g
    v_new = b2 * v + (1.0 - b2) * g * g
    m_hat = m_new / (1.0 - b1 ** t)
    v_hat = v_new / (1.0 - b2 ** t)
    theta_new = theta - lr * wd * theta - lr * m_hat / (np.sqrt(v_hat) + eps)
    return theta_new.astype(np.float32), m_new.astype(np.float32), v_new.astype(np.float32)


# ---------------------------------------------------------------------------
# Stage 3: cast and all-gather
# ---------------------------------------------------------------------------

def all_gather(plan: Plan, per_segment_values, params) -> None:
    """Write each owner's values into the full buffer of every rank of its
    group (all N_d ranks; HSDP: the N_s ranks of the owner's replica group)."""
    group = plan.n_shard
    for seg, vals in zip(plan.segments, per_segment_values):
        sl = slice(seg.full_off, seg.full_off + seg.length)
        first = (seg.rank // group) * group
        for q in range(first, first + group):
            params[q][sl] = vals


# ---------------------------------------------------------------------------
# The step
# ---------------------------------------------------------------------------

def sharded_step(plan: Plan, grads, grad_dtype: str, master, m, v, params, hp: dict, t: int,
                 reduced_out=None) -> None:
    """In place: master/m/v (state layout) and params[q] (full layout, bf16 bits).

    ``reduced_out`` (optional, state layout, fp32) receives the averaged shard
    gradient of every valid element.
    """
    if t < 1:
        raise ValueError("t is the 1-based index of the update")
    reduced = reduce_scatter(plan, grads, grad_dtype, mean=True)
    casts = []
    for seg, g in zip(plan.segments, reduced):
        st = slice(seg.state_off, seg.state_off + seg.length)
        th, mm, vv = adamw(master[st], m[st], v[st], g, hp, t)
        master[st], m[st], v[st] = th, mm, vv
        if reduced_out is not None:
            reduced_out[st] = g
        casts.append(bf16_rne(th))
    all_gather(plan, casts, params)


def unsharded_step(grads, grad_dtype: str, theta_full, m_full, v_full, n_valid: int, hp: dict, t: int,
                   n_rep: int = 1):
    """Plain data-parallel definition on logical (full-index) arrays.

    Returns (theta', m', v', bf16 bits) over the first ``n_valid`` elements; each
    of the N_d ranks would hold a copy of the bf16 bits.
    """
    g = all_reduce(grads, grad_dtype, n_valid, mean=True, n_rep=n_rep)
    th, mm, vv = adamw(theta_full[:n_valid], m_full[:n_valid], v_full[:n_valid], g, hp, t)
    return th, mm, vv, bf16_rne(th)


def elementwise_step(grad_columns, grad_dtype: str, theta, m, v, hp: dict, t: int, n_rep: int = 1):
    """The step for a sample of elements given their inputs directly.

    ``grad_columns[q]`` holds rank q's gradient at the sampled elements.  Used to
    check full-size runs one element at a time; it composes the same stages.
    """
    n_d = len(grad_columns)
    g = average(hybrid_sum([grads_as_f32(c, grad_dtype) for c in grad_columns], n_rep), n_d)
    th, mm, vv = adamw(theta, m, v, g, hp, t)
    return th, mm, vv, bf16_rne(th), g


def rs_update_ag(plan: Plan, grads, update) -> list:
    """reduce-scatter (sum) -> per-shard ``update`` -> all-gather, in fp32.

    Returns the N_d gathered fp32 buffers.  With ``update`` the identity this is
    an all-reduce (sum).
    """
    sums = reduce_scatter(plan, grads, "f32", mean=False)
    outs = [np.full(plan.full_len_padded, np.nan, dtype=np.float32) for _ in range(plan.n_d)]
    all_gather(plan, [np.asarray(update(s), dtype=np.float32) for s in sums], outs)
    return outs


# ---------------------------------------------------------------------------
# Megatron distributed-optimizer flow with gradient clipping
# ---------------------------------------------------------------------------
#
# The reduce-scatter leaves each rank's averaged shard of the gradient in that
# rank's own 1/N_d slice of its grad buffer ("07 · 显存模型", section 2.1 item 1:
# the buffer stays full size, the result is written back into the rank's
# slice).  Global-norm clipping is not on the pages; the reading taken is
# PyTorch's clip_grad_norm_: total norm = sqrt of the sum of squares of every
# reduced gradient element (each counted once), coefficient =
# min(1, max_norm / (norm + 1e-6)), every gradient element multiplied by it
# in fp32 before the optimizer.  Here the norm is taken in fp64 and the
# coefficient is rounded once to fp32.

def reduce_scatter_write_back(plan: Plan, grads, grad_dtype: str = "f32"):
    """Averaged shard gradients, also written into each owner's grad slice."""
    if grad_dtype != "f32":
        raise ValueError("write-back is defined for fp32 grad buffers")
    reduced = reduce_scatter(plan, grads, grad_dtype, mean=True)
    for seg, g in zip(plan.segments, reduced):
        grads[seg.rank][seg.full_off:seg.full_off + seg.length] = g
    return reduced


def global_grad_norm(reduced) -> float:
    """sqrt(sum of squares) over every reduced gradient element, in fp64."""
    total = 0.0
    for g in reduced:
        g64 = np.asarray(g, dtype=np.float32).astype(np.float64)
        total += float(np.dot(g64, g64))
    return float(np.sqrt(total))


def clip_coefficient(norm: float, max_norm) -> np.float32:
    c = float(np.float32(max_norm)) / (norm + 1e-6)
    return np.float32(min(1.0, c))


def sharded_step_clipped(plan: Plan, grads, master, m, v, params, hp: dict, t: int, max_norm):
    """reduce-scatter with write-back -> global norm -> clip -> AdamW -> cast ->
    all-gather.  Returns (norm, coefficient).  fp32 grads.  HSDP: after the
    all-reduce across replica groups every group's owner holds the same
    averaged slice, so each group's owner gets it written back, and the norm
    counts every element once (the first group's segments)."""
    reduced = reduce_scatter_write_back(plan, grads, "f32")
    norm = global_grad_norm([g for seg, g in zip(plan.segments, reduced) if seg.rank < plan.n_shard])
    coef = clip_coefficient(norm, max_norm)
    casts = []
    for seg, g in zip(plan.segments, reduced):
        st = slice(seg.state_off, seg.state_off + seg.length)
        gc = (g * coef).astype(np.float32)
        th, mm, vv = adamw(master[st], m[st], v[st], gc, hp, t)
        master[st], m[st], v[st] = th, mm, vv
        casts.append(bf16_rne(th))
    all_gather(plan, casts, params)
    return norm, coef


# ---------------------------------------------------------------------------
# FSDP2 unshard (all-gather before forward / backward)
# ---------------------------------------------------------------------------

def unshard(plan: Plan, master, params) -> None:
    """FSDP2's unshard of a parameter group: every rank's sharded fp32 param
    (here: its slots of the master buffer) is cast to the all-gather dtype
    (bf16, round to nearest even - MixedPrecisionPolicy's param dtype) and
    all-gathered into every rank's full buffer of its group ("Parallelism
    strategies: which state to shard", section 二.5: copy-in, one all-gather,
    copy-out; "FSDP2 Qwen3 Decoder Layer Walkthrough", section "Step 0")."""
    casts = [bf16_rne(master[seg.state_off:seg.state_off + seg.length]) for seg in plan.segments]
    all_gather(plan, casts, params)


def shard(plan: Plan, full, master) -> None:
    """FSDP2's shard of the full fp32 parameters ("Parallelism strategies:
    which state to shard", section 二.5: fully_shard splits every parameter on
    dim 0 into per-rank shards): each owned element goes to its state slot, in
    every replica group's copy for HSDP (the plan's segments list every copy).
    Slots no segment owns are left as they were."""
    full = np.asarray(full, dtype=np.float32)
    for seg in plan.segments:
        master[seg.state_off:seg.state_off + seg.length] = full[seg.full_off:seg.full_off + seg.length]
