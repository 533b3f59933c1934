"""Oracle layout planner (test infrastructure only; see ``oracle/__init__``).

Rules, each from the pages or, where they are silent, the plainest reading:

FSDP2 Shard(0)  ("FSDP2 Qwen3 Decoder Layer Walkthrough", section "FSDP2 设置"
    and the per-rank shard table; "Parallelism strategies: which state to
    shard", section 二.5 "FSDP1 与 FSDP2"): every parameter is split on dim 0
    into N_d shards.  With ``rows = shape[0]`` and ``cols`` the product of the
    other dims, the shard height is ``c = ceil(rows / N_d)``; rank r owns rows
    ``[r*c, min((r+1)*c, rows))`` (possibly none) and holds a padded shard of
    ``c*cols`` slots.  Parameters are concatenated in the given order, with no
    gaps, in each rank's full-size grad and param buffers.

DistOpt flat ("07 · 显存模型", section 2.1 item 1 and section 8 item 4;
    "Parallelism strategies: which state to shard", section 二.2): all
    parameters form one flat buffer of length P padded up to a multiple of
    lcm(N_d, 128); it is cut into N_d equal contiguous shards that ignore
    parameter boundaries.  State index = flat index; slots >= P are padding.

State placement (FSDP2; the pages are silent): the fp32 master/m/v buffers are
    rank-major - rank 0's shard, then rank 1's, ... - each rank's shard being
    ``state_len_per_rank`` slots.  Inside a rank, segments follow parameter
    order, and each starts at the first slot at or after the previous segment's
    end whose index is congruent to the segment's full-buffer offset modulo 16,
    so that both sides line up for vector access.  ``state_len_per_rank`` is the
    largest rank's extent rounded up to 16.  Gaps and shard padding are never
    written.

Per-parameter buffers ("Parallelism strategies: which state to shard",
    section 二.5: FSDP2 keeps every parameter, and its gradient, as a tensor of
    its own; copy-in gathers them before the reduce-scatter, copy-out scatters
    the all-gather's result back): with param_align = 16 the parameters sit in
    a virtual full index at offsets rounded up to multiples of 16 elements
    (our choice, so each tensor's vector boundaries line up with the index);
    the gaps belong to no rank.  Offsets, segments and state are otherwise as
    for flat buffers; param_align = 1 is the flat layout.

HSDP ("Parallelism strategies: which state to shard", section 二.6): the N_d
    ranks form an N_r x N_s mesh (replicate, shard); global rank = r * N_s + j.
    Inside each replica group the parameters are FSDP2 Shard(0) over N_s ranks;
    the N_r groups hold identical copies.  State: N_r copies of the N_s-rank
    FSDP2 state, replica r's copy at r * (N_s * state_len_per_rank).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

STATE_ALIGN = 16
DISTOPT_ALIGN = 128


@dataclass(frozen=True)
class Segment:
    param: int        # parameter index (-1 for a DistOpt shard, which spans params)
    rank: int
    full_off: int     # first element in every rank's full grad/param buffer
    state_off: int    # first slot in master/m/v
    length: int       # valid elements (owned by this rank)
    padded_len: int   # state slots reserved for this segment


@dataclass(frozen=True)
class Plan:
    mode: str
    n_d: int
    shapes: tuple
    param_offsets: tuple
    valid_elems: int          # P
    full_len_padded: int      # length of each grad / param buffer
    state_len_per_rank: int
    segments: tuple
    n_rep: int = 1            # HSDP replica groups (1 otherwise)

    @property
    def n_shard(self) -> int:
        return self.n_d // self.n_rep

    @property
    def state_len_total(self) -> int:
        return self.n_d * self.state_len_per_rank


def numel(shape) -> int:
    n = 1
    for d in shape:
        n *= d
    return n


def rows_cols(shape) -> tuple[int, int]:
    """Dim 0 and the product of the remaining dims (1 for a 1-D parameter)."""
    rows = shape[0]
    cols = 1
    for d in shape[1:]:
        cols *= d
    return rows, cols


def shard_rows(rows: int, n_d: int) -> int:
    """Padded shard height c = ceil(rows / N_d)."""
    return -(-rows // n_d)


def shard_shape(shape, n_d: int) -> tuple:
    """Per-rank (padded) local shard shape of a Shard(0) parameter."""
    return (shard_rows(shape[0], n_d),) + tuple(shape[1:])


def _offsets(shapes, align: int = 1):
    """Start of each parameter (rounded up to ``align``) and the extent."""
    offs, at = [], 0
    for s in shapes:
        at = -(-at // align) * align
        offs.append(at)
        at += numel(s)
    return tuple(offs), at


def plan_fsdp2(shapes, n_d: int, param_align: int = 1) -> Plan:
    shapes = tuple(tuple(s) for s in shapes)
    offs, extent = _offsets(shapes, param_align)
    total = sum(numel(s) for s in shapes)
    cursor = [0] * n_d                    # next free slot within each rank's shard
    local = []                            # (param, rank, full_off, local_state_off, len, padded)
    for i, shape in enumerate(shapes):
        rows, cols = rows_cols(shape)
        c = shard_rows(rows, n_d)
        for r in range(n_d):
            first_row = min(r * c, rows)
            valid_rows = max(0, min(c, rows - r * c))
            full_off = offs[i] + first_row * cols
            s = cursor[r]
            while s % STATE_ALIGN != full_off % STATE_ALIGN:
                s += 1
            local.append((i, r, full_off, s, valid_rows * cols, c * cols))
            cursor[r] = s + c * cols
    per_rank = max(cursor) if cursor else 0
    per_rank = -(-per_rank // STATE_ALIGN) * STATE_ALIGN
    segs = tuple(Segment(i, r, f, r * per_rank + s, n, p) for (i, r, f, s, n, p) in local)
    return Plan("fsdp2", n_d, shapes, offs, total, extent, per_rank, segs)


def plan_distopt(shapes, n_d: int) -> Plan:
    shapes = tuple(tuple(s) for s in shapes)
    offs, total = _offsets(shapes)
    unit = n_d * DISTOPT_ALIGN // math.gcd(n_d, DISTOPT_ALIGN)     # lcm(N_d, 128)
    padded = -(-total // unit) * unit
    shard = padded // n_d
    segs = tuple(Segment(-1, r, r * shard, r * shard, max(0, min(shard, total - r * shard)), shard)
                 for r in range(n_d))
    return Plan("distopt", n_d, shapes, offs, total, padded, shard, segs)


def plan_hsdp(shapes, n_rep: int, n_shard: int, param_align: int = 1) -> Plan:
    """N_r replica groups of an N_s-rank FSDP2 layout; segment ranks are global."""
    inner = plan_fsdp2(shapes, n_shard, param_align)
    copy = n_shard * inner.state_len_per_rank
    segs = tuple(Segment(s.param, r * n_shard + s.rank, s.full_off, r * copy + s.state_off, s.length, s.padded_len)
                 for r in range(n_rep) for s in inner.segments)
    return Plan("hsdp", n_rep * n_shard, inner.shapes, inner.param_offsets, inner.valid_elems,
                inner.full_len_padded, inner.state_len_per_rank, segs, n_rep)


def plan_layout(shapes, n_d: int, mode: str, n_rep: int = 1, param_align: int = 1) -> Plan:
    """param_align 16: per-parameter buffers (FSDP2 / HSDP only)."""
    if param_align not in (1, 16) or (param_align != 1 and mode == "distopt"):
        raise ValueError("param_align: 1, or 16 for FSDP2 / HSDP")
    if mode == "fsdp2":
        return plan_fsdp2(shapes, n_d, param_align)
    if mode == "distopt":
        return plan_distopt(shapes, n_d)
    if mode == "hsdp":
        if n_rep < 1 or n_d % n_rep:
            raise ValueError("N_d must be a multiple of the replica count")
        return plan_hsdp(shapes, n_rep, n_d // n_rep, param_align)
    raise ValueError(mode)


def owned_indices(plan: Plan):
    """(full index, state index) for every valid element, in segment order
    (HSDP: every replica's copy, so each full index appears N_r times)."""
    import numpy as np
    full, state = [], []
    for s in plan.segments:
        full.append(np.arange(s.full_off, s.full_off + s.length, dtype=np.int64))
        state.append(np.arange(s.state_off, s.state_off + s.length, dtype=np.int64))
    if not full:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(full), np.concatenate(state)
