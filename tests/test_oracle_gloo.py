"""Parallel-vs-single-process equality on CPU with gloo, as the pages check
their mechanisms on 4 CPU processes ("Parallelism strategies: which state to
shard", section 二.2, the 4-process all-reduce = reduce-scatter + all-gather
check).

Four gloo processes run the step with real collectives - FSDP2's copy-in of
each parameter's torch.chunk pieces (padded to the first piece's rows), one
reduce_scatter_tensor, AdamW on the rank's own shard, the bf16 cast, one
all_gather_into_tensor and the copy-out; HSDP as 2 replica groups of 2
(reduce-scatter in the shard group, all-reduce across the replica group,
gather in the shard group); DistOpt's flat equal shards; and the clipped
flow (write-back, the norm from an all-reduce of sums of squares) - and every
rank's results must equal the single-process oracle bit for bit.
The gradients are multiples of 2^-12 small enough that every sum is exact in
any order, so the collectives' own reduction order cannot matter.  This pins
the oracle's stage loops (and its plan's shard geometry) to torch.distributed's
collectives and torch.chunk, implementations that share nothing with it.
"""
import json
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import synth_inputs as S
from oracle import plan as OP
from oracle import step as OS

HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
WORLD = 4
SHAPES = [(7, 5), (13,), (3, 64), (1,), (9, 3), (2, 2, 3)]
SEED, T = 77, 10
CLIP = 1e-3   # below the gradients' norm, so the coefficient is < 1
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exact_grad(q: int, n: int) -> np.ndarray:
    """Rank q's gradient: the generator's N(0, 1e-3) value rounded to a
    multiple of 2^-12 (integers of magnitude < 2^6 times 2^-12)."""
    g = S.grad_f32(SEED, q, np.arange(n)).astype(np.float64)
    return (np.round(g * 4096.0) / 4096.0).astype(np.float32)


def _state_by_index(n: int):
    idx = np.arange(n)
    return S.master_f32(SEED, idx), S.adam_m_f32(SEED, idx), S.adam_v_f32(SEED, idx)


def _all_gather_bits(bits: np.ndarray, world: int, group=None) -> np.ndarray:
    """all_gather_into_tensor of bf16 bit patterns (carried as int32: gloo
    gathers no 16-bit integers)."""
    out = torch.zeros(world * bits.size, dtype=torch.int32)
    dist.all_gather_into_tensor(out, torch.from_numpy(bits.astype(np.int32)), group=group)
    return out.numpy().astype(np.uint16)


def _toy(rank, world):
    g = torch.arange(8, dtype=torch.float32) + 10.0 * rank
    shard = torch.zeros(8 // world)
    dist.reduce_scatter_tensor(shard, g)
    full = torch.zeros(8)
    dist.all_gather_into_tensor(full, 0.5 * shard)
    return {"shard": shard.tolist(), "gathered": full.tolist()}


def _fsdp2(rank, world, n_rep=1, max_norm=None):
    """FSDP2 (n_rep = 1) or HSDP over n_rep replica groups of world // n_rep
    ranks: reduce-scatter inside the rank's shard group, all-reduce of the
    shard across the replica group, all-gather inside the shard group.  With
    max_norm: the averaged shard written back into the rank's own gradient
    buffer, the global norm from an all-reduce (SUM) of the first group's
    fp64 sums of squares, and AdamW on the clipped gradient."""
    n_s = world // n_rep
    groups = [dist.new_group(list(range(r * n_s, (r + 1) * n_s))) for r in range(n_rep)] if n_rep > 1 else [None]
    across = [dist.new_group(list(range(s, world, n_s))) for s in range(n_s)] if n_rep > 1 else None
    shard_group = groups[rank // n_s]
    me = rank % n_s
    plan = OP.plan_layout(SHAPES, world, "hsdp" if n_rep > 1 else "fsdp2", n_rep=n_rep)
    n = plan.full_len_padded
    grad = torch.from_numpy(_exact_grad(rank, n))
    th, m, v = _state_by_index(n)
    offs = plan.param_offsets
    # copy-in: piece r of every parameter, padded to the first piece's rows, rank-major
    pieces, geometry = [], []
    for i, shape in enumerate(SHAPES):
        t = grad[offs[i]:offs[i] + int(np.prod(shape))].view(shape)
        ch = torch.chunk(t, n_s, dim=0)
        rows = ch[0].shape[0]
        cols = t[0].numel()
        geometry.append((rows * cols, [c.numel() for c in ch] + [0] * (n_s - len(ch))))
        pieces.append([c.reshape(-1) for c in ch] + [t.new_zeros(0)] * (n_s - len(ch)))
    block = sum(g[0] for g in geometry)
    send = torch.zeros(n_s * block)
    for r in range(n_s):
        o = r * block
        for i, (padded, _) in enumerate(geometry):
            p = pieces[i][r]
            send[o:o + p.numel()] = p
            o += padded
    recv = torch.zeros(block)
    dist.reduce_scatter_tensor(recv, send, group=shard_group)
    if across is not None:
        dist.all_reduce(recv, group=across[me])
    G = (recv / float(world)).numpy()
    seg = {(s.param, s.rank): s for s in plan.segments}
    coef = np.float32(1.0)
    wrote = grad.numpy().copy()
    if max_norm is not None:
        o, sq = 0, 0.0
        for i, (padded, sizes) in enumerate(geometry):
            k = sizes[me]
            if k:
                s = seg[(i, rank)]
                wrote[s.full_off:s.full_off + k] = G[o:o + k]       # the owner's slice of its own buffer
                if rank < n_s:                                       # each element once: the first group's
                    sq += float(np.dot(G[o:o + k].astype(np.float64), G[o:o + k].astype(np.float64)))
            o += padded
        total = torch.tensor([sq], dtype=torch.float64)
        dist.all_reduce(total)
        norm = float(np.sqrt(total.item()))
        coef = OS.clip_coefficient(norm, max_norm)
        G = (G * coef).astype(np.float32)
    # AdamW on this rank's own segments, state slots from the oracle's plan
    master = np.zeros(plan.state_len_total, np.float32)
    mom = np.zeros_like(master)
    var = np.zeros_like(master)
    cast = np.zeros(block, np.uint16)
    o = 0
    checks = []
    for i, (padded, sizes) in enumerate(geometry):
        k = sizes[me]
        s = seg.get((i, rank))
        checks.append(k == (s.length if s else 0))
        if k:
            f = np.arange(s.full_off, s.full_off + k)
            t1, m1, v1 = OS.adamw(th[f], m[f], v[f], G[o:o + k], HP, T)
            master[s.state_off:s.state_off + k] = t1
            mom[s.state_off:s.state_off + k] = m1
            var[s.state_off:s.state_off + k] = v1
            cast[o:o + k] = OS.bf16_rne(t1)
        o += padded
    # all-gather of the bf16 shards in the shard group, then copy-out into this rank's full buffer
    gathered = _all_gather_bits(cast, n_s, shard_group)
    params = np.zeros(n, np.uint16)
    for r in range(n_s):
        o = r * block
        for i, (padded, sizes) in enumerate(geometry):
            params[offs[i] + sum(sizes[:r]):offs[i] + sum(sizes[:r]) + sizes[r]] = gathered[o:o + sizes[r]]
            o += padded
    out = {"master": master, "m": mom, "v": var, "params": params, "checks": checks}
    if max_norm is not None:
        out.update(norm=norm, coef=float(coef), grad=wrote)
    return out


def _distopt(rank, world):
    plan = OP.plan_layout(SHAPES, world, "distopt")
    n = plan.full_len_padded
    L = n // world
    grad = torch.from_numpy(_exact_grad(rank, n))
    th, m, v = _state_by_index(n)
    recv = torch.zeros(L)
    dist.reduce_scatter_tensor(recv, grad)
    G = (recv / float(world)).numpy()
    lo = rank * L
    t1, m1, v1 = OS.adamw(th[lo:lo + L], m[lo:lo + L], v[lo:lo + L], G, HP, T)
    return {"lo": lo, "master": t1, "m": m1, "v": v1, "params": _all_gather_bits(OS.bf16_rne(t1), world)}


def _rank_main(rank, world, port, out_dir, case):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {"toy": _toy, "fsdp2": _fsdp2, "distopt": _distopt,
               "hsdp": lambda r, w: _fsdp2(r, w, n_rep=2),
               "fsdp2_clip": lambda r, w: _fsdp2(r, w, max_norm=CLIP),
               "hsdp_clip": lambda r, w: _fsdp2(r, w, n_rep=2, max_norm=CLIP)}[case](rank, world)
    finally:
        dist.destroy_process_group()
    np.save(os.path.join(out_dir, f"r{rank}.npy"), np.array([res], dtype=object), allow_pickle=True)


def _run(case, tmp_path):
    mp.start_processes(_rank_main, args=(WORLD, _free_port(), str(tmp_path), case), nprocs=WORLD,
                       start_method="spawn")
    return [np.load(tmp_path / f"r{r}.npy", allow_pickle=True)[0] for r in range(WORLD)]


def _single_process(mode, n_rep=1):
    plan = OP.plan_layout(SHAPES, WORLD, mode, n_rep=n_rep)
    n = plan.full_len_padded
    grads = [_exact_grad(q, n) for q in range(WORLD)]
    fi, si = OP.owned_indices(plan)
    th, m, v = _state_by_index(n)
    state = []
    for a in (th, m, v):
        s = np.zeros(plan.state_len_total, np.float32)
        s[si] = a[fi]
        state.append(s)
    params = [np.zeros(n, np.uint16) for _ in range(WORLD)]
    OS.sharded_step(plan, grads, "f32", *state, params, HP, T)
    return plan, state, params


def test_four_processes_reproduce_the_pages_toy(tmp_path):
    with open(os.path.join(GOLDEN, "zero1_toy.json")) as f:
        g = json.load(f)
    res = _run("toy", tmp_path)
    assert res[0]["shard"] == g["reduce_scatter_rank0"]
    for r in res:
        assert r["gathered"] == g["all_gather_of_half_sum"]
    # and the oracle's own reduce-scatter / all-gather helpers agree
    grads = [np.float32(10 * r) + np.arange(8, dtype=np.float32) for r in range(WORLD)]
    plan = OP.plan_fsdp2([(8,)], WORLD)
    assert OS.rs_update_ag(plan, grads, lambda s: np.float32(0.5) * s)[0].tolist() == res[0]["gathered"]


@pytest.mark.parametrize("mode,n_rep", [("fsdp2", 1), ("hsdp", 2)])
def test_fsdp2_with_real_collectives_equals_the_oracle(tmp_path, mode, n_rep):
    """FSDP2 over 4 ranks, and HSDP as 2 replica groups of 2 (gloo subgroups)."""
    res = _run(mode, tmp_path)
    plan, state, params = _single_process(mode, n_rep)
    for r, out in enumerate(res):
        assert all(out["checks"]), "torch.chunk pieces differ from the plan's segment lengths"
        for s in plan.segments:
            if s.rank != r or not s.length:
                continue
            sl = slice(s.state_off, s.state_off + s.length)
            for name, k in (("master", 0), ("m", 1), ("v", 2)):
                assert np.array_equal(out[name][sl].view(np.uint32), state[k][sl].view(np.uint32)), (name, s)
        assert np.array_equal(out["params"], params[r])
    assert plan.valid_elems == sum(int(np.prod(s)) for s in SHAPES)


def test_distopt_with_real_collectives_equals_the_oracle(tmp_path):
    res = _run("distopt", tmp_path)
    plan, state, params = _single_process("distopt")
    P = plan.valid_elems
    for r, out in enumerate(res):
        lo, k = out["lo"], len(out["master"])
        valid = slice(0, max(0, min(k, P - lo)))      # padding past P is no one's
        for name, i in (("master", 0), ("m", 1), ("v", 2)):
            got = out[name][valid].view(np.uint32)
            assert np.array_equal(got, state[i][lo:lo + got.size].view(np.uint32)), name
        assert np.array_equal(out["params"][:P], params[r][:P])


@pytest.mark.parametrize("mode,n_rep", [("fsdp2", 1), ("hsdp", 2)])
def test_clipped_flow_with_real_collectives_equals_the_oracle(tmp_path, mode, n_rep):
    """The distributed-optimizer flow with clipping: each rank writes the
    averaged shard back into its own buffer, the norm comes from an all-reduce
    of the first group's sums of squares (exact here: the squares of multiples
    of 2^-12 and their sums are exact in fp64), and every rank's results equal
    the single-process oracle bit for bit."""
    res = _run(mode + "_clip", tmp_path)
    plan = OP.plan_layout(SHAPES, WORLD, mode, n_rep=n_rep)
    n = plan.full_len_padded
    grads = [_exact_grad(q, n) for q in range(WORLD)]
    fi, si = OP.owned_indices(plan)
    th, m, v = _state_by_index(n)
    state = []
    for a in (th, m, v):
        s = np.zeros(plan.state_len_total, np.float32)
        s[si] = a[fi]
        state.append(s)
    params = [np.zeros(n, np.uint16) for _ in range(WORLD)]
    norm, coef = OS.sharded_step_clipped(plan, grads, *state, params, HP, T, CLIP)
    assert coef < 1
    for r, out in enumerate(res):
        assert out["norm"] == norm and out["coef"] == float(coef)
        assert np.array_equal(out["grad"].view(np.uint32), grads[r].view(np.uint32))
        for sg in plan.segments:
            if sg.rank != r or not sg.length:
                continue
            sl = slice(sg.state_off, sg.state_off + sg.length)
            for name, k in (("master", 0), ("m", 1), ("v", 2)):
                assert np.array_equal(out[name][sl].view(np.uint32), state[k][sl].view(np.uint32)), (name, sg)
        assert np.array_equal(out["params"], params[r])
