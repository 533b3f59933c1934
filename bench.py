#!/usr/bin/env python
"""Benchmark of the GB300 fused sharded mixed-precision step.

Prints ONE JSON line (rank 0).  A "step" is one pass of the whole hot path -
reduce-scatter of the N_d gradient buffers (rank-ordered fp32 sum / N_d),
AdamW on the fp32 master/m/v shard, bf16 cast and all-gather into the N_d
param buffers - over the workload's synthetic inputs, which are resident in
HBM when the timed region starts.  Default workload: the Qwen3-0.6B-shaped
stack with N_d = 8 in FSDP2 Shard(0) layout (596,049,920 params, 72 B moved
per param).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|IDX]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

Other flows (each reports its own bytes per param): --clip MAX_NORM,
--writeback, --no-gather, --unshard, --fp32-gather, and --per-param (alone or
with any of those); --n-d N and --param-slice a:b change the workload,
--layers K steps K copies of it back to back (one plan per layer; the plain
step, --no-gather or --unshard), --graph
captures the timed steps.  The default run also times the other workloads
after the headline one (the "workloads" list of the JSON line).

Multi-GPU (torchrun, one rank per GPU): the step does not shard across GPUs
(the N_d ranks already live on one device), so every GPU runs an independent
replica; value = all ranks' params / max-over-ranks time ("weak" scaling).
The control plane (barrier, max) uses gloo; the data path has no collective.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sharded-step params/s and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = tuple(os.path.join(ROOT, "fsdp_sharded_mixed_pass_gb300", "csrc", f)
                   for f in ("fsp_args.h", "fsp_kernels.cuh"))
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "sharded_step_kernel_dram_traffic_workloads_1_3_4_5.txt")
# Working sets under this many L2 sizes get an L2 flush before every timed step.
L2_FLUSH_FACTOR = 4
L2_BYTES = 129_000_000      # GB300's L2; the device's own figure is used when a GPU is present
HOLD_CYCLES = 400_000       # ~0.2 ms of GPU spin before each individually timed (L2-flushed) step
BAD_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------------
# run-time context
# --------------------------------------------------------------------------

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("fsp", "reference"), default="fsp")
    ap.add_argument("--workload", default="qwen3_0p6b_fsdp2")
    ap.add_argument("--n-d", type=int, default=None,
                    help="run the workload with this many data-parallel ranks instead of its own N_d")
    ap.add_argument("--param-slice", default=None,
                    help="a:b - only params a..b-1 of the workload (small cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--e2e-chunk", type=int, default=0, help="elements per host-pipeline chunk (0: library default)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--clip", type=float, default=None, metavar="MAX_NORM",
                    help="time the distributed-optimizer flow instead: reduce-scatter written back into the "
                         "owners' grad slices, global norm, clipped AdamW (fp32 grads, FSDP2/DistOpt/HSDP)")
    ap.add_argument("--no-gather", action="store_true",
                    help="time the ZeRO-3 step instead: reduce-scatter + AdamW, parameters left sharded")
    ap.add_argument("--writeback", action="store_true",
                    help="time the step that also writes the averaged gradient into the owners' slices "
                         "(distributed optimizer; fp32 grads, FSDP2 / DistOpt)")
    ap.add_argument("--fp32-gather", action="store_true",
                    help="time the step whose all-gather writes the fp32 master into fp32 param buffers "
                         "(full-size buffers; with --unshard: the fp32 unshard)")
    ap.add_argument("--unshard", action="store_true",
                    help="time the FSDP2 unshard instead (fp32 shards -> bf16 -> every rank's full buffer)")
    ap.add_argument("--per-param", action="store_true",
                    help="every rank's gradient and parameter of every parameter in a tensor of its own "
                         "(FSDP2 / HSDP; the step reads and writes them in place)")
    ap.add_argument("--layers", type=int, default=1,
                    help="K copies of the workload, one plan each, stepped back to back per step (the plain step, "
                         "--no-gather or --unshard)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the block that times the other workloads after the default one")
    ap.add_argument("--workload-steps", type=int, default=20,
                    help="timed steps per workload in the workloads block")
    ap.add_argument("--graph", action="store_true",
                    help="capture the timed steps in one CUDA graph (removes host launch overhead; small cases)")
    return ap.parse_args(argv)


class Dist:
    """gloo control plane for barrier and max-over-ranks (no data-path use)."""

    def __init__(self, n_gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist
        if n_gpus != self.world and self.world > 1:
            log(f"warning: --gpus {n_gpus} but WORLD_SIZE {self.world}")

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def read_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_src_hash(text: str | None = None) -> str:
    """sha256 prefix of the step kernels' code (their argument block and
    device source) with comments and whitespace removed, so that only a
    change of code makes a stored ncu capture stale."""
    import re
    if text is None:
        text = ""
        for path in KERNEL_SRC:
            with open(path, encoding="utf-8") as f:
                text += f.read() + "\n"
    code = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    code = re.sub(r"//[^\n]*", " ", code)
    code = " ".join(code.split())
    return hashlib.sha256(code.encode()).hexdigest()[:12]


def workload_own_n_d(name: str) -> int:
    import synth_inputs as S
    return (S.workload(int(name)) if name.isdigit() else S.workload(name)).n_d


def _traffic_record() -> dict:
    kv = {}
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    return kv


def traffic_per_elem(workload_name: str):
    """ncu DRAM bytes per element of the step kernel, if the committed capture
    was taken on the current kernel source and workload family."""
    try:
        kv = _traffic_record()
        if kv.get("kernel_src") != kernel_src_hash():
            return None
        return float(kv[f"bytes_per_elem.{workload_name}"])
    except Exception:
        return None


def traffic_basis(workload_name: str, elems: int) -> str | None:
    """How the reported traffic was obtained: one captured launch of this size,
    or a smaller one scaled by the elements."""
    try:
        n = int(_traffic_record()[f"elements.{workload_name}"])
    except Exception:
        return None
    what = "ncu dram__bytes_read.sum + dram__bytes_write.sum of one launch"
    if n == elems:
        return f"{what} of this size ({n} elements)"
    return f"{what} of {n} elements, scaled to {elems}"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if device_id:
            cmd += ["-i", device_id]
        try:
            self.p = subprocess.Popen(cmd, stdout=self.tmp, stderr=subprocess.DEVNULL)
        except Exception as e:  # no nvidia-smi
            self.p, self.err = None, str(e)
        self.t0 = self.t1 = None

    def start_window(self):
        time.sleep(1.0)
        self.t0 = datetime.datetime.now()

    def end_window(self):
        self.t1 = datetime.datetime.now()
        time.sleep(0.15)

    def result(self) -> dict:
        if self.p is None:
            return {"error": self.err}
        self.p.terminate()
        try:
            self.p.wait(5)
        except Exception:
            self.p.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = []
        for line in self.tmp.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
            except ValueError:
                continue
            if self.t0 and self.t1 and not (self.t0 <= ts <= self.t1):
                continue
            rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return {"error": "no samples inside the timed region"}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[4]) for r in rows if r[4].replace(".", "").isdigit())
                if any(r[4].replace(".", "").isdigit() for r in rows) else None}


def clocks_bad(c: dict) -> bool:
    if "error" in c:
        return False
    if any(r in BAD_REASONS for r in c.get("reasons", [])):
        return True
    sm, mx = c.get("sm_mhz"), c.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.5 * mx and not c.get("reasons"))


# --------------------------------------------------------------------------
# workload on the device
# --------------------------------------------------------------------------

# (N_s, N_r) meshes the library instantiates its bulk-copy step kernel for;
# other meshes run the per-thread generic kernel.
BULK_MESHES = frozenset([(n, 1) for n in (1, 2, 3, 4, 5, 6, 7, 8, 12, 16)] + [(2, 2), (4, 2), (8, 2), (2, 4), (4, 4)])


def step_kernel_name(w) -> str:
    """The step kernel a workload's mesh runs (the roofline's dominant kernel)."""
    return "sharded_step_kernel" if (w.n_d // w.n_rep, w.n_rep) in BULK_MESHES else "sharded_step_generic_kernel"


def resolve_workload(name: str, param_slice: str | None, n_d: int | None = None):
    """The named workload, optionally on params a..b-1 only and/or with another
    rank count N_d (HSDP keeps its replica groups; N_d must be a multiple)."""
    import dataclasses
    import synth_inputs as S
    w = S.workload(int(name)) if name.isdigit() else S.workload(name)
    label = w.name
    if n_d is not None and n_d != w.n_d:
        if not 1 <= n_d <= 64 or n_d % w.n_rep:
            raise SystemExit(f"--n-d {n_d}: need 1..64 and a multiple of the {w.n_rep} replica groups")
        w = dataclasses.replace(w, n_d=n_d)
        label = f"{w.name}@N_d={n_d}"
    shapes = w.shapes
    if param_slice:
        a, b = (int(x) if x else None for x in param_slice.split(":"))
        shapes = shapes[a:b]
        label = f"{label}[{param_slice}]"
    return w, tuple(shapes), label


class DeviceWorkload:
    def __init__(self, w, shapes, device, per_param: bool = False, fp32_gather: bool = False,
                 no_gather: bool = False):
        import torch
        import fsdp_sharded_mixed_pass_gb300 as fsp
        from synth_inputs import device as D
        self.w, self.device = w, device
        self.per_param = per_param
        gdt = torch.float32 if w.grad_dtype == "f32" else torch.bfloat16
        if per_param:
            # every rank's gradient and bf16 parameter of every parameter as a tensor of its own
            self.plan = fsp.plan_layout_params(shapes, w.n_d, n_replicate=w.n_rep)
            p = self.plan
            sizes = [math.prod(sh) for sh in shapes]
            self.grads = [[torch.empty(n, dtype=gdt, device=device) for n in sizes] for _ in range(w.n_d)]
            for q, row in enumerate(self.grads):
                for g in row:
                    D.fill_grad(g, w.data_seed, q, w.grad_dtype)
            pdt = torch.float32 if fp32_gather else torch.bfloat16
            # ZeRO-3 (no gather): a table of gradients only
            self.params = None if no_gather else [[torch.zeros(n, dtype=pdt, device=device) for n in sizes]
                                                  for _ in range(w.n_d)]
            self.table = fsp.ParamTable(p, self.grads, self.params)
        else:
            self.plan = fsp.plan_layout(shapes, w.n_d, w.mode, n_replicate=w.n_rep)
            p = self.plan
            self.grads = [torch.empty(p.full_len_padded, dtype=gdt, device=device) for _ in range(w.n_d)]
            for q, g in enumerate(self.grads):
                D.fill_grad(g, w.data_seed, q, w.grad_dtype)
            pdt = torch.float32 if fp32_gather else torch.bfloat16
            self.params = [torch.zeros(p.full_len_padded, dtype=pdt, device=device) for _ in range(w.n_d)]
        self.fp32_gather = fp32_gather
        self.state = [torch.zeros(p.state_len_total, dtype=torch.float32, device=device) for _ in range(3)]
        D.fill_state_segments(*self.state, w.data_seed, [(s.full_off, s.state_off, s.length) for s in p.segments])
        torch.cuda.synchronize(device)
        self.t = w.step
        self.clip = None
        self.unshard = False
        self.no_gather = False
        self.writeback = False
        self.norm_out = torch.zeros(4, dtype=torch.float32, device=device)

    def step(self, stream):
        import fsdp_sharded_mixed_pass_gb300 as fsp
        if self.per_param:
            if self.unshard:
                fsp.unshard_params(self.plan, self.table, self.state[0], stream=stream)
            elif self.clip is not None:
                fsp.sharded_step_clipped_params(self.plan, self.table, *self.state, self.w.hparams(), self.t,
                                                self.clip, self.norm_out, stream=stream)
            elif self.writeback:
                fsp.sharded_step_writeback_params(self.plan, self.table, *self.state, self.w.hparams(), self.t,
                                                  stream=stream)
            else:
                fsp.sharded_step_params(self.plan, self.table, *self.state, self.w.hparams(), self.t, stream=stream)
        elif self.unshard:
            fsp.unshard(self.plan, self.state[0], self.params, stream=stream, fp32=self.fp32_gather)
        elif self.fp32_gather:
            fsp.sharded_step_fp32_gather(self.plan, self.grads, *self.state, self.params, self.w.hparams(), self.t,
                                         stream=stream)
        elif self.writeback:
            fsp.sharded_step_writeback(self.plan, self.grads, *self.state, self.params, self.w.hparams(), self.t,
                                       stream=stream)
        elif self.clip is not None:
            fsp.sharded_step_clipped(self.plan, self.grads, *self.state, self.params, self.w.hparams(), self.t,
                                     self.clip, self.norm_out, stream=stream)
        else:
            fsp.sharded_step(self.plan, self.grads, *self.state, None if self.no_gather else self.params,
                             self.w.hparams(), self.t, stream=stream)
        self.t += 1

    def bytes_per_param(self) -> int:
        w = self.w
        pbytes = 4 if self.fp32_gather else 2
        if self.unshard:            # fp32 master in, one bf16 (fp32) per rank of its group out
            return 4 * w.n_rep + pbytes * w.n_d
        if self.no_gather:          # grads in, state in and out, no params
            return w.n_d * w.grad_bytes + 24 * w.n_rep
        if self.writeback:          # the step plus the owner's averaged slice written back
            return w.n_d * w.grad_bytes + w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
        if self.clip is not None:   # pass 1: N_d grads in, one slice out per group; pass 3: 1 grad + state + params
            return w.n_d * w.grad_bytes + w.grad_bytes * w.n_rep + w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
        return w.n_d * w.grad_bytes + 24 * w.n_rep + pbytes * w.n_d


class LayerStack:
    """``layers`` independent copies of a workload, each with its own plan and
    buffers, stepped one after another on one stream: the per-layer steps of a
    model whose layers each have the workload's size (FSDP2 steps one layer's
    shards at a time).  Same interface as DeviceWorkload for the timing."""

    def __init__(self, w, shapes, device, layers: int):
        self.layers = [DeviceWorkload(w, shapes, device) for _ in range(layers)]
        self.w, self.device = w, device
        self.plan = type("P", (), {"valid_elems": layers * self.layers[0].plan.valid_elems})

    def step(self, stream):
        for layer in self.layers:
            layer.step(stream)

    def bytes_per_param(self) -> int:
        return self.layers[0].bytes_per_param()

    def close(self):
        for layer in self.layers:
            layer.plan.close()


def time_device(wl: DeviceWorkload, steps: int, warmup: int, dist: Dist, clocks_id, graph: bool = False,
                flush_bytes: int = 0):
    """Device time of ``steps`` steps on one stream, in ms.

    With ``flush_bytes`` > 0 (working sets that fit in L2) every timed step is
    preceded by an untimed write of ``flush_bytes`` to a scratch buffer and a
    read of it back, so each step starts from a cold L2 that holds no line of
    its own and no dirty line whose write-back the step would pay for, and by
    a short GPU-side spin that keeps the stream busy while the host enqueues
    the step; each step then has its own event pair and the result is the sum
    of the steps' own durations."""
    import torch
    stream = torch.cuda.Stream(device=wl.device)
    for _ in range(warmup):
        wl.step(stream)
    stream.synchronize()
    flush = torch.empty((flush_bytes + 15) // 16 * 16, dtype=torch.uint8, device=wl.device) \
        if flush_bytes > 0 else None
    graphs = []
    if graph:
        # the K timed launches (each with its own update index t) as one graph,
        # or, with flushes between them, one graph per step
        for _ in range(steps if flush is not None else 1):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for _ in range(1 if flush is not None else steps):
                    wl.step(stream)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for g in graphs:
                g.replay()  # warm replay
        stream.synchronize()
    sampler = ClockSampler(clocks_id)
    sampler.start_window()
    n_ev = steps if flush is not None else 1
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
    dist.barrier()
    torch.cuda.synchronize(wl.device)
    with torch.cuda.stream(stream):
        if flush is None:
            starts[0].record(stream)
            if graphs:
                graphs[0].replay()
            else:
                for _ in range(steps):
                    wl.step(stream)
            ends[0].record(stream)
        else:
            for i in range(steps):
                flush.fill_(i & 0xFF)
                flush.view(torch.int32).max()   # read back: only clean lines stay in L2
                # hold the GPU (no memory traffic) while the host enqueues the step,
                # so that the host's launch time is not inside the step's events
                torch.cuda._sleep(HOLD_CYCLES)
                starts[i].record(stream)
                if graphs:
                    graphs[i].replay()
                else:
                    wl.step(stream)
                ends[i].record(stream)
    ends[-1].synchronize()
    torch.cuda.synchronize(wl.device)
    dist.barrier()
    sampler.end_window()
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends))
    return ms, sampler.result()


def time_e2e(wl: DeviceWorkload, steps: int, dist: Dist, chunk_elems: int = 0):
    """The same step through the C ABI's host-buffer entry point: every step
    copies the N_d gradient buffers from pinned host memory to the device and
    the N_d bf16 param buffers back (chunked, H2D / kernel / D2H overlapped),
    all inside the timed region; the fp32 state stays on the device."""
    import torch
    import fsdp_sharded_mixed_pass_gb300 as fsp
    p = wl.plan
    need = sum(g.numel() * g.element_size() for g in wl.grads) + sum(x.numel() * x.element_size() for x in wl.params)
    pinned = True
    try:
        host_g = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in wl.grads]
        host_p = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in wl.params]
    except RuntimeError as e:   # pinned memory exhausted: pageable buffers work too, slower
        log(f"pinning {need / 1e9:.1f} GB of host memory failed ({e}); using pageable buffers")
        host_g = host_p = None
        torch.cuda.empty_cache()
        pinned = False
        host_g = [torch.empty(g.shape, dtype=g.dtype) for g in wl.grads]
        host_p = [torch.empty(x.shape, dtype=x.dtype) for x in wl.params]
    for h, g in zip(host_g, wl.grads):
        h.copy_(g)
    ws = torch.empty(fsp.host_step_workspace_bytes(p, wl.w.grad_dtype, chunk_elems), dtype=torch.uint8,
                     device=wl.device)
    stream = torch.cuda.Stream(device=wl.device)

    def one():
        fsp.sharded_step_host(p, host_g, *wl.state, host_p, wl.w.hparams(), wl.t, ws, chunk_elems=chunk_elems,
                              stream=stream)
        wl.t += 1
        stream.synchronize()

    one()
    dist.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    dt = time.perf_counter() - t0
    dist.barrier()
    h2d = p.valid_elems * wl.w.n_d * wl.w.grad_bytes
    d2h = p.valid_elems * wl.w.n_d * 2
    del host_g, host_p, ws
    return dt, h2d, d2h, pinned


def host_memory_available() -> int:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return 0


# --------------------------------------------------------------------------
# CPU oracle timing
# --------------------------------------------------------------------------

def _sample_pieces(shapes, max_elems):
    """The workload's params in order; a param over ``max_elems`` elements (an
    embedding) is cut into blocks of whole rows of at most ``max_elems``
    elements, each taken as a param of its own - the step treats every element
    alike, so a block of rows stands for the rows of the whole param."""
    for s in shapes:
        n = math.prod(s)
        if n <= max_elems or len(s) < 2:
            yield tuple(s)
            continue
        row = n // s[0]
        per = max(1, max_elems // row)
        for r0 in range(0, s[0], per):
            yield (min(per, s[0] - r0),) + tuple(s[1:])


def _param_runs(shapes, max_elems):
    """The workload's params (oversized ones cut into row blocks) grouped in
    order into consecutive runs of about ``max_elems`` elements each."""
    runs, cur, total = [], [], 0
    for s in _sample_pieces(shapes, max_elems):
        n = math.prod(s)
        if cur and total + n > max_elems:
            runs.append((tuple(cur), total))
            cur, total = [], 0
        cur.append(s)
        total += n
    if cur:
        runs.append((tuple(cur), total))
    return runs or [((), 0)]


def cpu_sample_shapes(shapes, max_elems=16_000_000):
    """A contiguous run of the workload's params of about ``max_elems``
    elements (the first of ``_param_runs``)."""
    return _param_runs(shapes, max_elems)[0]


def cpu_sample_runs(shapes, max_elems, count):
    """``count`` samples for as many host cores: runs of ``_param_runs`` spread
    evenly over the workload (so the samples together cover its mix of
    params), reused from the start when there are fewer runs than cores."""
    runs = _param_runs(shapes, max_elems)
    if len(runs) > count:
        return [runs[k * len(runs) // count][0] for k in range(count)]
    return [runs[k % len(runs)][0] for k in range(count)]


def oracle_inputs(w, shapes, use_device: bool):
    """Host inputs of the sample in the oracle's layout (generated on the device
    by the shared generator when one is present - same bits as the host one)."""
    import numpy as np
    import synth_inputs as S
    from oracle import plan as OP
    op = OP.plan_layout(shapes, w.n_d, w.mode, n_rep=w.n_rep)
    fi, si = OP.owned_indices(op)
    n = op.full_len_padded
    if use_device:
        import torch
        from synth_inputs import device as D
        grads = []
        for q in range(w.n_d):
            t = torch.empty(n, dtype=torch.float32 if w.grad_dtype == "f32" else torch.bfloat16, device="cuda")
            D.fill_grad(t, w.data_seed, q, w.grad_dtype)
            a = t.cpu().numpy() if w.grad_dtype == "f32" else t.view(torch.int16).cpu().numpy().view(np.uint16)
            grads.append(a)
        del t
    else:
        idx = np.arange(n)
        grads = [S.grad_f32(w.data_seed, q, idx) if w.grad_dtype == "f32" else S.grad_bf16_bits(w.data_seed, q, idx)
                 for q in range(w.n_d)]
    state = []
    for fn in (S.master_f32, S.adam_m_f32, S.adam_v_f32):
        a = np.zeros(op.state_len_total, np.float32)
        a[si] = fn(w.data_seed, fi)
        state.append(a)
    params = [np.zeros(n, np.uint16) for _ in range(w.n_d)]
    return op, grads, state, params


# elements of each host core's sample in the all-core oracle timing
CPU_POOL_ELEMS = 4_000_000


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def pool_size(w, elems_per_worker: int) -> int:
    """One oracle process per host core, fewer if their inputs and numpy
    temporaries (about 160 B per element beside the buffers) would take more
    than half of the available host memory."""
    per_worker = elems_per_worker * (w.n_d * (w.grad_bytes + 2) + 12 + 160)
    avail = host_memory_available()
    k = host_cores()
    if avail and per_worker:
        k = min(k, max(1, int(0.5 * avail // per_worker)))
    return k


def _oracle_worker(w, shapes, warmup, steps, seconds, barrier, results):
    """One host core's share of the oracle timing (a spawned process: numpy
    runs elementwise work on the calling thread, so one process is one core).
    It builds its own sample's inputs with the host generator, runs the warm-up
    steps, waits for the others, then times ``steps`` oracle steps, or as many
    as fit in ``seconds`` when ``steps`` is 0."""
    try:
        from oracle import step as OS
        op, grads, state, params = oracle_inputs(w, shapes, use_device=False)
        t = w.step
        for _ in range(warmup):
            OS.sharded_step(op, grads, w.grad_dtype, *state, params, w.hparams(), t)
            t += 1
        barrier.wait(timeout=900)
        reps, t0 = 0, time.perf_counter()
        while (reps < steps) if steps else (time.perf_counter() - t0 < seconds):
            OS.sharded_step(op, grads, w.grad_dtype, *state, params, w.hparams(), t)
            reps += 1
            t += 1
        results.put((op.valid_elems, reps, time.perf_counter() - t0, None))
    except BaseException as e:   # reported to the parent, which raises it
        try:
            barrier.abort()
        except Exception:
            pass
        results.put((0, 0, 0.0, f"{type(e).__name__}: {e}"))


def time_oracle_pool(w, shapes, workers: int, elems_per_worker: int, warmup: int = 0, steps: int = 0,
                     seconds: float = 10.0, limit_s: float = 1200.0):
    """The oracle on ``workers`` host cores at once, one spawned process each
    on its own run of consecutive params (an oversized one as blocks of its
    rows), all timed over the same window.  Returns
    (elements x steps summed over the processes, the longest process's time,
    each process's sample size in elements)."""
    import multiprocessing as mp
    import queue
    samples = cpu_sample_runs(shapes, elems_per_worker, workers)
    ctx = mp.get_context("spawn")   # a fresh interpreter: safe beside this process's CUDA context
    barrier, results = ctx.Barrier(workers), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w, sm, warmup, steps, seconds, barrier, results),
                         daemon=True) for sm in samples]
    for p in procs:
        p.start()
    out, deadline = [], time.monotonic() + limit_s
    try:
        while len(out) < len(procs):
            try:
                out.append(results.get(timeout=5))
            except queue.Empty:
                dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                if dead or time.monotonic() > deadline:
                    barrier.abort()
                    raise RuntimeError(f"oracle pool: exit codes {dead}" if dead else "oracle pool: time limit")
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
    errors = [e for *_, e in out if e]
    if errors:
        raise RuntimeError(f"oracle pool: {errors[0]}")
    return sum(n * r for n, r, _, _ in out), max(s for _, _, s, _ in out), [n for n, *_ in out]


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def time_oracle(w, shapes, seconds: float, use_device: bool, max_reps: int = 1000):
    from oracle import step as OS
    op, grads, state, params = oracle_inputs(w, shapes, use_device)
    t = w.step
    reps, total = 0, 0.0
    while total < seconds and reps < max_reps:
        t0 = time.perf_counter()
        OS.sharded_step(op, grads, w.grad_dtype, *state, params, w.hparams(), t)
        total += time.perf_counter() - t0
        reps += 1
        t += 1
    return op.valid_elems, reps, total


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def config_block(w, label, plan):
    per = w.n_d * w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
    extra = {}
    if w.grad_bytes != 4:
        # the 6 N_d + 24 B/param formula counts 4-byte gradients; with bf16 grads the step moves less
        extra["bytes_per_param_if_fp32_grads"] = 6 * w.n_d + 24 * w.n_rep
    return {
        "workload": label,
        "n_d": w.n_d,
        "mode": w.mode,
        "n_replicate": w.n_rep,
        "grad_dtype": w.grad_dtype,
        "params": plan.valid_elems,
        "bytes_per_param": per,
        **extra,
        "bytes_per_step": per * plan.valid_elems,
        "parallelism": "replicas",
    }


def step_config(w, label, plan, flush_bytes: int) -> dict:
    """The config block of the plain step on a workload: the same dict on both
    arms (the GPU arm adds the flow's own keys for other flows)."""
    per = w.n_d * w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
    return dict(config_block(w, label, plan), bytes_per_param=per, l2=l2_note(per * plan.valid_elems, flush_bytes))


def l2_note(moved: int, flush_bytes: int) -> str:
    if flush_bytes:
        return (f"L2 flushed before every timed step (an untimed {flush_bytes / 1e6:.0f} MB write, "
                f"then a read of it)")
    return f"inputs larger than L2: every step streams the whole {moved / 1e9:.2f} GB working set"


# The workloads the default run also times, after its headline workload (the
# one-layer case, the DistOpt layout, the ragged N_d = 6 case, the bf16-grad
# N_d = 16 stack, the HSDP 2 x 4 mesh), one after another, each freed before
# the next.
EXTRA_WORKLOADS = ("qwen3_layer", "qwen3_0p6b_distopt", "ragged_500", "dense_1p5b_bf16grad", "qwen3_0p6b_hsdp_2x4",
                   ("qwen3_layer", 28), ("qwen3_0p6b_fsdp2", 28, "1:12"))
# (name, K[, a:b]): K copies of the workload (of its params a..b-1) stepped back
# to back (LayerStack) - the one-layer step as it runs in a model of 28 such
# layers, and the 28 decoder layers of the Qwen3-0.6B stack (params 1..11 are
# its first layer) stepped one layer at a time


def workload_entry(wl, label, ms, steps, clocks, flush_bytes, peak, graph_ms_per_step=None) -> dict:
    """One workload's line of the workloads block."""
    P = wl.plan.valid_elems
    per = wl.bytes_per_param()
    t = ms / 1e3 / steps
    gbs = per * P / t / 1e9
    e = {"workload": label, "n_d": wl.w.n_d, "mode": wl.w.mode, "n_replicate": wl.w.n_rep,
         "grad_dtype": wl.w.grad_dtype, "params": P, "bytes_per_param": per, "steps": steps,
         "ms_per_step": ms / steps, "params_per_s": P / t, "hbm_gbs": gbs, "frac_of_measured": gbs / peak,
         "frac_of_nominal_8000": gbs / 8000.0, "kernel": step_kernel_name(wl.w),
         "l2": l2_note(per * P, flush_bytes),
         "clocks": {k: clocks.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "error") if k in clocks}}
    if graph_ms_per_step is not None:
        e["graph_ms_per_step"] = graph_ms_per_step
    return e


def time_workloads(names, steps, warmup, dist, clocks_id, dev, l2, peak, param_slice=None) -> list:
    """Each named workload (optionally params a..b-1 only) built, timed as the
    headline one is, and freed."""
    import torch
    out = []
    for spec in names:
        name, layers, own_slice = (tuple(spec) + (None,))[:3] if isinstance(spec, tuple) else (spec, 1, None)
        w, shapes, label = resolve_workload(name, own_slice or param_slice, None)
        if layers > 1:
            label = f"{label} x{layers} (one plan per layer, stepped back to back)"
        wl = None
        try:
            wl = LayerStack(w, shapes, dev, layers) if layers > 1 else DeviceWorkload(w, shapes, dev)
            flush = 2 * l2 if wl.bytes_per_param() * wl.plan.valid_elems <= L2_FLUSH_FACTOR * l2 else 0
            n_steps = steps
            ms, clocks = time_device(wl, n_steps, warmup, dist, clocks_id, False, flush)
            if "error" in clocks and ms > 0:
                # a timed region shorter than the sampler's period saw no clock sample:
                # time again with enough steps to span ~150 ms (a flushed step takes
                # ~0.3 ms of wall time with its flush)
                n_steps = max(n_steps, 500) if flush else max(n_steps, int(math.ceil(n_steps * 150.0 / ms)))
                ms, clocks = time_device(wl, n_steps, warmup, dist, clocks_id, False, flush)
            if clocks_bad(clocks):
                ms, clocks = time_device(wl, n_steps, warmup, dist, clocks_id, False, flush)
            graph_ms = None
            if flush:   # small enough for launch cost to show: also one CUDA graph per step
                g_ms, _ = time_device(wl, steps, warmup, dist, clocks_id, True, flush)
                graph_ms = g_ms / steps
            entry = workload_entry(wl, label, ms, n_steps, clocks, flush, peak, graph_ms)
            if layers > 1:
                entry["layers"] = layers
                entry["ms_per_layer"] = entry["ms_per_step"] / layers
            out.append(entry)
        except Exception as e:   # one workload failing leaves the others' lines
            out.append({"workload": label, "error": f"{type(e).__name__}: {e}"[:300]})
        finally:   # the next workload may need the memory
            if isinstance(wl, LayerStack):
                wl.close()
            elif wl is not None:
                wl.plan.close()
            del wl
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
    return out


def run_fsp(args):
    import torch
    dist = Dist(args.gpus)
    dev = torch.device("cuda", dist.local_rank)
    torch.cuda.set_device(dev)
    w, shapes, label = resolve_workload(args.workload, args.param_slice, args.n_d)
    if args.per_param and w.mode == "distopt":
        raise SystemExit("--per-param: FSDP2 / HSDP workloads")
    if args.clip is not None and w.grad_dtype != "f32":
        raise SystemExit("--clip: fp32 gradients")
    if args.writeback and (w.grad_dtype != "f32" or w.n_rep != 1):
        raise SystemExit("--writeback: fp32 gradients, FSDP2 or DistOpt")
    if args.fp32_gather and (args.clip is not None or args.no_gather or args.writeback):
        raise SystemExit("--fp32-gather: the plain step or --unshard")
    if args.per_param and args.no_gather and (args.clip is not None or args.writeback or args.unshard):
        raise SystemExit("--per-param --no-gather: the plain step only (the table has no parameter tensors)")
    if args.layers > 1 and (args.clip is not None or args.per_param or args.writeback or args.fp32_gather):
        raise SystemExit("--layers: the plain step, --no-gather or --unshard")
    if args.layers > 1:
        wl = LayerStack(w, shapes, dev, args.layers)
        label = f"{label} x{args.layers} (one plan per layer, stepped back to back)"
    else:
        wl = DeviceWorkload(w, shapes, dev, per_param=args.per_param, fp32_gather=args.fp32_gather,
                            no_gather=args.no_gather and args.per_param)
    for target in wl.layers if isinstance(wl, LayerStack) else [wl]:
        target.clip = args.clip
        target.unshard = args.unshard
        target.no_gather = args.no_gather
        target.writeback = args.writeback
    plan = wl.plan
    props = torch.cuda.get_device_properties(dev)
    clocks_id = ("GPU-" + str(props.uuid)) if getattr(props, "uuid", None) else None

    l2 = int(getattr(props, "L2_cache_size", 0) or L2_BYTES)
    flush_bytes = 2 * l2 if wl.bytes_per_param() * plan.valid_elems <= L2_FLUSH_FACTOR * l2 else 0
    ms, clocks = time_device(wl, args.steps, args.warmup, dist, clocks_id, args.graph, flush_bytes)
    remeasured = False
    if clocks_bad(clocks):
        log(f"clocks rejected ({clocks}); measuring again")
        ms, clocks = time_device(wl, args.steps, args.warmup, dist, clocks_id, args.graph, flush_bytes)
        remeasured = True
    ms_max = dist.max(ms)
    P = plan.valid_elems
    total_params = P * args.steps * dist.world
    value = total_params / (ms_max / 1e3)
    per = wl.bytes_per_param()
    launch_s = ms / 1e3 / args.steps
    achieved = per * P / launch_s / 1e9
    peak, peak_src = read_peak()
    # per-element traffic was captured at each workload's own N_d
    tpe = traffic_per_elem(w.name) if args.n_d in (None, workload_own_n_d(args.workload)) else None

    e2e = None
    if (not args.no_e2e and args.clip is None and not args.unshard and not args.no_gather and not args.per_param
            and not args.writeback and not args.fp32_gather and args.layers == 1):
        # every rank on this node needs its own host copy of the grads and params
        per_rank = P * w.n_d * (w.grad_bytes + 2)
        local = int(os.environ.get("LOCAL_WORLD_SIZE", dist.world))
        avail = host_memory_available()
        too_big = bool(avail) and per_rank * local > 0.8 * avail
        if dist.max(1.0 if too_big else 0.0) > 0:   # every rank takes the same branch
            e2e = {"error": f"host memory: {local} ranks x {per_rank / 1e9:.1f} GB of host buffers "
                            f"exceed 80% of the {avail / 1e9:.0f} GB available"}
        else:
            dt, h2d, d2h, pinned = time_e2e(wl, args.e2e_steps, dist, args.e2e_chunk)
            dt = dist.max(dt)
            kind = "pinned" if pinned else "pageable"
            e2e = {"value": P * args.e2e_steps * dist.world / dt, "unit": UNIT,
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                   "api": f"fsp_sharded_step_host (C ABI): {kind} host grads in, {kind} host bf16 params out, "
                          "chunked H2D / kernel / D2H pipeline"}

    default_run = (args.clip is None and not args.unshard and not args.no_gather and not args.per_param
                   and not args.writeback and not args.fp32_gather and not args.graph and args.param_slice is None
                   and args.n_d is None and args.layers == 1)
    workloads = None
    if default_run and dist.world == 1 and not args.no_workloads:
        headline = workload_entry(wl, label, ms, args.steps, clocks, flush_bytes, peak)
        wl.plan.close()
        del wl
        torch.cuda.empty_cache()
        names = [n for n in EXTRA_WORKLOADS if n != w.name]   # the headline's own stack entry stays
        workloads = [headline] + time_workloads(names, args.workload_steps, max(3, min(args.warmup, 5)), dist,
                                                clocks_id, dev, l2, peak)

    cpu = None
    if dist.world == 1 and not args.no_cpu_baseline:
        sshapes, _ = cpu_sample_shapes(shapes)
        n, reps, secs = time_oracle(w, sshapes, args.cpu_seconds, use_device=True)
        one = {"value": n * reps / secs,
               "sample": f"{len(sshapes)} params ({n} elements) of {w.name}, N_d={w.n_d}, "
                         f"oracle step repeated {reps}x ({secs:.1f} s)"}
        cpu = {"value": one["value"], "unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
               "host_cores": host_cores(), "sample": one["sample"], "value_1_core": one["value"]}
        k = pool_size(w, CPU_POOL_ELEMS)
        if k > 1:
            try:
                done, psecs, sizes = time_oracle_pool(w, shapes, k, CPU_POOL_ELEMS, seconds=args.cpu_seconds)
                cpu.update(value=done / psecs, cores=k,
                           sample=f"{k} processes, one per host core, each repeating the oracle step on its own "
                                  f"run of consecutive params of {w.name}, spread over the workload, params "
                                  f"larger than a run as blocks of rows ({min(sizes)}-{max(sizes)} elements), "
                                  f"N_d={w.n_d}, for {psecs:.1f} s",
                           sample_1_core=one["sample"])
            except Exception as e:
                cpu["pool_error"] = str(e)[:300]
        for e in workloads or []:
            if e.get("workload") == "qwen3_layer" and "error" not in e:
                # the one-layer workload's oracle step on one core too (its whole plan)
                import synth_inputs as S
                w0 = S.workload("qwen3_layer")
                n0, r0, s0 = time_oracle(w0, w0.shapes, min(args.cpu_seconds, 3.0), use_device=True)
                e["cpu_oracle_1_core"] = {"value": n0 * r0 / s0, "unit": UNIT, "cores": 1, "kind": "oracle",
                                          "sample": f"the whole plan ({n0} elements), oracle step repeated "
                                                    f"{r0}x ({s0:.1f} s)"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(step_config(w, label, plan, flush_bytes), bytes_per_param=per,
                       l2=l2_note(per * P, flush_bytes), **(
            {"flow": f"distributed optimizer with clipping, max_norm {args.clip} (4 kernels per step)"}
            if args.clip is not None else {"flow": "FSDP2 unshard (bf16 all-gather of the fp32 shards)"}
            if args.unshard else {"flow": "ZeRO-3 step: reduce-scatter + AdamW, no all-gather"}
            if args.no_gather else {"flow": "distributed-optimizer step with the averaged gradient written back "
                                            "into the owners' grad slices (one kernel)"}
            if args.writeback else {}),
                       **({"param_dtype": "fp32 (all-gather of the fp32 master)"} if args.fp32_gather else {}),
                       **({"buffers": "per-parameter tensors (each rank's gradient and bf16 parameter of each "
                                      "parameter in a tensor of its own)"} if args.per_param else {})),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "frac_of_nominal_8000": achieved / 8000.0, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "traffic": tpe * P if tpe is not None and args.clip is None and not args.unshard
                     and not args.no_gather and not args.per_param and not args.writeback and not args.fp32_gather
                     else None,
                     "traffic_basis": traffic_basis(w.name, P) if tpe is not None and args.clip is None
                     and not args.unshard and not args.no_gather and not args.per_param and not args.writeback
                     and not args.fp32_gather else None,
                     "kernel": "unshard_kernel" if args.unshard else step_kernel_name(w),
                     "kernel_src": kernel_src_hash()},
        "e2e": e2e,
        "cpu_baseline": cpu,
        **({"workloads": workloads} if workloads is not None else {}),
        "gpu_launches": args.steps * args.layers * (4 if args.clip is not None else 1),
        "launch": "one CUDA graph of the K steps" if args.graph else "one launch per step from the host",
        "clocks": clocks,
    }
    if remeasured:
        line["clocks_remeasured"] = True
    if dist.rank == 0:
        print(json.dumps(line), flush=True)
    dist.close()


def run_reference(args):
    dist_rank = int(os.environ.get("RANK", "0"))
    if dist_rank != 0:
        return
    w, shapes, label = resolve_workload(args.workload, args.param_slice, args.n_d)
    # per step and core, a bounded sample sized so the whole run stays within ~2 minutes
    budget_elems = max(100_000, min(16_000_000, int(120 * 15e6 / max(1, args.steps + args.warmup))))
    per_core = min(budget_elems, CPU_POOL_ELEMS)
    k = pool_size(w, per_core)
    pool_error = None
    if k > 1:
        try:
            done, secs, sizes = time_oracle_pool(w, shapes, k, per_core, warmup=args.warmup, steps=args.steps)
            value, sample_elems = done / secs, sum(sizes)
            sample = (f"{k} processes, one per host core, each stepping the oracle on its own run of consecutive "
                      f"params of {w.name}, spread over the workload, params larger than a run as blocks of "
                      f"rows ({min(sizes)}-{max(sizes)} elements) per step, N_d={w.n_d}")
        except Exception as e:
            pool_error, k = str(e)[:300], 1
    if k == 1:
        sshapes, _ = cpu_sample_shapes(shapes, budget_elems)
        use_device = False
        try:
            import torch
            use_device = torch.cuda.is_available()
            if use_device:
                from synth_inputs import device as D
                D.lib()
        except Exception:
            use_device = False
        from oracle import step as OS
        op, grads, state, params = oracle_inputs(w, sshapes, use_device)
        t = w.step
        for _ in range(args.warmup):
            OS.sharded_step(op, grads, w.grad_dtype, *state, params, w.hparams(), t)
            t += 1
        t0 = time.perf_counter()
        for _ in range(args.steps):
            OS.sharded_step(op, grads, w.grad_dtype, *state, params, w.hparams(), t)
            t += 1
        secs = time.perf_counter() - t0
        value, sample_elems = op.valid_elems * args.steps / secs, op.valid_elems
        sample = f"{len(sshapes)} params ({op.valid_elems} elements) of {w.name} per step, N_d={w.n_d}"
    # the config of the workload itself, as the GPU arm reports it; what was
    # timed (a bounded sample of that workload per step) beside it
    full_p = sum(math.prod(sh) for sh in shapes)
    plan_like = type("P", (), {"valid_elems": full_p})
    per = w.n_d * w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
    l2 = L2_BYTES
    try:   # the GPU arm's flush decision uses the device's own L2 size
        import torch
        if torch.cuda.is_available():
            l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or L2_BYTES)
    except Exception:
        pass
    flush_bytes = 2 * l2 if per * full_p <= L2_FLUSH_FACTOR * l2 else 0
    cfg = step_config(w, label, plan_like, flush_bytes)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": full_p / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        # the step is elementwise: ms_per_step is the whole workload's step at the sample's measured rate
        "sample": {"params_per_step": sample_elems, "ms_per_step": secs * 1e3 / args.steps,
                   "ms_per_step_basis": f"the full workload ({full_p} params) at the measured rate of the "
                                        f"{sample_elems}-element sample"},
        "cpu_baseline": dict({"value": value, "unit": UNIT, "cores": k, "kind": "oracle",
                              "cpu": cpu_model(), "host_cores": host_cores(), "sample": sample},
                             **({"pool_error": pool_error} if pool_error else {})),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_fsp(args)


if __name__ == "__main__":
    main()
