"""ctypes binding of libfsp.so (``include/fsp.h``): argument marshalling only.

Every step of the sharded update runs in the library's CUDA kernel; nothing
here computes any of it, and there is no fallback: if the library is missing
the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libfsp.so")

FSP_OK, FSP_EINVAL, FSP_ENOMEM, FSP_ECUDA, FSP_EUNSUPPORTED = range(5)
MODES = {"fsdp2": 0, "distopt": 1, "hsdp": 2}
DTYPES = {"f32": 0, "bf16": 1}

# Every symbol include/fsp.h declares.
EXPORTS = ("fsp_plan_layout", "fsp_plan_layout_hsdp", "fsp_plan_layout_params", "fsp_plan_param", "fsp_plan_info_get",
           "fsp_plan_segment", "fsp_plan_ledger", "fsp_plan_tiles", "fsp_plan_round_order", "fsp_plan_destroy",
           "fsp_sharded_step", "fsp_sharded_step_device_t", "fsp_sharded_step_clipped", "fsp_sharded_step_debug",
           "fsp_sharded_step_writeback", "fsp_sharded_step_fp32_gather", "fsp_unshard_fp32", "fsp_shard",
           "fsp_host_step_workspace_bytes", "fsp_sharded_step_host", "fsp_param_table_create", "fsp_param_table_destroy",
           "fsp_sharded_step_params", "fsp_sharded_step_params_device_t", "fsp_sharded_step_clipped_params",
           "fsp_sharded_step_writeback_params",
           "fsp_unshard_params",
           "fsp_sharded_step_noalloc", "fsp_unshard", "fsp_device_error", "fsp_selftest_bounded_wait", "fsp_status_string",
           "fsp_last_error")


class FspError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class _PlanInfo(ctypes.Structure):
    _fields_ = [("n_d", ctypes.c_int32), ("n_params", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("tile_elems", ctypes.c_int32), ("valid_elems", ctypes.c_int64),
                ("full_len_padded", ctypes.c_int64), ("state_len_per_rank", ctypes.c_int64),
                ("state_len_total", ctypes.c_int64), ("n_segments", ctypes.c_int64), ("n_tiles", ctypes.c_int64),
                ("n_replicate", ctypes.c_int32), ("n_shard", ctypes.c_int32), ("param_align", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class _Tile(ctypes.Structure):
    _fields_ = [("full_begin", ctypes.c_int64), ("state_begin", ctypes.c_int64), ("len", ctypes.c_int32),
                ("rank", ctypes.c_int32), ("param", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class _Segment(ctypes.Structure):
    _fields_ = [("param", ctypes.c_int32), ("rank", ctypes.c_int32), ("full_off", ctypes.c_int64),
                ("state_off", ctypes.c_int64), ("len", ctypes.c_int64), ("padded_len", ctypes.c_int64)]


class _Ledger(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("resident_ddp", "resident_distopt", "resident_zero2",
                                               "resident_fsdp", "reduce_scatter_sent", "all_gather_sent",
                                               "step_hbm_bytes", "resident_hsdp", "cross_group_all_reduce_sent")]


class _HParams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "beta1", "beta2", "eps", "weight_decay")]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with fsdp_sharded_mixed_pass_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.fsp_plan_layout.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32), i32, i32, i32,
                                  ctypes.POINTER(vp)]
    L.fsp_plan_layout_hsdp.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32), i32, i32,
                                       i32, ctypes.POINTER(vp)]
    L.fsp_plan_layout_params.argtypes = [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32), i32, i32,
                                         i32, ctypes.POINTER(vp)]
    L.fsp_plan_param.argtypes = [vp, i32, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64)]
    L.fsp_param_table_create.argtypes = [vp, ctypes.POINTER(vp), i32, ctypes.POINTER(vp), i32, ctypes.POINTER(vp)]
    L.fsp_param_table_destroy.argtypes = [vp]
    L.fsp_param_table_destroy.restype = None
    L.fsp_sharded_step_params.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(_HParams), i64, vp]
    L.fsp_unshard_params.argtypes = [vp, vp, vp, vp]
    L.fsp_sharded_step_params_device_t.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(_HParams), vp, i32, vp]
    L.fsp_sharded_step_writeback_params.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(_HParams), i64, vp]
    L.fsp_sharded_step_clipped_params.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(_HParams), i64, ctypes.c_float,
                                                  vp, vp]
    L.fsp_plan_info_get.argtypes = [vp, ctypes.POINTER(_PlanInfo)]
    L.fsp_plan_segment.argtypes = [vp, i64, ctypes.POINTER(_Segment)]
    L.fsp_plan_ledger.argtypes = [vp, i32, ctypes.POINTER(_Ledger)]
    L.fsp_plan_tiles.argtypes = [vp, i32, ctypes.POINTER(_Tile), ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
    L.fsp_plan_round_order.argtypes = [vp, i32, ctypes.POINTER(_Tile), ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
    L.fsp_plan_destroy.argtypes = [vp]
    L.fsp_plan_destroy.restype = None
    step_args = [vp, ctypes.POINTER(vp), i32, vp, vp, vp, ctypes.POINTER(vp), ctypes.POINTER(_HParams), i64]
    L.fsp_sharded_step.argtypes = step_args + [vp]
    L.fsp_sharded_step_debug.argtypes = step_args + [vp, vp]
    L.fsp_sharded_step_noalloc.argtypes = step_args + [vp]
    L.fsp_sharded_step_writeback.argtypes = step_args + [vp]
    L.fsp_sharded_step_fp32_gather.argtypes = step_args + [vp]
    L.fsp_unshard_fp32.argtypes = [vp, vp, ctypes.POINTER(vp), vp]
    L.fsp_shard.argtypes = [vp, vp, vp, vp, vp, vp]
    L.fsp_sharded_step_clipped.argtypes = step_args + [ctypes.c_float, vp, vp]
    L.fsp_sharded_step_clipped.restype = ctypes.c_int
    L.fsp_sharded_step_device_t.argtypes = step_args[:-1] + [vp, i32, vp]
    L.fsp_sharded_step_device_t.restype = ctypes.c_int
    L.fsp_unshard.argtypes = [vp, vp, ctypes.POINTER(vp), vp]
    L.fsp_unshard.restype = ctypes.c_int
    for fn in ("fsp_plan_layout", "fsp_plan_layout_hsdp", "fsp_plan_layout_params", "fsp_plan_param",
               "fsp_plan_info_get", "fsp_plan_segment", "fsp_plan_ledger", "fsp_sharded_step", "fsp_sharded_step_debug",
               "fsp_sharded_step_noalloc", "fsp_sharded_step_writeback", "fsp_sharded_step_fp32_gather",
               "fsp_unshard_fp32", "fsp_shard", "fsp_param_table_create", "fsp_sharded_step_params",
               "fsp_sharded_step_clipped_params", "fsp_sharded_step_params_device_t", "fsp_unshard_params",
               "fsp_sharded_step_writeback_params"):
        getattr(L, fn).restype = ctypes.c_int
    L.fsp_host_step_workspace_bytes.argtypes = [vp, i32, i64, ctypes.POINTER(ctypes.c_size_t)]
    L.fsp_host_step_workspace_bytes.restype = ctypes.c_int
    L.fsp_sharded_step_host.argtypes = step_args + [vp, ctypes.c_size_t, i64, vp]
    L.fsp_sharded_step_host.restype = ctypes.c_int
    L.fsp_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.fsp_device_error.restype = ctypes.c_int
    L.fsp_selftest_bounded_wait.argtypes = [ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]
    L.fsp_selftest_bounded_wait.restype = ctypes.c_int
    L.fsp_status_string.argtypes = [ctypes.c_int]
    L.fsp_status_string.restype = ctypes.c_char_p
    L.fsp_last_error.argtypes = []
    L.fsp_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def _check(status: int, what: str):
    if status != FSP_OK:
        L = lib()
        raise FspError(status, f"{what}: {L.fsp_status_string(status).decode()}: {L.fsp_last_error().decode()}")


@dataclass(frozen=True)
class Segment:
    param: int
    rank: int
    full_off: int
    state_off: int
    length: int
    padded_len: int


class Plan:
    """A layout plan (owns the library handle)."""

    def __init__(self, handle: int, shapes, mode: str):
        self._h = ctypes.c_void_p(handle)
        self.shapes = tuple(tuple(int(d) for d in s) for s in shapes)
        self.mode = mode
        info = _PlanInfo()
        _check(lib().fsp_plan_info_get(self._h, ctypes.byref(info)), "fsp_plan_info_get")
        self.n_d = info.n_d
        self.n_params = info.n_params
        self.tile_elems = info.tile_elems
        self.valid_elems = info.valid_elems
        self.full_len_padded = info.full_len_padded
        self.state_len_per_rank = info.state_len_per_rank
        self.state_len_total = info.state_len_total
        self.n_segments = info.n_segments
        self.n_tiles = info.n_tiles
        self.n_replicate = info.n_replicate
        self.n_shard = info.n_shard
        self.param_align = info.param_align
        self._segments = None
        self._param_offsets = None

    @property
    def handle(self):
        return self._h

    @property
    def segments(self) -> tuple:
        if self._segments is None:
            out, seg = [], _Segment()
            for i in range(self.n_segments):
                _check(lib().fsp_plan_segment(self._h, i, ctypes.byref(seg)), "fsp_plan_segment")
                out.append(Segment(seg.param, seg.rank, seg.full_off, seg.state_off, seg.len, seg.padded_len))
            self._segments = tuple(out)
        return self._segments

    @property
    def param_offsets(self) -> tuple:
        """Each parameter's first full index (virtual for per-parameter plans)."""
        if self._param_offsets is None:
            off, n = ctypes.c_int64(), ctypes.c_int64()
            out = []
            for i in range(self.n_params):
                _check(lib().fsp_plan_param(self._h, i, ctypes.byref(off), ctypes.byref(n)), "fsp_plan_param")
                out.append(off.value)
            self._param_offsets = tuple(out)
        return self._param_offsets

    def tiles(self, unit: int = 0) -> list:
        """The work tiles as (full_begin, state_begin, len, rank, param) tuples:
        the plan's own (unit 0) or split at multiples of ``unit`` elements (the
        step kernels run full-size buffers on unit 2048; see ``fsp_plan_tiles``)."""
        n = ctypes.c_int64()
        _check(lib().fsp_plan_tiles(self._h, int(unit), None, 0, ctypes.byref(n)), "fsp_plan_tiles")
        buf = (_Tile * max(1, n.value))()
        _check(lib().fsp_plan_tiles(self._h, int(unit), buf, n.value, ctypes.byref(n)), "fsp_plan_tiles")
        return [(t.full_begin, t.state_begin, t.len, t.rank, t.param) for t in buf[:n.value]]

    def round_order(self, grid: int) -> list:
        """The tiles in the order a bulk step launch of ``grid`` CTAs strides
        over them (CTA b takes entries b, b + grid, ...), as ``tiles`` tuples;
        see ``fsp_plan_round_order``."""
        n = ctypes.c_int64()
        _check(lib().fsp_plan_round_order(self._h, int(grid), None, 0, ctypes.byref(n)), "fsp_plan_round_order")
        buf = (_Tile * max(1, n.value))()
        _check(lib().fsp_plan_round_order(self._h, int(grid), buf, n.value, ctypes.byref(n)), "fsp_plan_round_order")
        return [(t.full_begin, t.state_begin, t.len, t.rank, t.param) for t in buf[:n.value]]

    def ledger(self, grad_dtype: str = "f32") -> dict:
        led = _Ledger()
        _check(lib().fsp_plan_ledger(self._h, DTYPES[grad_dtype], ctypes.byref(led)), "fsp_plan_ledger")
        return {n: getattr(led, n) for n, _ in _Ledger._fields_}

    def close(self):
        if self._h is not None and self._h.value:
            lib().fsp_plan_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def plan_layout(shapes, n_d: int, mode: str = "fsdp2", n_replicate: int = 1) -> Plan:
    """FSDP2 Shard(0) (``mode="fsdp2"``), DistOpt flat (``"distopt"``) or HSDP
    (``"hsdp"``: ``n_replicate`` groups of ``n_d // n_replicate`` shard ranks)."""
    shapes = [tuple(int(d) for d in s) for s in shapes]
    dims = [d for s in shapes for d in s]
    nd = [len(s) for s in shapes]
    dims_arr = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    nd_arr = (ctypes.c_int32 * max(1, len(nd)))(*nd)
    out = ctypes.c_void_p()
    if mode not in MODES:
        raise ValueError(f"unknown mode {mode!r}")
    if mode == "hsdp":
        if n_replicate < 1 or n_d % n_replicate:
            raise ValueError("n_d must be a multiple of n_replicate")
        _check(lib().fsp_plan_layout_hsdp(dims_arr, nd_arr, len(shapes), int(n_replicate), int(n_d // n_replicate),
                                          ctypes.byref(out)), "fsp_plan_layout_hsdp")
    else:
        _check(lib().fsp_plan_layout(dims_arr, nd_arr, len(shapes), int(n_d), MODES[mode], ctypes.byref(out)),
               "fsp_plan_layout")
    return Plan(out.value, shapes, mode)


def plan_layout_params(shapes, n_d: int, n_replicate: int = 1) -> Plan:
    """Per-parameter plan (``fsp_plan_layout_params``): FSDP2 over ``n_d``
    ranks, or HSDP with ``n_replicate`` groups of ``n_d // n_replicate``; the
    step then reads and writes each rank's per-parameter tensors in place."""
    shapes = [tuple(int(d) for d in s) for s in shapes]
    dims = [d for s in shapes for d in s]
    nd = [len(s) for s in shapes]
    dims_arr = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    nd_arr = (ctypes.c_int32 * max(1, len(nd)))(*nd)
    if n_replicate < 1 or n_d % n_replicate:
        raise ValueError("n_d must be a multiple of n_replicate")
    out = ctypes.c_void_p()
    _check(lib().fsp_plan_layout_params(dims_arr, nd_arr, len(shapes), int(n_replicate), int(n_d // n_replicate),
                                        ctypes.byref(out)), "fsp_plan_layout_params")
    return Plan(out.value, shapes, "fsdp2" if n_replicate == 1 else "hsdp")


class ParamTable:
    """Per-parameter tensors registered for a per-parameter plan
    (``fsp_param_table_create``): ``grads[q][i]`` is rank q's gradient of
    parameter i, ``params[q][i]`` its parameter tensor, bf16 or fp32 (or
    ``params=None``).  Keeps references to the tensors so they outlive the table."""

    def __init__(self, plan: Plan, grads, params=None, grad_dtype: str | None = None,
                 param_dtype: str | None = None):
        if len(grads) != plan.n_d or any(len(g) != plan.n_params for g in grads):
            raise ValueError(f"need {plan.n_d} x {plan.n_params} gradient tensors")
        if params is not None and (len(params) != plan.n_d or any(len(x) != plan.n_params for x in params)):
            raise ValueError(f"need {plan.n_d} x {plan.n_params} param tensors")
        gd = grad_dtype or (_grad_dtype([grads[0][0]], None) if plan.n_params else "f32")
        self.plan, self.grad_dtype = plan, gd
        self._refs = (grads, params)
        n = plan.n_d * plan.n_params
        g = (ctypes.c_void_p * max(1, n))(*[_ptr(x) for row in grads for x in row])
        p = None if params is None else (ctypes.c_void_p * max(1, n))(*[_ptr(x) for row in params for x in row])
        out = ctypes.c_void_p()
        if param_dtype is None:
            import torch
            first = next((x for row in (params or []) for x in row), None)
            param_dtype = "f32" if first is not None and getattr(first, "dtype", None) == torch.float32 else "bf16"
        self.param_dtype = param_dtype
        _check(lib().fsp_param_table_create(plan.handle, g, DTYPES[gd], p, DTYPES[param_dtype], ctypes.byref(out)),
               "fsp_param_table_create")
        self._h = out

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h is not None and self._h.value:
            lib().fsp_param_table_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def sharded_step_params(plan: Plan, table: ParamTable, master, exp_avg, exp_avg_sq, hparams: dict, step: int,
                        stream=None) -> None:
    """The fused step on the per-parameter tensors of ``table`` (asynchronous)."""
    _check(lib().fsp_sharded_step_params(plan.handle, table.handle, ctypes.c_void_p(_ptr(master)),
                                         ctypes.c_void_p(_ptr(exp_avg)), ctypes.c_void_p(_ptr(exp_avg_sq)),
                                         ctypes.byref(_hp(hparams)), int(step),
                                         ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_params")


def sharded_step_params_device_t(plan: Plan, table: ParamTable, master, exp_avg, exp_avg_sq, hparams: dict,
                                 step_dev, advance: bool = True, stream=None) -> None:
    """``sharded_step_params`` with t read from (and advanced in) device memory."""
    _check(lib().fsp_sharded_step_params_device_t(plan.handle, table.handle, ctypes.c_void_p(_ptr(master)),
                                                  ctypes.c_void_p(_ptr(exp_avg)), ctypes.c_void_p(_ptr(exp_avg_sq)),
                                                  ctypes.byref(_hp(hparams)), ctypes.c_void_p(_ptr(step_dev)),
                                                  1 if advance else 0, ctypes.c_void_p(_stream_handle(stream))),
           "fsp_sharded_step_params_device_t")


def sharded_step_writeback_params(plan: Plan, table: ParamTable, master, exp_avg, exp_avg_sq, hparams: dict,
                                  step: int, stream=None) -> None:
    """``sharded_step_writeback`` on the per-parameter tensors of ``table``."""
    _check(lib().fsp_sharded_step_writeback_params(plan.handle, table.handle, ctypes.c_void_p(_ptr(master)),
                                                   ctypes.c_void_p(_ptr(exp_avg)), ctypes.c_void_p(_ptr(exp_avg_sq)),
                                                   ctypes.byref(_hp(hparams)), int(step),
                                                   ctypes.c_void_p(_stream_handle(stream))),
           "fsp_sharded_step_writeback_params")


def sharded_step_clipped_params(plan: Plan, table: ParamTable, master, exp_avg, exp_avg_sq, hparams: dict,
                                step: int, max_norm: float, norm_out, stream=None) -> None:
    """``sharded_step_clipped`` on the per-parameter tensors of ``table``."""
    _check(lib().fsp_sharded_step_clipped_params(plan.handle, table.handle, ctypes.c_void_p(_ptr(master)),
                                                 ctypes.c_void_p(_ptr(exp_avg)), ctypes.c_void_p(_ptr(exp_avg_sq)),
                                                 ctypes.byref(_hp(hparams)), int(step), float(max_norm),
                                                 ctypes.c_void_p(_ptr(norm_out)),
                                                 ctypes.c_void_p(_stream_handle(stream))),
           "fsp_sharded_step_clipped_params")


def unshard_params(plan: Plan, table: ParamTable, master, stream=None) -> None:
    """FSDP2 unshard into the per-parameter bf16 tensors of ``table``."""
    _check(lib().fsp_unshard_params(plan.handle, table.handle, ctypes.c_void_p(_ptr(master)),
                                    ctypes.c_void_p(_stream_handle(stream))), "fsp_unshard_params")


def _ptr(x) -> int:
    return int(x) if isinstance(x, int) else int(x.data_ptr())


def _grad_dtype(grad_bufs, grad_dtype):
    if grad_dtype is not None:
        return grad_dtype
    import torch
    dt = grad_bufs[0].dtype
    if dt == torch.float32:
        return "f32"
    if dt == torch.bfloat16:
        return "bf16"
    raise TypeError(f"unsupported gradient dtype {dt}")


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _hp(hparams) -> _HParams:
    h = _HParams()
    for k in ("lr", "beta1", "beta2", "eps", "weight_decay"):
        setattr(h, k, float(hparams[k]))
    return h


def _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype):
    if len(grad_bufs) != plan.n_d or (param_bufs is not None and len(param_bufs) != plan.n_d):
        raise ValueError(f"need {plan.n_d} grad and param buffers")
    gd = _grad_dtype(grad_bufs, grad_dtype)
    g = (ctypes.c_void_p * plan.n_d)(*[_ptr(b) for b in grad_bufs])
    # param_bufs None: no all-gather (ZeRO-3 / FSDP2 reshard; gather later with unshard)
    p = None if param_bufs is None else (ctypes.c_void_p * plan.n_d)(*[_ptr(b) for b in param_bufs])
    return [plan.handle, g, DTYPES[gd], ctypes.c_void_p(_ptr(master)), ctypes.c_void_p(_ptr(exp_avg)),
            ctypes.c_void_p(_ptr(exp_avg_sq)), p, ctypes.byref(_hp(hparams)), int(step)]


def sharded_step(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step: int,
                 stream=None, grad_dtype: str | None = None) -> None:
    """One fused reduce-scatter + AdamW + bf16 all-gather step (asynchronous).
    ``param_bufs=None`` skips the all-gather (ZeRO-3: gather later with
    ``unshard``)."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step(*args, ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step")


def sharded_step_debug(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step: int,
                       reduced_grad, stream=None, grad_dtype: str | None = None) -> None:
    """``sharded_step`` that also stores the averaged shard gradient."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step_debug(*args, ctypes.c_void_p(_ptr(reduced_grad)),
                                        ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_debug")


def sharded_step_writeback(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step: int,
                           stream=None, grad_dtype: str | None = None) -> None:
    """``sharded_step`` that also stores every element's averaged gradient into
    its owner's slice of the owner's fp32 grad buffer (one pass)."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step_writeback(*args, ctypes.c_void_p(_stream_handle(stream))),
           "fsp_sharded_step_writeback")


def sharded_step_fp32_gather(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict,
                             step: int, stream=None, grad_dtype: str | None = None) -> None:
    """``sharded_step`` whose all-gather writes the fp32 master into fp32 param buffers."""
    if param_bufs is None:
        raise ValueError("param_bufs is required")
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step_fp32_gather(*args, ctypes.c_void_p(_stream_handle(stream))),
           "fsp_sharded_step_fp32_gather")


def sharded_step_noalloc(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step: int,
                         stream=None, grad_dtype: str | None = None) -> None:
    """``sharded_step`` that allocates no device memory (for callers that cannot
    call cudaMalloc; ``param_bufs=None``: the ZeRO-3 step); see
    ``fsp_sharded_step_noalloc`` in include/fsp.h for its size limit and the
    rule that overlapping calls race."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step_noalloc(*args, ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_noalloc")


def device_error() -> int:
    """Reads and clears the device error word (0: every step since the last
    read completed; see ``fsp_device_error``).  Synchronous."""
    bits = ctypes.c_uint32(0)
    _check(lib().fsp_device_error(ctypes.byref(bits)), "fsp_device_error")
    return int(bits.value)


def host_step_workspace_bytes(plan: Plan, grad_dtype: str = "f32", chunk_elems: int = 0) -> int:
    """Device workspace bytes ``sharded_step_host`` needs (chunk_elems 0: 2^24)."""
    out = ctypes.c_size_t(0)
    _check(lib().fsp_host_step_workspace_bytes(plan.handle, DTYPES[grad_dtype], int(chunk_elems), ctypes.byref(out)),
           "fsp_host_step_workspace_bytes")
    return int(out.value)


def sharded_step_host(plan: Plan, host_grads, master, exp_avg, exp_avg_sq, host_params, hparams: dict, step: int,
                      workspace, chunk_elems: int = 0, stream=None, grad_dtype: str | None = None) -> None:
    """The step with gradients and bf16 params in host (pinned) memory and the
    fp32 state on the device; ``workspace`` is a device tensor of at least
    ``host_step_workspace_bytes`` bytes.  Asynchronous on ``stream``."""
    args = _step_args(plan, host_grads, master, exp_avg, exp_avg_sq, host_params, hparams, step, grad_dtype)
    nbytes = workspace.numel() * workspace.element_size() if not isinstance(workspace, int) else 0
    _check(lib().fsp_sharded_step_host(*args, ctypes.c_void_p(_ptr(workspace)), nbytes, int(chunk_elems),
                                       ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_host")


def selftest_bounded_wait(limit_ms: int = 100) -> int:
    """Runs the bounded-wait self-test (a wait nothing completes) and returns
    the device error word it left (bit 4 when the bound worked)."""
    bits = ctypes.c_uint32(0)
    _check(lib().fsp_selftest_bounded_wait(int(limit_ms), ctypes.byref(bits)), "fsp_selftest_bounded_wait")
    return int(bits.value)


def sharded_step_clipped(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step: int,
                         max_norm: float, norm_out, stream=None, grad_dtype: str | None = None) -> None:
    """Reduce-scatter with write-back into the owners' grad slices, global-norm
    clipping, AdamW, cast, all-gather; ``norm_out`` (device, 2 floats) receives
    {norm, coefficient}.  fp32 grads; FSDP2, DistOpt or HSDP plans."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, step, grad_dtype)
    _check(lib().fsp_sharded_step_clipped(*args, float(max_norm), ctypes.c_void_p(_ptr(norm_out)),
                                          ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_clipped")


def shard(plan: Plan, full, master, exp_avg=None, exp_avg_sq=None, stream=None) -> None:
    """FSDP2 shard: copy every owned element of the full fp32 parameters into
    ``master`` (every replica copy for HSDP); zero ``exp_avg`` / ``exp_avg_sq``
    when given.  Asynchronous."""
    z = lambda x: ctypes.c_void_p(None if x is None else _ptr(x))  # noqa: E731
    _check(lib().fsp_shard(plan.handle, ctypes.c_void_p(_ptr(full)), ctypes.c_void_p(_ptr(master)), z(exp_avg),
                           z(exp_avg_sq), ctypes.c_void_p(_stream_handle(stream))), "fsp_shard")


def unshard(plan: Plan, master, param_bufs, stream=None, fp32: bool = False) -> None:
    """FSDP2 unshard: cast every rank's fp32 shard to bf16 (``fp32=True``:
    copy it as it is into fp32 buffers) and gather it into every rank's full
    param buffer (of its group).  Asynchronous."""
    if len(param_bufs) != plan.n_d:
        raise ValueError(f"need {plan.n_d} param buffers")
    p = (ctypes.c_void_p * plan.n_d)(*[_ptr(b) for b in param_bufs])
    fn = lib().fsp_unshard_fp32 if fp32 else lib().fsp_unshard
    _check(fn(plan.handle, ctypes.c_void_p(_ptr(master)), p, ctypes.c_void_p(_stream_handle(stream))),
           "fsp_unshard_fp32" if fp32 else "fsp_unshard")


def sharded_step_device_t(plan: Plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams: dict, step_dev,
                          advance: bool = True, stream=None, grad_dtype: str | None = None) -> None:
    """``sharded_step`` with the update index in device memory (``step_dev``: a
    one-element int64 CUDA tensor), advanced by one after the step when
    ``advance`` - the form to capture once in a CUDA graph and replay."""
    args = _step_args(plan, grad_bufs, master, exp_avg, exp_avg_sq, param_bufs, hparams, 1, grad_dtype)[:-1]
    _check(lib().fsp_sharded_step_device_t(*args, ctypes.c_void_p(_ptr(step_dev)), int(bool(advance)),
                                           ctypes.c_void_p(_stream_handle(stream))), "fsp_sharded_step_device_t")
