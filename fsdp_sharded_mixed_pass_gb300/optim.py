"""An optimizer-shaped handle over the library: one data-parallel group's plan
and fp32 master / Adam m / Adam v state on one device, and the update index.

It allocates the state (PyTorch device memory) and calls the C ABI; every
computation - shard, step, unshard - runs in the library's kernels.
"""
from __future__ import annotations

from . import fsp as _fsp


def _on_stream(stream):
    """A torch stream context for a stream argument of the binding (None: the
    current stream, an int: a raw cudaStream_t)."""
    import torch
    if stream is None:
        return torch.cuda.stream(torch.cuda.current_stream())
    if isinstance(stream, int):
        return torch.cuda.stream(torch.cuda.ExternalStream(stream))
    return torch.cuda.stream(stream)


class ShardedAdamW:
    """``ShardedAdamW(shapes, n_d, mode="fsdp2")`` - FSDP2 Shard(0) (``"fsdp2"``),
    DistOpt flat shards (``"distopt"``) or HSDP (``"hsdp"`` with
    ``n_replicate`` groups) over ``n_d`` ranks held as buffers on ``device``.

    ``load_full(full)`` shards full fp32 parameters (the plan's full index,
    ``plan.full_len_padded`` elements) into the master and zeroes m and v;
    ``step(grad_bufs, param_bufs)`` applies update t + 1 (the fused
    reduce-scatter + AdamW + bf16 all-gather; ``param_bufs=None`` leaves the
    parameters sharded); ``unshard(param_bufs)`` gathers the current master.
    ``load_params(tensors)`` does what ``load_full`` does from one fp32 tensor
    per parameter.  ``ShardedAdamW.on_tensors(shapes, n_d, grads, params)``
    works on per-parameter tensors instead of full-size buffers (FSDP2's own
    layout): ``step()`` and ``unshard()`` take no buffers.

    ``capturable=True`` keeps the update index in device memory: ``step``
    reads it there and advances it on the device, so a step can be captured
    once in a CUDA graph and replayed (make one eager ``step`` first - it sets
    up what the library keeps on the device - then capture).  ``t`` then reads
    the device counter (a synchronising copy).
    """

    def __init__(self, shapes, n_d: int, mode: str = "fsdp2", n_replicate: int = 1, lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 1e-2, device="cuda",
                 capturable: bool = False):
        self._setup(_fsp.plan_layout(shapes, n_d, mode, n_replicate=n_replicate), lr, betas, eps, weight_decay,
                    device, capturable)

    @classmethod
    def on_tensors(cls, shapes, n_d: int, grads, params=None, n_replicate: int = 1, lr: float = 1e-3,
                   betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 1e-2, device="cuda",
                   capturable: bool = False) -> "ShardedAdamW":
        """FSDP2's own layout: ``grads[q][i]`` and ``params[q][i]`` are rank q's
        gradient and (bf16 or fp32) parameter tensors of parameter i, registered
        once; ``step()`` and ``unshard()`` then read and write them in place
        (FSDP2, or HSDP with ``n_replicate`` groups)."""
        self = cls.__new__(cls)
        self._setup(_fsp.plan_layout_params(shapes, n_d, n_replicate=n_replicate), lr, betas, eps, weight_decay,
                    device, capturable)
        self.table = _fsp.ParamTable(self.plan, grads, params)
        return self

    def _setup(self, plan, lr, betas, eps, weight_decay, device, capturable):
        import torch
        self.plan = plan
        self.table = None
        self.device = device
        n = self.plan.state_len_total
        self.master = torch.zeros(n, dtype=torch.float32, device=device)
        self.exp_avg = torch.zeros(n, dtype=torch.float32, device=device)
        self.exp_avg_sq = torch.zeros(n, dtype=torch.float32, device=device)
        self.hparams = dict(lr=float(lr), beta1=float(betas[0]), beta2=float(betas[1]), eps=float(eps),
                            weight_decay=float(weight_decay))
        # capturable: the index of the NEXT update, on the device
        self._next_t = torch.ones(1, dtype=torch.int64, device=device) if capturable else None
        self._t = 0

    @property
    def capturable(self) -> bool:
        return self._next_t is not None

    @property
    def t(self) -> int:
        """Index of the last update applied (0 before the first)."""
        if self._next_t is not None:
            return int(self._next_t.item()) - 1
        return self._t

    @t.setter
    def t(self, value: int) -> None:
        """Resume at update ``value`` + 1 (e.g. after loading a checkpoint)."""
        if value < 0:
            raise ValueError("t must be >= 0")
        if self._next_t is not None:
            self._next_t.fill_(int(value) + 1)
        else:
            self._t = int(value)

    @property
    def full_len(self) -> int:
        """Elements of every rank's full gradient / parameter buffer."""
        return self.plan.full_len_padded

    def load_full(self, full, stream=None) -> None:
        _fsp.shard(self.plan, full, self.master, self.exp_avg, self.exp_avg_sq, stream=stream)
        if self._next_t is not None:
            with _on_stream(stream):
                self._next_t.fill_(1)
        else:
            self._t = 0

    def load_params(self, tensors, stream=None) -> None:
        """``load_full`` from one fp32 tensor per parameter (any shape with the
        parameter's element count): they are copied into the plan's full index
        on ``stream``, then sharded."""
        import torch
        offs = self.plan.param_offsets
        if len(tensors) != len(offs):
            raise ValueError(f"need {len(offs)} parameter tensors")
        with _on_stream(stream):
            full = torch.zeros(self.full_len, dtype=torch.float32, device=self.device)
            for o, x in zip(offs, tensors):
                full[o:o + x.numel()] = x.reshape(-1)
        self.load_full(full, stream=stream)   # same stream: the copies land first, the buffer outlives the kernel

    def step(self, grad_bufs=None, param_bufs=None, stream=None, grad_dtype: str | None = None) -> None:
        if self.table is not None:
            if grad_bufs is not None or param_bufs is not None:
                raise ValueError("this optimizer steps its registered tensors: pass no buffers")
            if self._next_t is not None:
                _fsp.sharded_step_params_device_t(self.plan, self.table, self.master, self.exp_avg, self.exp_avg_sq,
                                                  self.hparams, self._next_t, advance=True, stream=stream)
                return
            _fsp.sharded_step_params(self.plan, self.table, self.master, self.exp_avg, self.exp_avg_sq,
                                     self.hparams, self._t + 1, stream=stream)
            self._t += 1
            return
        if self._next_t is not None:
            _fsp.sharded_step_device_t(self.plan, grad_bufs, self.master, self.exp_avg, self.exp_avg_sq,
                                       param_bufs, self.hparams, self._next_t, advance=True, stream=stream,
                                       grad_dtype=grad_dtype)
            return
        _fsp.sharded_step(self.plan, grad_bufs, self.master, self.exp_avg, self.exp_avg_sq, param_bufs,
                          self.hparams, self._t + 1, stream=stream, grad_dtype=grad_dtype)
        self._t += 1   # only once the step was accepted

    def unshard(self, param_bufs=None, stream=None) -> None:
        if self.table is not None:
            if param_bufs is not None:
                raise ValueError("this optimizer gathers into its registered tensors: pass no buffers")
            _fsp.unshard_params(self.plan, self.table, self.master, stream=stream)
            return
        _fsp.unshard(self.plan, self.master, param_bufs, stream=stream)
