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

    ``capturable=True`` keeps the update index in device memory: ``step``
    reads it there and advances it on the device, so a step can be captured
    once in a CUDA graph and replayed (make one eager ``step`` first - it sets
    up what the library keeps on the device - then capture).  ``t`` then reads
    the device counter (a synchronising copy).
    """

    def __init__(self, shapes, n_d: int, mode: str = "fsdp2", n_replicate: int = 1, lr: float = 1e-3,
                 betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 1e-2, device="cuda",
                 capturable: bool = False):
        import torch
        self.plan = _fsp.plan_layout(shapes, n_d, mode, n_replicate=n_replicate)
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

    def step(self, grad_bufs, param_bufs, stream=None, grad_dtype: str | None = None) -> None:
        if self._next_t is not None:
            _fsp.sharded_step_device_t(self.plan, grad_bufs, self.master, self.exp_avg, self.exp_avg_sq,
                                       param_bufs, self.hparams, self._next_t, advance=True, stream=stream,
                                       grad_dtype=grad_dtype)
            return
        _fsp.sharded_step(self.plan, grad_bufs, self.master, self.exp_avg, self.exp_avg_sq, param_bufs,
                          self.hparams, self._t + 1, stream=stream, grad_dtype=grad_dtype)
        self._t += 1   # only once the step was accepted

    def unshard(self, param_bufs, stream=None) -> None:
        _fsp.unshard(self.plan, self.master, param_bufs, stream=stream)
