"""The synthetic workloads: parameter shapes, N_d, layout mode, grad dtype.

Shapes follow the model descriptions they stand for (no weights or data are
involved; values come from the seeded generator in this package):

* ``qwen3_layer``  - one simplified Qwen3 decoder layer exactly as listed in
  "FSDP2 Qwen3 Decoder Layer Walkthrough", section "参数列表（单层）"
  (d=512, 8 q heads / 4 kv heads of 64, ffn 1024): 11 params, 2,360,448
  elements; N_d=4, FSDP2 Shard(0).
* ``qwen3_0p6b_fsdp2`` - a Qwen3-0.6B-shaped stack: tied embedding
  151936x1024 first, 28 layers of d=1024 with 16 q / 8 kv heads of 128,
  q/k-norm over the head dim, ffn 3072, final norm last: 310 params,
  596,049,920 elements; N_d=8, FSDP2 Shard(0).
* ``qwen3_0p6b_distopt`` - the same stack as one flat buffer split into 8
  contiguous shards (Megatron distributed optimizer / ZeRO-1).
* ``ragged_500`` - 500 params, rows uniform in 1..4099 excluding multiples of
  6, cols uniform in {1, 64, 1024, 4096}; N_d=6, FSDP2 with padding.
* ``dense_1p5b_bf16grad`` - 24 layers of d=2048, 16 q / 4 kv heads of 128,
  ffn 5632 (no embedding, no q/k-norm named): 216 params, 1,082,228,736
  elements; N_d=16, bf16 gradients reduced in fp32.
* ``qwen3_0p6b_hsdp_2x4`` - the Qwen3-0.6B-shaped stack under HSDP
  ("Parallelism strategies: which state to shard", section 二.6): 2 replica
  groups of 4 shard ranks (N_d=8), fp32 grads.

All share AdamW lr 3e-4, betas (0.9, 0.95), eps 1e-8, weight decay 0.1 and
update index t=10; data seed 0x5EED0000 + workload index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

MASK64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def _mix(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    shapes: tuple
    n_d: int
    mode: str            # "fsdp2" | "distopt" | "hsdp"
    grad_dtype: str      # "f32" | "bf16"
    n_rep: int = 1       # HSDP replica groups (N_d = n_rep x shard-group size)
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    step: int = 10
    description: str = field(default="", compare=False)

    @property
    def data_seed(self) -> int:
        return 0x5EED0000 + self.index

    @property
    def numel(self) -> int:
        total = 0
        for s in self.shapes:
            n = 1
            for d in s:
                n *= d
            total += n
        return total

    @property
    def grad_bytes(self) -> int:
        return 4 if self.grad_dtype == "f32" else 2

    def hparams(self) -> dict:
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay)


def qwen3_layer_shapes(d, n_q, n_kv, d_h, ffn, qk_norm=True):
    """One decoder layer's weights in the walkthrough's order."""
    s = [(d,), (n_q * d_h, d), (n_kv * d_h, d), (n_kv * d_h, d)]
    if qk_norm:
        s += [(d_h,), (d_h,)]
    s += [(d, n_q * d_h), (d,), (ffn, d), (ffn, d), (d, ffn)]
    return s


def qwen3_0p6b_shapes():
    shapes = [(151936, 1024)]
    for _ in range(28):
        shapes += qwen3_layer_shapes(1024, 16, 8, 128, 3072)
    shapes.append((1024,))
    return tuple(shapes)


def dense_1p5b_shapes():
    shapes = []
    for _ in range(24):
        shapes += qwen3_layer_shapes(2048, 16, 4, 128, 5632, qk_norm=False)
    return tuple(shapes)


def ragged_shapes(n_params=500, n_d=6, seed=0xF5D0, max_rows=4099, col_choices=(1, 64, 1024, 4096)):
    """Rows uniform in 1..max_rows with multiples of n_d rejected; cols uniform
    over ``col_choices``; drawn from the sequential SplitMix64 stream of ``seed``."""
    state = seed & MASK64

    def nxt():
        nonlocal state
        state = (state + _GAMMA) & MASK64
        return _mix(state)

    shapes = []
    while len(shapes) < n_params:
        rows = 1 + nxt() % max_rows
        if rows % n_d == 0:
            continue
        cols = col_choices[nxt() % len(col_choices)]
        shapes.append((rows, cols) if cols != 1 else (rows,))
    return tuple(shapes)


WORKLOADS = (
    Workload(0, "qwen3_layer", tuple(qwen3_layer_shapes(512, 8, 4, 64, 1024)), 4, "fsdp2", "f32",
             description="one simplified Qwen3 decoder layer, N_d=4, FSDP2 Shard(0)"),
    Workload(1, "qwen3_0p6b_fsdp2", qwen3_0p6b_shapes(), 8, "fsdp2", "f32",
             description="Qwen3-0.6B-shaped stack, N_d=8, FSDP2 Shard(0), fp32 grads"),
    Workload(2, "qwen3_0p6b_distopt", qwen3_0p6b_shapes(), 8, "distopt", "f32",
             description="Qwen3-0.6B-shaped stack, N_d=8, DistOpt flat shards, fp32 grads"),
    Workload(3, "ragged_500", ragged_shapes(), 6, "fsdp2", "f32",
             description="500 ragged params, N_d=6, FSDP2 Shard(0) with padding, fp32 grads"),
    Workload(4, "dense_1p5b_bf16grad", dense_1p5b_shapes(), 16, "fsdp2", "bf16",
             description="24-layer d=2048 GQA/SwiGLU stack, N_d=16, FSDP2, bf16 grads reduced in fp32"),
    Workload(5, "qwen3_0p6b_hsdp_2x4", qwen3_0p6b_shapes(), 8, "hsdp", "f32", n_rep=2,
             description="Qwen3-0.6B-shaped stack, HSDP: 2 replica groups x 4 shard ranks, fp32 grads"),
)


def workload(key) -> Workload:
    if isinstance(key, int):
        return WORKLOADS[key]
    for w in WORKLOADS:
        if w.name == key:
            return w
    raise KeyError(key)
