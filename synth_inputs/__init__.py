"""Seeded synthetic inputs for the sharded mixed-precision step.

This module is the one piece that both the CUDA path and the oracle use, and it
holds none of the step's arithmetic: it only turns (seed, array, rank, logical
element index) into a number.  The same generator exists twice, once here in
numpy (host) and once as a CUDA kernel in ``synth_inputs/csrc/synth.cu``; both
are integer-only up to one final, correctly rounded fp32 multiply, so they give
bit-identical values, which a GPU test checks.

Generator (written from its published definition):

* SplitMix64's output function (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014) used counter-style:
  ``word(key, i, j) = mix64(key + GAMMA * (3*i + j + 1))``.
* ``key = mix64(mix64(seed) ^ (array_id << 32 | rank))``.
* uniform in [0, hi): ``(word >> 40) * 2**-24 * hi``.
* approximately normal N(0, sigma): Irwin-Hall sum of twelve 16-bit uniforms
  taken from three words, centred and scaled to unit variance exactly
  (``(2*S - 12*65535) * 2**-17``), then ``* sigma``.  It has mean 0 and
  variance 1 - 2**-32 and is bounded by +-6 sigma.  It stands in for a
  Gaussian because it needs no transcendental function and is therefore
  bit-reproducible on host and device.
* bf16 gradients: the high 16 bits of the fp32 value (truncation).  This is the
  generator's own quantisation and differs on purpose from the round-to-nearest
  cast that the step applies to parameters.

Array ids: a rank's gradient is (array_id=0, rank=q); master 100, Adam m 101,
Adam v 102 (rank 0).  Every value is keyed by the element's *logical* index in
the model's flat parameter order, so the same model gives the same numbers
whatever the layout.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX_C1 = 0xBF58476D1CE4E5B9
MIX_C2 = 0x94D049BB133111EB

ARRAY_GRAD = 0
ARRAY_MASTER = 100
ARRAY_M = 101
ARRAY_V = 102

# Value distributions of the workloads: grads ~N(0, 1e-3), master ~N(0, 0.02),
# Adam m ~N(0, 1e-4), Adam v ~U[0, 1e-6]; the second parameter of N is a
# standard deviation.
SIGMA_GRAD = np.float32(1e-3)
SIGMA_MASTER = np.float32(0.02)
SIGMA_M = np.float32(1e-4)
V_HI = np.float32(1e-6)


def mix64_int(z: int) -> int:
    """SplitMix64 output mix on a Python int (mod 2**64)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_C1) & MASK64
    z = ((z ^ (z >> 27)) * MIX_C2) & MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output mix on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX_C1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX_C2)
    return z ^ (z >> np.uint64(31))


def splitmix64_sequence(seed: int, count: int) -> list[int]:
    """The sequential SplitMix64 generator (state += GAMMA; output mix(state))."""
    out, state = [], seed & MASK64
    for _ in range(count):
        state = (state + GAMMA) & MASK64
        out.append(mix64_int(state))
    return out


def stream_key(seed: int, array_id: int, rank: int) -> int:
    return mix64_int(mix64_int(seed) ^ (((array_id & 0xFFFFFFFF) << 32) | (rank & 0xFFFFFFFF)))


def _words(key: int, idx: np.ndarray, j: int) -> np.ndarray:
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        ctr = idx * np.uint64(3) + np.uint64(j + 1)
        return mix64(np.uint64(key) + np.uint64(GAMMA) * ctr)


_CHUNK = 1 << 16   # elements per pass: keeps the temporaries in cache


def _normal_chunk(key: int, flat: np.ndarray, sigma) -> np.ndarray:
    with np.errstate(over="ignore"):
        ctr = flat.astype(np.uint64)[:, None] * np.uint64(3) + np.arange(1, 4, dtype=np.uint64)[None, :]
        w = mix64(np.uint64(key) + np.uint64(GAMMA) * ctr)          # (n, 3) words
    # the twelve 16-bit fields of the three words, summed (order-free)
    s = w.view(np.uint16).reshape(-1, 12).sum(axis=1, dtype=np.int64)
    n = 2 * s - 12 * 65535
    unit = n.astype(np.float32) * np.float32(2.0 ** -17)  # exact: |n| < 2**24
    return unit * np.float32(sigma)


def normal_f32(key: int, idx: np.ndarray, sigma) -> np.ndarray:
    """Irwin-Hall(12) approximate N(0, sigma) in fp32 at logical indices ``idx``."""
    idx = np.asarray(idx, dtype=np.int64)
    flat = idx.reshape(-1)
    out = np.empty(flat.size, dtype=np.float32)
    for a in range(0, flat.size, _CHUNK):
        out[a:a + _CHUNK] = _normal_chunk(key, flat[a:a + _CHUNK], sigma)
    return out.reshape(idx.shape)


def uniform_f32(key: int, idx: np.ndarray, hi) -> np.ndarray:
    """Uniform in [0, hi) in fp32 at logical indices ``idx`` (24-bit grid)."""
    w = _words(key, np.asarray(idx, dtype=np.int64), 0)
    u = (w >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)  # exact
    return (u * np.float32(hi)).astype(np.float32)


def bf16_bits_trunc(x: np.ndarray) -> np.ndarray:
    """High half of the fp32 bit pattern: the generator's bf16 quantisation."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------
# Per-array convenience, all keyed by logical index.
# ---------------------------------------------------------------------------

def grad_f32(seed: int, rank: int, idx) -> np.ndarray:
    return normal_f32(stream_key(seed, ARRAY_GRAD, rank), idx, SIGMA_GRAD)


def grad_bf16_bits(seed: int, rank: int, idx) -> np.ndarray:
    return bf16_bits_trunc(grad_f32(seed, rank, idx))


def master_f32(seed: int, idx) -> np.ndarray:
    return normal_f32(stream_key(seed, ARRAY_MASTER, 0), idx, SIGMA_MASTER)


def adam_m_f32(seed: int, idx) -> np.ndarray:
    return normal_f32(stream_key(seed, ARRAY_M, 0), idx, SIGMA_M)


def adam_v_f32(seed: int, idx) -> np.ndarray:
    return uniform_f32(stream_key(seed, ARRAY_V, 0), idx, V_HI)


from .workloads import WORKLOADS, Workload, workload  # noqa: E402,F401
