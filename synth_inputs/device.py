"""Device side of the seeded input generator: fills torch CUDA tensors with the
same bits the host generator in ``synth_inputs`` produces."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import synth_inputs as S

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "_build", "libsynth.so")
_lib = None


def build() -> str:
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC", "-shared", os.path.join(HERE, "csrc", "synth.cu"), "-o", tmp]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on synth.cu:\n{r.stdout}")
    os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run synth_inputs.device.build()")
        L = ctypes.CDLL(LIB)
        for name, vt in (("synth_fill_normal_f32", ctypes.c_float), ("synth_fill_normal_bf16trunc", ctypes.c_float),
                         ("synth_fill_uniform_f32", ctypes.c_float)):
            fn = getattr(L, name)
            fn.restype = ctypes.c_int
            fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int64, vt, ctypes.c_void_p]
        _lib = L
    return _lib


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"{what} failed (CUDA error)")


def fill_normal_f32(ptr: int, n: int, key: int, start: int, sigma, stream=None):
    _check(lib().synth_fill_normal_f32(ctypes.c_void_p(ptr), n, key, start, float(sigma), _stream(stream)),
           "synth_fill_normal_f32")


def fill_normal_bf16trunc(ptr: int, n: int, key: int, start: int, sigma, stream=None):
    _check(lib().synth_fill_normal_bf16trunc(ctypes.c_void_p(ptr), n, key, start, float(sigma), _stream(stream)),
           "synth_fill_normal_bf16trunc")


def fill_uniform_f32(ptr: int, n: int, key: int, start: int, hi, stream=None):
    _check(lib().synth_fill_uniform_f32(ctypes.c_void_p(ptr), n, key, start, float(hi), _stream(stream)),
           "synth_fill_uniform_f32")


def fill_grad(t, seed: int, rank: int, grad_dtype: str, start: int = 0, n: int | None = None, stream=None):
    """Rank ``rank``'s gradient at logical indices start .. start+n-1 into tensor ``t``."""
    n = t.numel() if n is None else n
    key = S.stream_key(seed, S.ARRAY_GRAD, rank)
    if grad_dtype == "f32":
        fill_normal_f32(t.data_ptr(), n, key, start, S.SIGMA_GRAD, stream)
    else:
        fill_normal_bf16trunc(t.data_ptr(), n, key, start, S.SIGMA_GRAD, stream)


def fill_state_segments(master, m, v, seed: int, segments, stream=None):
    """master / m / v values at every owned slot, keyed by the slot's logical
    (full-buffer) index.  ``segments``: iterable of (full_off, state_off, len)."""
    km = S.stream_key(seed, S.ARRAY_MASTER, 0)
    ka = S.stream_key(seed, S.ARRAY_M, 0)
    kv = S.stream_key(seed, S.ARRAY_V, 0)
    for full_off, state_off, n in segments:
        if n <= 0:
            continue
        fill_normal_f32(master.data_ptr() + 4 * state_off, n, km, full_off, S.SIGMA_MASTER, stream)
        fill_normal_f32(m.data_ptr() + 4 * state_off, n, ka, full_off, S.SIGMA_M, stream)
        fill_uniform_f32(v.data_ptr() + 4 * state_off, n, kv, full_off, S.V_HI, stream)
