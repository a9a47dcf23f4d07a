"""Seeded synthetic inputs: weights and token streams for the decode workloads.

This package is shared by the oracle tests, the CUDA-path tests and the
benchmark, and it holds none of the decode step's arithmetic: it maps
(seed, tensor id, element index) to numbers with a counter-based splitmix64
generator and Box-Muller normals (the exact recipe is in ``synth.c``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .workloads import WORKLOADS, Workload, TENSOR_IDS, token_stream_id  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_OUT = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``_build/libsynth.so`` (gcc, OpenMP)."""
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64 = ctypes.c_uint64
        lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double,
                                         ctypes.c_void_p]
        lib.synth_normal_f32.restype = None
        lib.synth_tokens_i32.argtypes = [u64, u64, u64, u64, ctypes.c_uint32, ctypes.c_void_p]
        lib.synth_tokens_i32.restype = None
        lib.synth_draw_u64.argtypes = [u64, u64, u64]
        lib.synth_draw_u64.restype = u64
        _lib = lib
    return _lib


def draw_u64(seed: int, tensor_id: int, n: int) -> int:
    return int(_load().synth_draw_u64(seed, tensor_id, n))


def normal(seed: int, tensor_id: int, start: int, count: int, mean: float, std: float,
           out: np.ndarray | None = None) -> np.ndarray:
    """float32 values mean + std*z for elements [start, start+count) of a tensor stream."""
    if out is None:
        out = np.empty(count, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == count
    _load().synth_normal_f32(seed, tensor_id, start, count, mean, std, out.ctypes.data)
    return out


def tokens(seed: int, tensor_id: int, start: int, count: int, vocab: int) -> np.ndarray:
    """int32 token ids uniform on [0, vocab) for positions [start, start+count)."""
    out = np.empty(count, dtype=np.int32)
    _load().synth_tokens_i32(seed, tensor_id, start, count, vocab, out.ctypes.data)
    return out


def fill_tensor(wl: Workload, name: str, out: np.ndarray, seed: int | None = None) -> np.ndarray:
    """Fill ``out`` (shape ``wl.shape(name)``) with the workload's recipe for tensor ``name``."""
    seed = wl.seed if seed is None else seed
    tid = TENSOR_IDS[name]
    flat = out.reshape(-1)
    mean, std_fn = wl.recipe(name)
    if name in wl.layered:
        per = flat.size // wl.n_layers
        for l in range(wl.n_layers):
            normal(seed, tid, l * per, per, mean, std_fn(l), flat[l * per:(l + 1) * per])
    else:
        normal(seed, tid, 0, flat.size, mean, std_fn(0), flat)
    return out


def fill_range(wl: Workload, name: str, start: int, out: np.ndarray, seed: int | None = None) -> np.ndarray:
    """Elements [start, start + out.size) of tensor ``name``'s flat stream
    (the same values ``fill_tensor`` produces there), for streaming a large
    tensor through a small host buffer."""
    seed = wl.seed if seed is None else seed
    tid = TENSOR_IDS[name]
    flat = out.reshape(-1)
    mean, std_fn = wl.recipe(name)
    if name not in wl.layered:
        return normal(seed, tid, start, flat.size, mean, std_fn(0), flat)
    shape = wl.shape(name)
    per = int(np.prod(shape[1:]))
    done = 0
    while done < flat.size:
        i = start + done
        l = i // per
        n = min(flat.size - done, (l + 1) * per - i)
        normal(seed, tid, i, n, mean, std_fn(l), flat[done:done + n])
        done += n
    return out


def make_weights(wl: Workload, seed: int | None = None) -> dict:
    """All weight tensors of a workload as float32 numpy arrays, row-major [out][in].

    When the workload shares the classifier with the embedding table, the
    dict's ``wcls`` entry is the very same array as ``emb``.
    """
    w = {}
    for name in wl.tensor_names():
        if name == "wcls" and wl.shared_wcls:
            w["wcls"] = w["emb"]
            continue
        w[name] = fill_tensor(wl, name, np.empty(wl.shape(name), dtype=np.float32), seed)
    return w


def kv_rows(wl: Workload, slot: int, n_pos: int, which: str, std: float = 1.0,
            seed: int | None = None) -> np.ndarray:
    """A synthetic KV-cache prefix (n_layers, n_pos, kv_dim) ~ N(0, std^2) for
    slot ``slot``; ``which`` is "k" or "v".  Stands in for rows 0..n_pos-1 that
    earlier steps would have written."""
    seed = wl.seed if seed is None else seed
    tid = (200 if which == "k" else 300) + slot
    out = np.empty((wl.n_layers, n_pos, wl.kv_dim), np.float32)
    if out.size:
        normal(seed, tid, 0, out.size, 0.0, std, out.reshape(-1))
    return out


def token_stream(wl: Workload, slot: int, count: int, start: int = 0, seed: int | None = None) -> np.ndarray:
    seed = wl.seed if seed is None else seed
    return tokens(seed, token_stream_id(slot), start, count, wl.vocab_size)
