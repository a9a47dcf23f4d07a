"""ORACLE -- test infrastructure, not part of the product.

Python access (ctypes) to ``l2_oracle.c``, the plain CPU statement of the
llama2.c decode step, and to ``sampler_oracle.c``, the statement of its
token sampler.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library under
``llama_transformer_decode_gb300`` never does, and the two share no code.

Every function here is marshalling only: the arithmetic is in the C file,
which cites the page and section each function follows.  Parity status of
each function (what pins it) is recorded in the tests under ``tests/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "l2_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_SSRC = os.path.join(_HERE, "sampler_oracle.c")
_SOUT = os.path.join(_HERE, "_build", "libsampler_oracle.so")
_lib = None
_slib = None

_FP = ctypes.POINTER(ctypes.c_float)


class OracleConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("dim", "hidden_dim", "n_layers", "n_heads", "n_kv_heads", "vocab_size", "seq_len")]


class OracleWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("token_embedding_table", "rms_att_weight", "rms_ffn_weight", "wq", "wk", "wv",
                 "wo", "w1", "w2", "w3", "rms_final_weight", "wcls")]


def compile_oracle(src: str, out: str, extra: tuple = ()) -> str:
    """gcc -O3 -fopenmp build of an oracle source file into a shared library."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O3", "-fopenmp", "-fPIC", "-shared", *extra, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    build_sampler(force)
    if not force and os.path.exists(_OUT) and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC):
        return _OUT
    return compile_oracle(_SRC, _OUT)


def build_sampler(force: bool = False) -> str:
    """The sampler's statement is built without contraction of a*b+c into one
    fused operation, so every fp32 operation is the one written."""
    if not force and os.path.exists(_SOUT) and os.path.getmtime(_SOUT) >= os.path.getmtime(_SSRC):
        return _SOUT
    os.makedirs(os.path.dirname(_SOUT), exist_ok=True)
    tmp = _SOUT + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", _SSRC,
                           "-o", tmp, "-lm"])
    os.replace(tmp, _SOUT)
    return _SOUT


def load_sampler(path: str | None = None):
    """The sampler oracle (built on first use); ``path`` loads another build of it."""
    global _slib
    if path is not None or _slib is None:
        lib = ctypes.CDLL(path or build_sampler())
        u64p = ctypes.POINTER(ctypes.c_uint64)
        lib.oracle_random_u32.argtypes = [u64p]
        lib.oracle_random_u32.restype = ctypes.c_uint32
        lib.oracle_sampler_exp.argtypes = [ctypes.c_float]
        lib.oracle_sampler_exp.restype = ctypes.c_float
        lib.oracle_argmax.argtypes = [ctypes.c_void_p, ctypes.c_int]
        lib.oracle_argmax.restype = ctypes.c_int
        lib.oracle_sample.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_float, u64p, u64p, u64p]
        lib.oracle_sample.restype = ctypes.c_int
        if path is not None:
            return lib
        _slib = lib
    return _slib


def random_u32(state: int, lib=None):
    """One xorshift* draw: (value, next state)."""
    st = ctypes.c_uint64(state)
    v = (lib or load_sampler()).oracle_random_u32(ctypes.byref(st))
    return int(v), int(st.value)


def sampler_exp(x: float, lib=None) -> float:
    return float((lib or load_sampler()).oracle_sampler_exp(float(x)))


def argmax(v, lib=None) -> int:
    v = np.ascontiguousarray(v, dtype=np.float32)
    return int((lib or load_sampler()).oracle_argmax(v.ctypes.data, v.size))


def sample(logits, temperature: float, topp: float, state: int, lib=None):
    """One token from fp32 logits: (index, next state, total S or P, scaled coin r)."""
    x = np.ascontiguousarray(logits, dtype=np.float32)
    st, tot, r = ctypes.c_uint64(state), ctypes.c_uint64(0), ctypes.c_uint64(0)
    idx = (lib or load_sampler()).oracle_sample(x.ctypes.data, x.size, float(temperature), float(topp),
                                                ctypes.byref(st), ctypes.byref(tot), ctypes.byref(r))
    if idx < 0:
        raise ValueError("oracle_sample rejected its input")
    return int(idx), int(st.value), int(tot.value), int(r.value)


def _declare(lib):
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.oracle_rmsnorm.argtypes = [vp, vp, vp, i]
    lib.oracle_softmax.argtypes = [vp, i]
    lib.oracle_matmul.argtypes = [vp, vp, vp, i, i]
    lib.oracle_rope.argtypes = [vp, i, i, i]
    lib.oracle_kv_head.argtypes = [i, i, i]
    lib.oracle_kv_head.restype = i
    lib.oracle_attention_head.argtypes = [vp, vp, vp, vp, i, i, i, vp]
    lib.oracle_forward.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                   vp, vp, i, i, vp, vp]
    lib.oracle_forward.restype = i
    lib.oracle_decode.argtypes = [ctypes.POINTER(OracleConfig), ctypes.POINTER(OracleWeights),
                                  vp, vp, vp, i, i, vp]
    lib.oracle_decode.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    for f in (lib.oracle_rmsnorm, lib.oracle_softmax, lib.oracle_matmul, lib.oracle_rope,
              lib.oracle_attention_head):
        f.restype = None
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use); ``path`` loads another build of it."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def num_threads(lib=None) -> int:
    """Threads the oracle's parallel loops run on (OpenMP's team size)."""
    return int((lib or load()).oracle_num_threads())


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def rmsnorm(x, w, lib=None) -> np.ndarray:
    x, w = _f32(x), _f32(w)
    o = np.empty_like(x)
    (lib or load()).oracle_rmsnorm(o.ctypes.data, x.ctypes.data, w.ctypes.data, x.size)
    return o


def softmax(x, lib=None) -> np.ndarray:
    x = _f32(x).copy()
    (lib or load()).oracle_softmax(x.ctypes.data, x.size)
    return x


def matmul(w, x, lib=None) -> np.ndarray:
    """W (d, n) @ x (n,)."""
    w, x = _f32(w), _f32(x)
    d, n = w.shape
    o = np.empty(d, dtype=np.float32)
    (lib or load()).oracle_matmul(o.ctypes.data, x.ctypes.data, w.ctypes.data, n, d)
    return o


def rope(vec, head_size: int, pos: int, lib=None) -> np.ndarray:
    v = _f32(vec).copy()
    (lib or load()).oracle_rope(v.ctypes.data, v.size, head_size, pos)
    return v


def kv_head(h: int, n_heads: int, n_kv_heads: int, lib=None) -> int:
    return int((lib or load()).oracle_kv_head(h, n_heads, n_kv_heads))


def attention_head(q, k_rows, v_rows, pos: int, lib=None):
    """One query head over cache rows 0..pos; k_rows, v_rows are (>= pos+1, head_size)."""
    q, k, v = _f32(q), _f32(k_rows), _f32(v_rows)
    hs = q.size
    out = np.empty(hs, dtype=np.float32)
    att = np.empty(pos + 1, dtype=np.float64)
    (lib or load()).oracle_attention_head(out.ctypes.data, q.ctypes.data, k.ctypes.data,
                                          v.ctypes.data, hs, hs, pos, att.ctypes.data)
    return out, att


class Model:
    """A decoder over host weights with one KV cache per batch slot.

    ``weights`` maps the tensor names of ``synth.Workload.tensor_names()`` to
    float32 arrays in the row-major [out][in] layout; the arrays are kept
    alive by this object.
    """

    def __init__(self, config: tuple, weights: dict, n_slots: int = 1, lib=None):
        self.lib = lib or load()
        self.cfg = OracleConfig(*config)
        dim, hidden, L, H, KV, V, S = config
        self.dim, self.n_layers, self.n_heads, self.vocab, self.seq_len = dim, L, H, V, S
        self.kv_dim = dim * KV // H
        self._keep = {k: _f32(v) for k, v in weights.items()}
        k = self._keep
        names = ("emb", "rms_att", "rms_ffn", "wq", "wk", "wv", "wo", "w1", "w2", "w3",
                 "rms_final", "wcls")
        self.w = OracleWeights(*[k[n].ctypes.data for n in names])
        self.key_cache = [np.zeros((L, S, self.kv_dim), np.float32) for _ in range(n_slots)]
        self.value_cache = [np.zeros((L, S, self.kv_dim), np.float32) for _ in range(n_slots)]

    def forward(self, token: int, pos: int, slot: int = 0, want_att: bool = False):
        logits = np.empty(self.vocab, np.float32)
        att = np.zeros((self.n_layers, self.n_heads, self.seq_len), np.float32) if want_att else None
        rc = self.lib.oracle_forward(ctypes.byref(self.cfg), ctypes.byref(self.w),
                                     self.key_cache[slot].ctypes.data,
                                     self.value_cache[slot].ctypes.data, int(token), int(pos),
                                     logits.ctypes.data, att.ctypes.data if want_att else None)
        if rc != 0:
            raise ValueError(f"oracle_forward rejected token={token} pos={pos}")
        return (logits, att) if want_att else logits

    def decode(self, tokens, pos0: int = 0, slot: int = 0) -> np.ndarray:
        """Teacher-forced logits (n, vocab) for tokens at positions pos0.."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty((toks.size, self.vocab), np.float32)
        rc = self.lib.oracle_decode(ctypes.byref(self.cfg), ctypes.byref(self.w),
                                    self.key_cache[slot].ctypes.data,
                                    self.value_cache[slot].ctypes.data, toks.ctypes.data, pos0,
                                    toks.size, out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_decode rejected its input")
        return out
