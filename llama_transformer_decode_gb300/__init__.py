"""GB300-native llama2.c decode step: Python binding of the C ABI in ``include/l2.h``.

The binding only marshals arguments: every step of forward(token, pos) ->
logits runs in the CUDA kernels of ``libl2decode.so``.  PyTorch supplies the
device memory (weights, output buffers) and the stream.  There is no CPU
fallback: if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _native
from ._native import EXPORTS, WEIGHT_FIELDS, L2Config, L2Weights, build  # noqa: F401

L2_OK, L2_EINVAL, L2_ESTATE, L2_ENOMEM, L2_ECUDA, L2_EDEVICE, L2_ETIMEOUT = 0, -1, -2, -3, -4, -5, -6
L2_FLAG_DEBUG, L2_FLAG_NO_GRAPH, L2_FLAG_NO_PDL, L2_FLAG_PERSIST, L2_FLAG_NO_TC = 0x1, 0x2, 0x4, 0x8, 0x10
L2_FLAG_BF16_WEIGHTS = 0x20
L2_FLAG_NO_ONE_CTA = 0x40

OPS = {"qkv": 0, "attention": 1, "wo": 2, "w13": 3, "w2": 4, "cls": 5}

# weight dict key (as in synth / the pages' TransformerWeights) -> C struct field
_KEYS = {"emb": "token_embedding_table", "rms_att": "rms_att_weight", "rms_ffn": "rms_ffn_weight",
         "wq": "wq", "wk": "wk", "wv": "wv", "wo": "wo", "w1": "w1", "w2": "w2", "w3": "w3",
         "rms_final": "rms_final_weight", "wcls": "wcls"}


class L2Error(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


def lib():
    return _native.load()


def _ptr(t) -> int:
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError("expected a contiguous float32 CUDA tensor")
    return t.data_ptr()


class Decoder:
    """One decoder handle (``l2_ctx``).

    ``config``: (dim, hidden_dim, n_layers, n_heads, n_kv_heads, vocab_size, seq_len).
    ``weights``: dict of contiguous float32 CUDA tensors keyed like
    ``synth.Workload.tensor_names()``; they are borrowed and kept alive here.
    ``stream``: a ``torch.cuda.Stream`` (default: a new one).
    """

    def __init__(self, config, weights: dict, max_batch: int = 1, flags: int = 0, stream=None):
        import torch
        self._lib = lib()
        self.config = tuple(int(v) for v in config)
        self.dim, self.hidden_dim, self.n_layers, self.n_heads, self.n_kv_heads, self.vocab_size, \
            self.seq_len = self.config
        self.kv_dim = self.dim * self.n_kv_heads // self.n_heads
        self.max_batch = max_batch
        self.flags = flags
        self.stream = stream if stream is not None else torch.cuda.Stream()
        self._weights = dict(weights)
        w = L2Weights(**{_KEYS[k]: _ptr(v) for k, v in self._weights.items()})
        cfg = L2Config(*self.config)
        h = ctypes.c_void_p()
        rc = self._lib.l2_create(ctypes.byref(cfg), ctypes.byref(w), max_batch, flags,
                                 ctypes.c_void_p(self.stream.cuda_stream), ctypes.byref(h))
        if rc != L2_OK:
            raise L2Error(rc, self._lib.l2_last_error(None).decode())
        self._h = h

    # -- helpers -------------------------------------------------------------
    def _check(self, rc: int) -> int:
        if rc < 0:
            raise L2Error(rc, self._lib.l2_last_error(self._h).decode())
        return rc

    @property
    def handle(self):
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            self._lib.l2_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- API -----------------------------------------------------------------
    def forward(self, token: int, pos: int, out=None):
        """Enqueue one step of slot 0; ``out`` is a CUDA tensor of vocab_size floats (or None)."""
        self._check(self._lib.l2_forward(self._h, int(token), int(pos),
                                         ctypes.c_void_p(_ptr(out) if out is not None else 0)))
        return out

    def forward_static(self, token: int, pos: int, out=None):
        """Like forward(), with nothing allocated on the path (l2_forward_static)."""
        self._check(self._lib.l2_forward_static(self._h, int(token), int(pos),
                                                ctypes.c_void_p(_ptr(out) if out is not None else 0)))
        return out

    def forward_batch(self, tokens, pos, out=None):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        ps = np.ascontiguousarray(pos, dtype=np.int32)
        if toks.size != ps.size:
            raise ValueError("tokens and pos differ in length")
        ip = ctypes.POINTER(ctypes.c_int)
        self._check(self._lib.l2_forward_batch(
            self._h, int(toks.size), toks.ctypes.data_as(ip), ps.ctypes.data_as(ip),
            ctypes.c_void_p(_ptr(out) if out is not None else 0)))
        return out

    def prefill(self, tokens, pos0: int = 0, slot: int = 0, out=None):
        """The prompt ``tokens`` at positions pos0.. of ``slot`` (l2_prefill);
        ``out`` a CUDA tensor [T][vocab_size] for every token's logits, or None."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        self._check(self._lib.l2_prefill(self._h, int(slot), int(toks.size),
                                         toks.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), int(pos0),
                                         ctypes.c_void_p(_ptr(out) if out is not None else 0)))
        return out

    def forward_dev_tokens(self, tokens_dev, pos, out=None):
        """One step whose tokens are read from ``tokens_dev`` (CUDA int32 [B])
        when it runs; ``pos`` an int (B = 1) or a list of B ints."""
        import torch
        pos = [int(pos)] if isinstance(pos, int) else [int(v) for v in pos]
        B = len(pos)
        assert tokens_dev.is_cuda and tokens_dev.dtype == torch.int32 and tokens_dev.numel() >= B
        parr = (ctypes.c_int * B)(*pos)
        self._check(self._lib.l2_forward_dev_tokens(self._h, B, ctypes.c_void_p(tokens_dev.data_ptr()), parr,
                                                    ctypes.c_void_p(_ptr(out) if out is not None else None)))
        return out

    def forward_host(self, token: int, pos: int, out: np.ndarray | None = None) -> np.ndarray:
        """Blocking step of slot 0 returning the logits in host memory."""
        if out is None:
            out = np.empty(self.vocab_size, np.float32)
        assert out.dtype == np.float32 and out.flags.c_contiguous and out.size >= self.vocab_size
        self._check(self._lib.l2_forward_host(self._h, int(token), int(pos), ctypes.c_void_p(out.ctypes.data)))
        return out

    def logits_ptr(self) -> int:
        return int(self._lib.l2_logits(self._h) or 0)

    def reset(self, slot: int = -1):
        self._check(self._lib.l2_reset(self._h, int(slot)))

    def position(self, slot: int = 0) -> int:
        return self._check(self._lib.l2_position(self._h, int(slot)))

    def sync(self):
        self._check(self._lib.l2_sync(self._h))

    def debug_wait_timeout(self, limit_us: int):
        """Enqueue a kernel whose bounded wait gives up after limit_us (l2_debug_wait_timeout)."""
        self._check(self._lib.l2_debug_wait_timeout(self._h, int(limit_us)))

    def debug_attention(self, layer: int, slot: int = 0) -> np.ndarray:
        n = self.position(slot)
        out = np.empty((self.n_heads, n), np.float32)
        self._check(self._lib.l2_debug_attention(self._h, int(slot), int(layer), ctypes.c_void_p(out.ctypes.data)))
        return out

    def kv_export(self, layer: int, n_pos: int | None = None, slot: int = 0):
        n = self.position(slot) if n_pos is None else int(n_pos)
        k = np.empty((n, self.kv_dim), np.float32)
        v = np.empty((n, self.kv_dim), np.float32)
        self._check(self._lib.l2_kv_export(self._h, int(slot), int(layer), n, ctypes.c_void_p(k.ctypes.data),
                                           ctypes.c_void_p(v.ctypes.data)))
        return k, v

    def kv_import(self, k: np.ndarray, v: np.ndarray, slot: int = 0):
        """k, v: (n_layers, n_pos, kv_dim) float32 host arrays."""
        k = np.ascontiguousarray(k, np.float32)
        v = np.ascontiguousarray(v, np.float32)
        assert k.shape == v.shape and k.ndim == 3 and k.shape[0] == self.n_layers and k.shape[2] == self.kv_dim
        self._check(self._lib.l2_kv_import(self._h, int(slot), int(k.shape[1]), ctypes.c_void_p(k.ctypes.data),
                                           ctypes.c_void_p(v.ctypes.data)))

    def launch_op(self, op, layer: int = 0, count: int = 1, batch: int = 1):
        """``count`` launches of one kernel of the step (l2_launch_op, or
        l2_launch_op_batch for a step of ``batch`` rows, the last one run)."""
        if batch == 1:
            self._check(self._lib.l2_launch_op(self._h, OPS.get(op, op), int(layer), int(count)))
        else:
            self._check(self._lib.l2_launch_op_batch(self._h, OPS.get(op, op), int(layer), int(batch), int(count)))

    def step_input_bytes(self) -> int:
        return int(self._lib.l2_step_input_bytes())

    def kernels_per_step(self, batch: int = 1) -> int:
        return self._check(self._lib.l2_kernels_per_step(self._h, int(batch)))


def sample(logits, temperature: float, topp: float, rng_state, out=None, stream=None):
    """Next token of each row of ``logits`` (CUDA fp32 [B][vocab]) with the
    pages' sampler (l2_sample): argmax at temperature 0, otherwise one
    xorshift* draw per row from ``rng_state`` (CUDA uint64/int64 [B], advanced
    in place), restricted to the top-p nucleus when 0 < topp < 1.  Returns
    ``out`` (CUDA int32 [B]); enqueued on ``stream`` (default: torch's current)."""
    import torch
    logits = logits if logits.dim() == 2 else logits.reshape(1, -1)
    B, V = logits.shape
    assert logits.dtype == torch.float32 and logits.is_cuda and logits.is_contiguous()
    assert rng_state.is_cuda and rng_state.numel() >= B and rng_state.element_size() == 8 and rng_state.is_contiguous()
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    assert out.dtype == torch.int32 and out.is_cuda and out.numel() >= B
    st = stream if stream is not None else torch.cuda.current_stream()
    rc = lib().l2_sample(ctypes.c_void_p(logits.data_ptr()), B, V, float(temperature), float(topp),
                         ctypes.c_void_p(rng_state.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                         ctypes.c_void_p(st.cuda_stream))
    if rc != L2_OK:
        raise L2Error(rc, lib().l2_last_error(None).decode())
    return out


def fail_alloc_at(n: int):
    """Fault injection: the n-th device allocation from now on fails (0 disables)."""
    lib().l2_debug_fail_alloc_at(int(n))


def fail_graph_at(n: int):
    """Fault injection: the n-th CUDA graph instantiation from now on fails (0 disables)."""
    lib().l2_debug_fail_graph_at(int(n))


def to_device(weights: dict, device="cuda") -> dict:
    """Copy host (numpy) weights to contiguous float32 CUDA tensors, keeping a
    shared classifier shared."""
    import torch
    out, seen = {}, {}
    for k, v in weights.items():
        if id(v) in seen:
            out[k] = out[seen[id(v)]]
            continue
        seen[id(v)] = k
        out[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device)
    return out
