"""The decode workloads: model shapes, weight recipes and token streams.

Five Llama-2-style shapes, all fp32, all with seeded random weights:

==========  =====  ======  ==  ==  ===  =====  ====  ===========================
name        dim    hidden  L   H   KV   vocab  seq   notes
==========  =====  ======  ==  ==  ===  =====  ====  ===========================
tiny        64     172     5   8   4    512    512   classifier shares the embedding table
gqa_small   288    768     6   6   4    32000  256   6 query heads on 4 KV heads
mid         768    2048    12  12  12   32000  1024
llama2_7b   4096   11008   32  32  32   32000  4096  matrix std 0.02/sqrt(layer+1)
batched_1b  2048   5632    22  32  4    32000  2048  B in {1, 16, 64} independent sequences
==========  =====  ======  ==  ==  ===  =====  ====  ===========================

Weights: matrices and the embedding/classifier ~ N(0, 0.02) (the 7B shape
scales its per-layer matrices by 1/sqrt(layer+1)); every RMSNorm gain vector
~ 1 + N(0, 0.01).  Tokens are uniform on [0, vocab).  The seed of workload
number c (1..5 in the order above) is 0x4C32000 + c.  Tensor ids follow the
order in which the llama2.c checkpoint stores the tensors, with the separate
classifier after the RoPE tables; the token stream of batch slot b has id
100 + b.
"""
from __future__ import annotations

import dataclasses
import math

TENSOR_IDS = {
    "emb": 0, "rms_att": 1, "wq": 2, "wk": 3, "wv": 4, "wo": 5, "rms_ffn": 6,
    "w1": 7, "w2": 8, "w3": 9, "rms_final": 10,
    # 11, 12: the RoPE tables of the early checkpoint format (computed, never drawn)
    "wcls": 13,
}

MATRICES = ("wq", "wk", "wv", "wo", "w1", "w2", "w3")


def token_stream_id(slot: int) -> int:
    return 100 + slot


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dim: int
    hidden_dim: int
    n_layers: int
    n_heads: int
    n_kv_heads: int
    vocab_size: int
    seq_len: int
    shared_wcls: bool = False
    layer_scaled: bool = False
    steps: int = 0                 # teacher-forced positions the workload decodes
    batches: tuple = (1,)
    std: float = 0.02
    rms_std: float = 0.01
    std_scale: tuple = ()          # ((tensor name, factor), ...) extra per-tensor std factors
    seed_override: int | None = None

    @property
    def seed(self) -> int:
        return self.seed_override if self.seed_override is not None else 0x4C32000 + self.index

    @property
    def head_size(self) -> int:
        return self.dim // self.n_heads

    @property
    def kv_dim(self) -> int:
        return self.dim * self.n_kv_heads // self.n_heads

    @property
    def layered(self) -> tuple:
        return MATRICES + ("rms_att", "rms_ffn")

    def config_tuple(self) -> tuple:
        return (self.dim, self.hidden_dim, self.n_layers, self.n_heads, self.n_kv_heads,
                self.vocab_size, self.seq_len)

    def tensor_names(self) -> tuple:
        return ("emb", "rms_att", "wq", "wk", "wv", "wo", "rms_ffn", "w1", "w2", "w3",
                "rms_final", "wcls")

    def shape(self, name: str) -> tuple:
        d, h, L, kv, V = self.dim, self.hidden_dim, self.n_layers, self.kv_dim, self.vocab_size
        return {
            "emb": (V, d), "rms_att": (L, d), "rms_ffn": (L, d), "rms_final": (d,),
            "wq": (L, d, d), "wk": (L, kv, d), "wv": (L, kv, d), "wo": (L, d, d),
            "w1": (L, h, d), "w2": (L, d, h), "w3": (L, h, d), "wcls": (V, d),
        }[name]

    def recipe(self, name: str):
        """(mean, layer -> std) of tensor ``name``."""
        factor = dict(self.std_scale).get(name, 1.0)
        if name.startswith("rms"):
            return 1.0, (lambda l: self.rms_std * factor)
        if name in MATRICES and self.layer_scaled:
            return 0.0, (lambda l: self.std * factor / math.sqrt(l + 1))
        return 0.0, (lambda l: self.std * factor)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 172, 5, 8, 4, 512, 512, shared_wcls=True, steps=128),
    "gqa_small": Workload("gqa_small", 2, 288, 768, 6, 6, 4, 32000, 256, steps=256),
    "mid": Workload("mid", 3, 768, 2048, 12, 12, 12, 32000, 1024, steps=1024),
    "llama2_7b": Workload("llama2_7b", 4, 4096, 11008, 32, 32, 32, 32000, 4096,
                          layer_scaled=True, steps=4096),
    "batched_1b": Workload("batched_1b", 5, 2048, 5632, 22, 32, 4, 32000, 2048,
                           steps=2048, batches=(1, 16, 64)),
}
