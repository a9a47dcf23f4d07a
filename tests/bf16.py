"""Round fp32 arrays to bf16 values (returned as fp32), for the tests of the
bf16 weight streaming: the oracle runs on the matrices this returns, which is
the model a handle created with L2_FLAG_BF16_WEIGHTS computes.

bf16 keeps the top 16 bits of an fp32 (sign, 8 exponent bits, 7 mantissa
bits); rounding is IEEE 754 round to nearest, ties to even: add 0x7FFF plus
the lowest kept bit, then clear the low 16 bits (a carry out of the mantissa
moves to the next binade, as it should).  Finite inputs only.
"""
import numpy as np


def round_bf16(a) -> np.ndarray:
    u = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + keep_lsb) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).reshape(np.shape(a))


# the matrices the handle streams as bf16 (embedding table, gains stay fp32)
BF16_MATRICES = ("wq", "wk", "wv", "wo", "w1", "w2", "w3", "wcls")


def rounded_model(weights: dict) -> dict:
    """The weights a bf16-streaming handle computes with: matrices rounded, the
    rest (embedding rows, RMSNorm gains) as given; a classifier shared with the
    embedding table is rounded as the classifier only."""
    out = dict(weights)
    for k in BF16_MATRICES:
        out[k] = round_bf16(weights[k])
    return out
