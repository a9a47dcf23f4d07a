"""Helpers for the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and compare them with the stated tolerances."""
from __future__ import annotations

import numpy as np

LOGIT_ABS = 2e-3    # max |delta logit| per step
LOGIT_REL = 1e-4    # max |delta logit| per step, relative to max |oracle logit|
ATT_ABS = 1e-5      # attention probabilities


def check_logits(gpu: np.ndarray, ref: np.ndarray, what: str = ""):
    """Per-step bound: max|d| <= 2e-3 and <= 1e-4 * max|oracle logit| of that step."""
    gpu = np.atleast_2d(gpu)
    ref = np.atleast_2d(ref)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.isfinite(gpu).all(), f"{what}: non-finite logits"
    d = np.abs(gpu.astype(np.float64) - ref).max(axis=1)
    scale = np.abs(ref).max(axis=1)
    bad = np.nonzero((d > LOGIT_ABS) | (d > LOGIT_REL * scale))[0]
    assert bad.size == 0, (f"{what}: step {bad[0]} max|d|={d[bad[0]]:.3e} "
                           f"(bound {min(LOGIT_ABS, LOGIT_REL * scale[bad[0]]):.3e})")
    return float((d / scale).max())


def decoder_for(wl, weights_dev, **kw):
    import llama_transformer_decode_gb300 as pkg
    return pkg.Decoder(wl.config_tuple(), weights_dev, **kw)


def gpu_decode(dec, tokens, pos0: int = 0, out=None):
    """Teacher-forced logits (n, vocab) of slot 0 on the GPU."""
    import torch
    n = len(tokens)
    if out is None:
        out = torch.empty((n, dec.vocab_size), device="cuda")
    for i, tok in enumerate(tokens):
        dec.forward(int(tok), pos0 + i, out[i])
    dec.sync()
    return out.cpu().numpy()
