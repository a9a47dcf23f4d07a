"""Small decode cases run with whichever build of the CUDA library is loaded
(the release build, or the bounds-checked one when the environment sets
L2DECODE_BOUNDS_CHECKED=1), for tests/test_gpu_bounds.py.  Test
infrastructure: run as `python -m tests.bounds_cases OUT.npz` from the
repository root it writes the cases' logits to an .npz file.

The cases cover every instrumented kernel: batch-1 decode (the fused GEMVs and
the flash-decoding attention, with the probability export), steps of several
rows on the CUDA cores and on the tensor cores (stream-K and cluster splits),
a prompt in chunks (the prompt-chunk attention), bf16 weights on both GEMV
paths, and l2_forward_static with its static attention scratch.
"""
import ctypes
import sys

import numpy as np

import synth
from synth import WORKLOADS

RAGGED = WORKLOADS["tiny"].replace(name="ragged_bounds", dim=60, hidden_dim=92, n_layers=3, n_heads=5, n_kv_heads=2,
                                   vocab_size=301, seq_len=70, shared_wcls=False, seed_override=83)
G8 = WORKLOADS["batched_1b"].replace(name="g8_bounds", dim=512, hidden_dim=1376, n_layers=2, n_heads=8,
                                     n_kv_heads=1, vocab_size=1000, seq_len=256, seed_override=89)


def _decode(pkg, torch, wl, w, n, flags=0):
    dec = pkg.Decoder(wl.config_tuple(), w, flags=flags)
    toks = synth.token_stream(wl, 0, n)
    out = torch.empty((n, wl.vocab_size), device="cuda")
    for i, t in enumerate(toks):
        dec.forward(int(t), i, out[i])
    dec.sync()
    extra = {}
    if flags & pkg.L2_FLAG_DEBUG:
        extra = {f"att{layer}": dec.debug_attention(layer) for layer in range(wl.n_layers)}
    dec.close()
    return out.cpu().numpy(), extra


def _batched(pkg, torch, wl, w, B, n_steps, flags=0):
    dec = pkg.Decoder(wl.config_tuple(), w, max_batch=B, flags=flags)
    offsets = [(b * 7) % 40 for b in range(B)]
    for b in range(B):
        if offsets[b]:
            dec.kv_import(synth.kv_rows(wl, b, offsets[b], "k"), synth.kv_rows(wl, b, offsets[b], "v"), slot=b)
    streams = [synth.token_stream(wl, b, offsets[b] + n_steps) for b in range(B)]
    out = torch.empty((n_steps, B, wl.vocab_size), device="cuda")
    for s in range(n_steps):
        dec.forward_batch([int(streams[b][offsets[b] + s]) for b in range(B)], [offsets[b] + s for b in range(B)],
                          out[s])
    dec.sync()
    dec.close()
    return out.cpu().numpy()


def run_cases() -> dict:
    import torch

    import llama_transformer_decode_gb300 as pkg
    res = {}
    tiny = WORKLOADS["tiny"]
    wt = pkg.to_device(synth.make_weights(tiny))
    res["tiny"], _ = _decode(pkg, torch, tiny, wt, 24)
    wr = pkg.to_device(synth.make_weights(RAGGED))
    res["ragged"], att = _decode(pkg, torch, RAGGED, wr, 20, flags=pkg.L2_FLAG_DEBUG)
    res.update({f"ragged_{k}": v for k, v in att.items()})
    res["tiny_b4"] = _batched(pkg, torch, tiny, wt, 4, 2)
    gq = WORKLOADS["gqa_small"]
    wg = pkg.to_device(synth.make_weights(gq))
    res["gqa_small_b16"] = _batched(pkg, torch, gq, wg, 16, 2)
    # a prompt in chunks of 64 and 6 rows
    dec = pkg.Decoder(gq.config_tuple(), wg)
    toks = synth.token_stream(gq, 0, 70)
    out = torch.empty((70, gq.vocab_size), device="cuda")
    dec.prefill(toks, pos0=0, out=out)
    dec.sync()
    res["gqa_small_prefill"] = out.cpu().numpy()
    dec.close()
    # l2_forward_static where attention merges two CTAs per KV head
    dec = pkg.Decoder(gq.config_tuple(), wg)
    dec.kv_import(synth.kv_rows(gq, 0, 200, "k"), synth.kv_rows(gq, 0, 200, "v"))
    out = torch.empty((2, gq.vocab_size), device="cuda")
    for i, t in enumerate(synth.token_stream(gq, 0, 2, start=200)):
        dec.forward_static(int(t), 200 + i, out[i])
    dec.sync()
    res["gqa_small_static"] = out.cpu().numpy()
    dec.close()
    # bf16 weights: batch 1 (CUDA cores) and 16 rows (tensor cores)
    w8 = pkg.to_device(synth.make_weights(G8))
    res["g8_bf16"], _ = _decode(pkg, torch, G8, w8, 6, flags=pkg.L2_FLAG_BF16_WEIGHTS)
    res["g8_bf16_b16"] = _batched(pkg, torch, G8, w8, 16, 2, flags=pkg.L2_FLAG_BF16_WEIGHTS)
    return res


def limited_cache_is_flagged() -> int:
    """With the checks told that each KV cache holds 10 positions of one head,
    a step at position 20 must be flagged (its reads and writes past that are
    skipped, all of them inside the real buffers).  Returns l2_sync's status."""
    import torch  # noqa: F401

    import llama_transformer_decode_gb300 as pkg
    tiny = WORKLOADS["tiny"]
    dec = pkg.Decoder(tiny.config_tuple(), pkg.to_device(synth.make_weights(tiny)))
    toks = synth.token_stream(tiny, 0, 21)
    for i in range(20):
        dec.forward(int(toks[i]), i)
    dec.sync()
    lib = pkg.lib()
    assert lib.l2_debug_limit_cache(dec.handle, ctypes.c_ulonglong(10 * tiny.dim // tiny.n_heads)) == pkg.L2_OK
    dec.forward(int(toks[20]), 20)
    rc = lib.l2_sync(dec.handle)
    dec.close()
    return rc


if __name__ == "__main__":
    import llama_transformer_decode_gb300 as pkg
    out = run_cases()
    out["_checked"] = np.array([pkg.lib().l2_debug_bounds_checked()])
    out["_limited_rc"] = np.array([limited_cache_is_flagged()])
    np.savez(sys.argv[1], **out)
