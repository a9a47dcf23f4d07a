"""Tensor-core GEMV path (batched steps and prompt chunks of 16 to 64 rows).

Steps of 16 or more rows run their matrix products as 3xTF32 MMAs on the
tensor cores.  Checked against the oracle with the same per-step logit bounds
as every other path: ragged batch sizes (16, 17, 33, 48, 64 rows, padded to
multiples of 16 for the MMA), K extents that are not multiples of the 32-column
tile (dim 60, hidden 92 and 172), vocabularies that end mid-tile, K split
across CTAs (the workspace and ticket merge), prompt chunks through the same
kernels, bitwise repeatability, the CUDA-core path with L2_FLAG_NO_TC on the
same inputs, and the launch count.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import check_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402

G8 = WORKLOADS["batched_1b"].replace(name="g8tc", dim=512, hidden_dim=1376, n_layers=2, n_heads=8, n_kv_heads=1,
                                     vocab_size=1000, seq_len=256, seed_override=95)
RAGGED = WORKLOADS["tiny"].replace(name="ragged_tc", dim=60, hidden_dim=92, n_layers=2, n_heads=5, n_kv_heads=2,
                                   vocab_size=301, seq_len=96, shared_wcls=False, seed_override=79)


def staggered(wl, B, n_steps, flags=0, weights=None, offsets=None):
    """n_steps batched steps of B slots at staggered positions; returns the
    logits (n_steps, B, vocab) and the oracle's."""
    w = weights if weights is not None else synth.make_weights(wl)
    if offsets is None:
        offsets = [(b * 7) % 40 for b in range(B)]
    ref = oracle.Model(wl.config_tuple(), w, n_slots=B)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=B, flags=flags)
    streams = [synth.token_stream(wl, 200 + b, offsets[b] + n_steps) for b in range(B)]
    for b in range(B):
        if offsets[b]:
            ref.decode(streams[b][: offsets[b]], slot=b)
        dec.kv_import(ref.key_cache[b][:, : offsets[b]], ref.value_cache[b][:, : offsets[b]], slot=b)
    out = torch.empty((n_steps, B, wl.vocab_size), device="cuda")
    refs = np.empty((n_steps, B, wl.vocab_size), np.float64)
    for s in range(n_steps):
        toks = [int(streams[b][offsets[b] + s]) for b in range(B)]
        pos = [offsets[b] + s for b in range(B)]
        dec.forward_batch(toks, pos, out[s])
        for b in range(B):
            refs[s, b] = ref.forward(toks[b], pos[b], slot=b)
    dec.sync()
    return dec, out.cpu().numpy(), refs


@pytest.mark.parametrize("wl,B", [(WORKLOADS["tiny"], 16), (WORKLOADS["tiny"], 17), (RAGGED, 33), (RAGGED, 64),
                                  (G8, 48), (WORKLOADS["gqa_small"], 20)],
                         ids=["tiny16", "tiny17", "ragged33", "ragged64", "g8_48", "gqa_small20"])
def test_tc_batched_against_oracle(wl, B):
    dec, got, refs = staggered(wl, B, 4)
    assert dec.kernels_per_step(B) == 5 * wl.n_layers + 2  # the embedding kernel runs first
    for b in range(B):
        check_logits(got[:, b], refs[:, b], f"{wl.name} B={B} slot {b}")


def test_tc_and_cuda_core_paths_agree_and_repeat():
    wl = G8
    w = synth.make_weights(wl)
    _, a, refs = staggered(wl, 24, 3, weights=w)
    _, a2, _ = staggered(wl, 24, 3, weights=w)
    dec, c, _ = staggered(wl, 24, 3, flags=pkg.L2_FLAG_NO_TC, weights=w)
    assert dec.kernels_per_step(24) == 5 * wl.n_layers + 1
    np.testing.assert_array_equal(a, a2)  # split-K partials are added in a fixed order
    for b in range(24):
        check_logits(a[:, b], refs[:, b], f"tensor cores slot {b}")
        check_logits(c[:, b], refs[:, b], f"CUDA cores slot {b}")


def test_tc_eager_matches_graph():
    wl = RAGGED
    w = synth.make_weights(wl)
    _, g, _ = staggered(wl, 16, 3, weights=w)
    _, e, _ = staggered(wl, 16, 3, flags=pkg.L2_FLAG_NO_GRAPH, weights=w)
    np.testing.assert_array_equal(g, e)


@pytest.mark.parametrize("wl,plan", [(G8, [64, 16, 30, 5]), (WORKLOADS["tiny"], [40, 17])], ids=["g8", "tiny"])
def test_tc_prefill_chunks(wl, plan):
    w = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=2)
    ref = oracle.Model(wl.config_tuple(), w, n_slots=2)
    toks = synth.token_stream(wl, 1, sum(plan))
    pos = 0
    for n in plan:
        out = torch.empty((n, wl.vocab_size), device="cuda")
        dec.prefill(toks[pos:pos + n], pos0=pos, slot=1, out=out)
        dec.sync()
        check_logits(out.cpu().numpy(), ref.decode(toks[pos:pos + n], pos0=pos, slot=1),
                     f"{wl.name} prefill rows {pos}..{pos + n - 1}")
        pos += n
    k, v = dec.kv_export(wl.n_layers - 1, n_pos=pos, slot=1)
    assert np.abs(k - ref.key_cache[1][wl.n_layers - 1, :pos]).max() <= 1e-4
    assert np.abs(v - ref.value_cache[1][wl.n_layers - 1, :pos]).max() <= 1e-4
