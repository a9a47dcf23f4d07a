"""bf16 weight streaming (L2_FLAG_BF16_WEIGHTS) against the oracle on the same
bf16-rounded matrices.

The handle converts its matrices to bf16 and keeps everything else fp32, so it
computes the model whose matrices are the bf16-rounded ones; the oracle runs
that model (tests/bf16.py rounds the matrices on the host, independently of the
device conversion), and the per-step logit bounds are the fp32 ones.  Batch-1
steps stream the bf16 words through the CUDA-core GEMV; steps of several rows
(batched sequences at staggered positions, prompt chunks) through the tensor
cores (kind::f16 with each input split into three bf16 parts, so the products
are exact).  Also: the flag's argument checks, and that the rounding changes
the result (so the comparison is not vacuous).
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.bf16 import rounded_model
from tests.gpu_util import check_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402

BF16 = pkg.L2_FLAG_BF16_WEIGHTS
G8 = WORKLOADS["batched_1b"].replace(name="g8bf", dim=512, hidden_dim=1376, n_layers=2, n_heads=8, n_kv_heads=1,
                                     vocab_size=1000, seq_len=256, seed_override=97)


@pytest.mark.parametrize("wl", [WORKLOADS["gqa_small"], WORKLOADS["mid"], G8], ids=["gqa_small", "mid", "g8"])
def test_bf16_decode_matches_the_rounded_model(wl):
    w = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), flags=BF16)
    toks = synth.token_stream(wl, 0, 40)
    out = torch.empty((len(toks), wl.vocab_size), device="cuda")
    for i, t in enumerate(toks):
        dec.forward(int(t), i, out[i])
    dec.sync()
    got = out.cpu().numpy()
    want = oracle.Model(wl.config_tuple(), rounded_model(w)).decode(toks)
    check_logits(got, want, f"{wl.name} bf16 weights")
    # the fp32 model is much further away: the comparison above is not vacuous
    full = oracle.Model(wl.config_tuple(), w).decode(toks[:8])
    assert np.abs(got[:8] - full).max() > 10 * np.abs(got[:8] - want[:8]).max()


@pytest.mark.parametrize("wl,B", [(G8, 2), (G8, 16), (WORKLOADS["gqa_small"], 17), (WORKLOADS["mid"], 48),
                                  (G8, 64)], ids=["g8_2", "g8_16", "gqa_small17", "mid48", "g8_64"])
def test_bf16_batched_steps_match_the_rounded_model(wl, B):
    w = synth.make_weights(wl)
    rw = rounded_model(w)
    n_steps = 3
    offsets = [(b * 37) % 90 for b in range(B)]
    ref = oracle.Model(wl.config_tuple(), rw, n_slots=B)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=B, flags=BF16)
    streams = [synth.token_stream(wl, 300 + b, offsets[b] + n_steps) for b in range(B)]
    for b in range(B):
        if offsets[b]:
            ref.decode(streams[b][: offsets[b]], slot=b)
        dec.kv_import(ref.key_cache[b][:, : offsets[b]], ref.value_cache[b][:, : offsets[b]], slot=b)
    out = torch.empty((n_steps, B, wl.vocab_size), device="cuda")
    want = np.empty((n_steps, B, wl.vocab_size), np.float64)
    for s in range(n_steps):
        toks = [int(streams[b][offsets[b] + s]) for b in range(B)]
        pos = [offsets[b] + s for b in range(B)]
        dec.forward_batch(toks, pos, out[s])
        for b in range(B):
            want[s, b] = ref.forward(toks[b], pos[b], slot=b)
    dec.sync()
    assert dec.kernels_per_step(B) == 5 * wl.n_layers + 2  # the tensor-core path's embedding kernel runs first
    got = out.cpu().numpy()
    for b in range(B):
        check_logits(got[:, b], want[:, b], f"{wl.name} bf16 B={B} slot {b}")
    # not vacuous: the fp32 model is much further away
    full = oracle.Model(wl.config_tuple(), w).decode(streams[0][: n_steps])
    if offsets[0] == 0:
        assert np.abs(got[:, 0] - full).max() > 10 * np.abs(got[:, 0] - want[:, 0]).max()


def test_bf16_prefill_chunks_and_graph_free_path():
    wl = WORKLOADS["mid"]
    w = synth.make_weights(wl)
    rw = rounded_model(w)
    toks = synth.token_stream(wl, 0, 100)
    for flags in (BF16, BF16 | pkg.L2_FLAG_NO_GRAPH):
        ref = oracle.Model(wl.config_tuple(), rw)
        dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), flags=flags)
        out = torch.empty((90, wl.vocab_size), device="cuda")
        dec.prefill(toks[:90], pos0=0, out=out)  # chunks of 64 and 26 rows on the tensor cores
        dec.sync()
        assert dec.position(0) == 90
        check_logits(out.cpu().numpy(), ref.decode(toks[:90]), f"bf16 prefill, flags {flags:#x}")
        step = torch.empty((10, wl.vocab_size), device="cuda")
        for i in range(90, 100):
            dec.forward(int(toks[i]), i, step[i - 90])
        dec.sync()
        check_logits(step.cpu().numpy(), ref.decode(toks[90:100], pos0=90), f"bf16 steps after prefill, flags {flags:#x}")


def test_bf16_prefill_one_token_per_step_without_tensor_cores():
    wl = WORKLOADS["mid"]
    w = synth.make_weights(wl)
    rw = rounded_model(w)
    toks = synth.token_stream(wl, 0, 30)
    for flags in (BF16 | pkg.L2_FLAG_NO_TC, BF16 | pkg.L2_FLAG_NO_TC | pkg.L2_FLAG_NO_GRAPH):
        ref = oracle.Model(wl.config_tuple(), rw)
        dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), flags=flags)
        out = torch.empty((20, wl.vocab_size), device="cuda")
        dec.prefill(toks[:20], pos0=0, out=out)
        dec.sync()
        assert dec.position(0) == 20
        check_logits(out.cpu().numpy(), ref.decode(toks[:20]), f"bf16 prefill, flags {flags:#x}")
        step = torch.empty((10, wl.vocab_size), device="cuda")
        for i in range(20, 30):
            dec.forward(int(toks[i]), i, step[i - 20])
        dec.sync()
        check_logits(step.cpu().numpy(), ref.decode(toks[20:30], pos0=20), f"bf16 steps after prefill, flags {flags:#x}")


def test_bf16_flag_checks():
    wl = WORKLOADS["gqa_small"]
    w = pkg.to_device(synth.make_weights(wl))
    for kw in ({"max_batch": 2, "flags": BF16 | pkg.L2_FLAG_NO_TC}, {"flags": BF16 | pkg.L2_FLAG_PERSIST}):
        with pytest.raises(pkg.L2Error) as e:
            pkg.Decoder(wl.config_tuple(), w, **kw)
        assert e.value.code == pkg.L2_EINVAL
    tiny = WORKLOADS["tiny"]  # hidden_dim 172: not divisible by 8
    with pytest.raises(pkg.L2Error) as e:
        pkg.Decoder(tiny.config_tuple(), pkg.to_device(synth.make_weights(tiny)), flags=BF16)
    assert e.value.code == pkg.L2_EINVAL
