"""bf16 weight streaming (L2_FLAG_BF16_WEIGHTS) against the oracle on the same
bf16-rounded matrices.

The handle converts its matrices to bf16 and keeps everything else fp32, so it
computes the model whose matrices are the bf16-rounded ones; the oracle runs
that model (tests/bf16.py rounds the matrices on the host, independently of the
device conversion), and the per-step logit bounds are the fp32 ones.  Also:
prompts go one token per step, the flag's argument checks, and that the
rounding changes the result (so the comparison is not vacuous).
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


def test_bf16_prefill_one_token_per_step_and_graph_free_path():
    wl = WORKLOADS["mid"]
    w = synth.make_weights(wl)
    rw = rounded_model(w)
    toks = synth.token_stream(wl, 0, 30)
    for flags in (BF16, BF16 | pkg.L2_FLAG_NO_GRAPH):
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
    for kw in ({"max_batch": 2, "flags": BF16}, {"flags": BF16 | pkg.L2_FLAG_PERSIST}):
        with pytest.raises(pkg.L2Error) as e:
            pkg.Decoder(wl.config_tuple(), w, **kw)
        assert e.value.code == pkg.L2_EINVAL
    tiny = WORKLOADS["tiny"]  # hidden_dim 172: not divisible by 8
    with pytest.raises(pkg.L2Error) as e:
        pkg.Decoder(tiny.config_tuple(), pkg.to_device(synth.make_weights(tiny)), flags=BF16)
    assert e.value.code == pkg.L2_EINVAL
