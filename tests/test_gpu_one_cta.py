"""The one-block step kernel (batch-1 steps of models with at most 4 MiB of
weights) against the oracle: logits at the parity bounds, probabilities
within 1e-5, on shapes that exercise its index arithmetic -- grouped heads
that do not divide evenly (6 query heads on 4 KV heads), head sizes of 8
and 12 (attention inside one warp per head) and 32 (three block-wide
phases), contexts long enough that a head's positions take many turns of a
warp, and hidden sizes that are not a multiple of 32 words.  Also: which
models it serves, the device-token and host-output entry points on it,
bitwise repeatability, and the cache rows it writes."""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import ATT_ABS, check_logits, gpu_decode

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402

GQA64 = WORKLOADS["tiny"].replace(name="gqa6on4", dim=48, hidden_dim=132, n_layers=2, n_heads=6, n_kv_heads=4,
                                  vocab_size=203, seq_len=300, shared_wcls=False, seed_override=91)
# head size 32: the attention runs as three block-wide phases instead of one warp per head
HS32 = WORKLOADS["tiny"].replace(name="hs32", dim=128, hidden_dim=344, n_layers=2, n_heads=4, n_kv_heads=2,
                                 vocab_size=700, seq_len=130, shared_wcls=False, seed_override=93,
                                 std_scale=(("wq", 4.0), ("wk", 4.0)))
HS12 = WORKLOADS["tiny"].replace(name="hs12", dim=96, hidden_dim=256, n_layers=3, n_heads=8, n_kv_heads=2,
                                 vocab_size=1000, seq_len=160, shared_wcls=False, seed_override=92,
                                 std_scale=(("wq", 6.0), ("wk", 6.0)))


def _decode_checked(wl, n_steps, att_every):
    w = synth.make_weights(wl)
    toks = synth.token_stream(wl, 0, n_steps)
    ref = oracle.Model(wl.config_tuple(), w)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), flags=pkg.L2_FLAG_DEBUG)
    assert dec.kernels_per_step() == 1, "the shape should run as one block"
    out = torch.empty((n_steps, wl.vocab_size), device="cuda")
    want = np.empty((n_steps, wl.vocab_size), np.float32)
    for t, tok in enumerate(toks):
        dec.forward(int(tok), t, out[t])
        if t % att_every == 0 or t == n_steps - 1:
            want[t], att = ref.forward(int(tok), t, want_att=True)
            dec.sync()
            for layer in range(wl.n_layers):
                d = float(np.abs(dec.debug_attention(layer) - att[layer, :, : t + 1]).max())
                assert d <= ATT_ABS, f"{wl.name} step {t} layer {layer}: attention differs by {d:.3e}"
        else:
            want[t] = ref.forward(int(tok), t)
    dec.sync()
    check_logits(out.cpu().numpy(), want, wl.name)
    return dec, ref


@pytest.mark.parametrize("wl,n_steps,att_every", [(GQA64, 300, 23), (HS12, 160, 17), (HS32, 130, 11)],
                         ids=["gqa6on4", "hs12", "hs32"])
def test_matches_oracle_to_the_end_of_the_context(wl, n_steps, att_every):
    dec, ref = _decode_checked(wl, n_steps, att_every)
    # the cache rows it wrote, in the pages' layout
    for layer in (0, wl.n_layers - 1):
        k, v = dec.kv_export(layer)
        rk, rv = ref.key_cache[0][layer, :n_steps], ref.value_cache[0][layer, :n_steps]
        assert np.abs(k - rk).max() <= 1e-4 * max(1.0, np.abs(rk).max())
        assert np.abs(v - rv).max() <= 1e-4 * max(1.0, np.abs(rv).max())
    dec.close()


def test_which_models_run_as_one_block():
    for name, one in (("tiny", True), ("gqa_small", False), ("mid", False)):
        wl = WORKLOADS[name]
        w = pkg.to_device(synth.make_weights(wl))
        for flags, want in ((0, one), (pkg.L2_FLAG_NO_ONE_CTA, False), (pkg.L2_FLAG_PERSIST, False)):
            dec = pkg.Decoder(wl.config_tuple(), w, flags=flags)
            k = dec.kernels_per_step()
            if want:
                assert k == 1, (name, flags)
            elif not flags & pkg.L2_FLAG_PERSIST:
                assert k == 5 * wl.n_layers + 1, (name, flags, k)
            dec.close()


def test_repeatable_and_host_output_and_device_tokens():
    wl = WORKLOADS["tiny"]
    w_host = synth.make_weights(wl)
    w = pkg.to_device(w_host)
    toks = synth.token_stream(wl, 3, 40)
    a = gpu_decode(pkg.Decoder(wl.config_tuple(), w), toks)
    b = gpu_decode(pkg.Decoder(wl.config_tuple(), w), toks)
    assert np.array_equal(a, b)
    # host output, one call per step
    dec = pkg.Decoder(wl.config_tuple(), w)
    host = np.stack([dec.forward_host(int(t), i).copy() for i, t in enumerate(toks)])
    assert np.array_equal(host, a)
    dec.close()
    # tokens read from device memory when the step runs
    dec = pkg.Decoder(wl.config_tuple(), w)
    tok_dev = torch.tensor([int(t) for t in toks], dtype=torch.int32, device="cuda")
    out = torch.empty((len(toks), wl.vocab_size), device="cuda")
    for i in range(len(toks)):
        dec.forward_dev_tokens(tok_dev[i:i + 1], [i], out[i:i + 1])
    dec.sync()
    assert np.array_equal(out.cpu().numpy(), a)
    dec.close()
    want = oracle.Model(wl.config_tuple(), w_host).decode(toks)
    check_logits(a, want, "tiny, one block")
