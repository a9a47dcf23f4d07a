"""The persistent batch-1 step kernel (L2_FLAG_PERSIST: one cooperative
launch per step) against the oracle, and against the default
one-kernel-per-matmul path.

Every small workload is checked at every teacher-forced step with the logit
bounds of the parity tests; the ragged shape (dim 60, head size 12, vocab
301) and a long cache (mid: 1024 positions, up to 8 attention chunks per KV
head merged by tickets) are included.  Cache rows written by the persistent
path are compared with the oracle's rows.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import check_logits, decoder_for, gpu_decode

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402

RAGGED = WORKLOADS["tiny"].replace(name="ragged", dim=60, hidden_dim=92, n_layers=3, n_heads=5, n_kv_heads=5,
                                   vocab_size=301, seq_len=40, shared_wcls=False, seed_override=77)
GQA_RAGGED = WORKLOADS["tiny"].replace(name="gqa_ragged", dim=96, hidden_dim=100, n_layers=2, n_heads=8,
                                       n_kv_heads=2, vocab_size=77, seq_len=300, shared_wcls=False, seed_override=79)


def persistent(wl, w):
    dec = decoder_for(wl, w, flags=pkg.L2_FLAG_PERSIST)
    assert dec.kernels_per_step() == 1, "the persistent step kernel is not in use"
    return dec


@pytest.mark.parametrize("name", ["tiny", "gqa_small", "mid", "ragged", "gqa_ragged"])
def test_persistent_matches_oracle(name):
    wl = {"ragged": RAGGED, "gqa_ragged": GQA_RAGGED}.get(name) or WORKLOADS[name]
    n = wl.seq_len if wl.seq_len <= 300 else 300
    w = synth.make_weights(wl)
    toks = synth.token_stream(wl, 0, n)
    ref = oracle.Model(wl.config_tuple(), w)
    want = ref.decode(toks)
    dec = persistent(wl, pkg.to_device(w))
    got = gpu_decode(dec, toks)
    rel = check_logits(got, want, f"{name} persistent")
    # the cache rows the kernel wrote are the oracle's (RoPE'd keys, values)
    for layer in (0, wl.n_layers - 1):
        k, v = dec.kv_export(layer, n_pos=n)
        kd = np.abs(k - ref.key_cache[0][layer, :n]).max()
        vd = np.abs(v - ref.value_cache[0][layer, :n]).max()
        assert kd <= 1e-4 and vd <= 1e-4, f"{name} layer {layer}: cache rows differ by {kd:.2e} / {vd:.2e}"
    print(f"{name}: persistent, worst relative logit error {rel:.2e}")


def test_mid_long_cache_persistent():
    # positions up to 1023: up to 8 chunks per KV head at the end
    wl = WORKLOADS["mid"]
    w = synth.make_weights(wl)
    toks = synth.token_stream(wl, 0, wl.seq_len)
    dec = persistent(wl, pkg.to_device(w))
    ref = oracle.Model(wl.config_tuple(), w)
    samples = (299, 511, 767, 1023)
    out = torch.empty(wl.vocab_size, device="cuda")
    got = {}
    for p in range(wl.seq_len):
        dec.forward(int(toks[p]), p, out)
        if p in samples:
            dec.sync()
            got[p] = out.cpu().numpy()
    for l in range(wl.n_layers):
        k, v = dec.kv_export(l, n_pos=max(samples))
        ref.key_cache[0][l, : max(samples)] = k
        ref.value_cache[0][l, : max(samples)] = v
    for p in samples:
        check_logits(got[p], ref.forward(int(toks[p]), p), f"mid pos {p} persistent")


@pytest.mark.parametrize("name", ["gqa_small", "ragged"])
def test_persistent_and_per_kernel_paths_agree(name):
    wl = RAGGED if name == "ragged" else WORKLOADS[name]
    w = pkg.to_device(synth.make_weights(wl))
    toks = synth.token_stream(wl, 0, 24)
    a = gpu_decode(persistent(wl, w), toks)
    multi = decoder_for(wl, w, flags=pkg.L2_FLAG_NO_ONE_CTA)  # the graph of per-matrix kernels
    assert multi.kernels_per_step() == 5 * wl.n_layers + 1
    b = gpu_decode(multi, toks)
    check_logits(a, b.astype(np.float64), f"{name}: persistent vs one kernel per matmul")


def test_persistent_is_deterministic_and_resumes():
    wl = WORKLOADS["gqa_small"]
    w = pkg.to_device(synth.make_weights(wl))
    toks = synth.token_stream(wl, 0, 40)
    a = gpu_decode(persistent(wl, w), toks)
    assert np.array_equal(a, gpu_decode(persistent(wl, w), toks))
    # rewind to position 20 and replay: the same logits
    dec = persistent(wl, w)
    gpu_decode(dec, toks[:30])
    assert np.array_equal(a[20:], gpu_decode(dec, toks[20:], pos0=20))
    # a cache imported from the oracle's rows continues like the oracle
    wh = synth.make_weights(wl)
    ref = oracle.Model(wl.config_tuple(), wh)
    ref.decode(toks[:25])
    dec = persistent(wl, w)
    dec.kv_import(ref.key_cache[0][:, :25], ref.value_cache[0][:, :25])
    assert dec.position() == 25
    check_logits(gpu_decode(dec, toks[25:], pos0=25), ref.decode(toks[25:], pos0=25), "gqa_small after import")


def test_persistent_host_entry_point():
    wl = WORKLOADS["tiny"]
    w = synth.make_weights(wl)
    toks = synth.token_stream(wl, 0, 12)
    dec = persistent(wl, pkg.to_device(w))
    got = np.stack([dec.forward_host(int(t), i) for i, t in enumerate(toks)])
    check_logits(got, oracle.Model(wl.config_tuple(), w).decode(toks), "tiny forward_host persistent")
