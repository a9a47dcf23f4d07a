"""Parity at the full workload sizes, in the launch configuration bench.py
times (CUDA graph + programmatic dependent launch), and for the 7B shape also
with the opt-in persistent step kernel.

7B shape: the first 8 teacher-forced steps against the oracle, then one run
to position 4095 whose steps at positions {255, 1023, 2047, 4095} are each
recomputed by the oracle from the same cache rows (exported from the GPU run),
with the attention probabilities of layers {0, 15, 31}.
batched_1b: batch of 1 for 8 steps; batches of 16 and 64 at staggered
positions over synthetic cache prefixes, slots {0, B/2, B-1} checked.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import ATT_ABS, check_logits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402


@pytest.fixture(scope="module")
def llama7b():
    wl = WORKLOADS["llama2_7b"]
    w = synth.make_weights(wl)
    dev = pkg.to_device(w)
    yield wl, w, dev
    del dev
    torch.cuda.empty_cache()


def test_llama7b_first_steps(llama7b):
    wl, w, dev = llama7b
    toks = synth.token_stream(wl, 0, 8)
    dec = pkg.Decoder(wl.config_tuple(), dev)
    out = torch.empty((8, wl.vocab_size), device="cuda")
    for t in range(8):
        dec.forward(int(toks[t]), t, out[t])
    dec.sync()
    ref = oracle.Model(wl.config_tuple(), w).decode(toks)
    rel = check_logits(out.cpu().numpy(), ref, "llama2_7b steps 0..7")
    print(f"llama2_7b steps 0..7: worst relative logit error {rel:.2e}")
    dec.close()


@pytest.mark.parametrize("path", ["per_kernel_debug", "persistent"])
def test_llama7b_sampled_positions(llama7b, path):
    # per_kernel_debug: one kernel per matmul (the path bench.py times) with
    # the attention probabilities exported; persistent: the opt-in persistent
    # step kernel (logits)
    wl, w, dev = llama7b
    samples = (255, 1023, 2047, 4095)
    debug = path == "per_kernel_debug"
    layers = (0, 15, 31) if debug else ()
    toks = synth.token_stream(wl, 0, wl.seq_len)
    dec = pkg.Decoder(wl.config_tuple(), dev, flags=pkg.L2_FLAG_DEBUG if debug else pkg.L2_FLAG_PERSIST)
    assert (dec.kernels_per_step() == 1) == (not debug)
    out = torch.empty(wl.vocab_size, device="cuda")
    got, att = {}, {}
    for p in range(wl.seq_len):
        dec.forward(int(toks[p]), p, out)
        if p in samples:
            dec.sync()
            got[p] = out.cpu().numpy()
            att[p] = {l: dec.debug_attention(l) for l in layers}
    ref = oracle.Model(wl.config_tuple(), w)
    for l in range(wl.n_layers):
        k, v = dec.kv_export(l, n_pos=max(samples))
        ref.key_cache[0][l, : max(samples)] = k
        ref.value_cache[0][l, : max(samples)] = v
    for p in samples:
        # the oracle's cache rows 0..p-1 are the GPU run's; row p is recomputed
        r, ra = ref.forward(int(toks[p]), p, want_att=True)
        rel = check_logits(got[p], r, f"llama2_7b pos {p} ({path})")
        for l in layers:
            d = float(np.abs(att[p][l] - ra[l, :, : p + 1]).max())
            assert d <= ATT_ABS, f"pos {p} layer {l}: attention differs by {d:.3e}"
        print(f"llama2_7b pos {p}: worst relative logit error {rel:.2e}")
    dec.close()


@pytest.fixture(scope="module")
def batched1b():
    wl = WORKLOADS["batched_1b"]
    w = synth.make_weights(wl)
    dev = pkg.to_device(w)
    yield wl, w, dev
    del dev
    torch.cuda.empty_cache()


def test_batched1b_batch_of_one(batched1b):
    wl, w, dev = batched1b
    toks = synth.token_stream(wl, 0, 8)
    dec = pkg.Decoder(wl.config_tuple(), dev)
    out = torch.empty((8, wl.vocab_size), device="cuda")
    for t in range(8):
        dec.forward(int(toks[t]), t, out[t])
    dec.sync()
    check_logits(out.cpu().numpy(), oracle.Model(wl.config_tuple(), w).decode(toks), "batched_1b B=1")
    dec.close()


@pytest.mark.parametrize("B", [16, 64])
def test_batched1b_staggered(batched1b, B):
    wl, w, dev = batched1b
    offsets = [b * wl.seq_len // B for b in range(B)]
    n_steps = 3
    dec = pkg.Decoder(wl.config_tuple(), dev, max_batch=B, flags=pkg.L2_FLAG_DEBUG)
    check = (0, B // 2, B - 1)
    ref = oracle.Model(wl.config_tuple(), w, n_slots=B)
    streams = [synth.token_stream(wl, b, offsets[b] + n_steps) for b in range(B)]
    for b in range(B):
        k = synth.kv_rows(wl, b, offsets[b], "k")
        v = synth.kv_rows(wl, b, offsets[b], "v")
        dec.kv_import(k, v, slot=b)
        if b in check:
            ref.key_cache[b][:, : offsets[b]] = k
            ref.value_cache[b][:, : offsets[b]] = v
    out = torch.empty((n_steps, B, wl.vocab_size), device="cuda")
    for s in range(n_steps):
        dec.forward_batch([int(streams[b][offsets[b] + s]) for b in range(B)],
                          [offsets[b] + s for b in range(B)], out[s])
        if s == n_steps - 1:
            dec.sync()
            gatt = {b: {l: dec.debug_attention(l, slot=b) for l in (0, wl.n_layers - 1)} for b in check}
    dec.sync()
    got = out.cpu().numpy()
    for b in check:
        refs, ra = [], None
        for s in range(n_steps):
            tok, pos = int(streams[b][offsets[b] + s]), offsets[b] + s
            if s == n_steps - 1:
                r, ra = ref.forward(tok, pos, slot=b, want_att=True)
            else:
                r = ref.forward(tok, pos, slot=b)
            refs.append(r)
        check_logits(got[:, b], np.stack(refs), f"batched_1b B={B} slot {b}")
        P = offsets[b] + n_steps
        for l in (0, wl.n_layers - 1):
            d = float(np.abs(gatt[b][l] - ra[l, :, :P]).max())
            assert d <= ATT_ABS, f"B={B} slot {b} layer {l}: attention differs by {d:.3e}"
    dec.close()
