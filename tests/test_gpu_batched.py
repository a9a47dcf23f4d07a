"""Batched steps (B independent sequences, each at its own position) against
the oracle, sequence by sequence.

Each slot b has its own token stream (synth stream 100 + b) and its own KV
cache.  Staggered starting positions are set up by teacher-forcing each slot's
prefix in the oracle and importing that cache (l2_kv_import), then all slots
step together with l2_forward_batch.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import ATT_ABS, check_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402


def run_batched(wl, B, n_steps, offsets, flags=0, weights=None, check_att_every=0):
    w = weights if weights is not None else synth.make_weights(wl)
    ref = oracle.Model(wl.config_tuple(), w, n_slots=B)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=B, flags=flags)
    streams = [synth.token_stream(wl, b, offsets[b] + n_steps) for b in range(B)]
    for b in range(B):
        if offsets[b]:
            ref.decode(streams[b][: offsets[b]], slot=b)
        dec.kv_import(ref.key_cache[b][:, : offsets[b]], ref.value_cache[b][:, : offsets[b]], slot=b)
        assert dec.position(b) == offsets[b]
    out = torch.empty((n_steps, B, wl.vocab_size), device="cuda")
    refs = np.empty((n_steps, B, wl.vocab_size), np.float32)
    for s in range(n_steps):
        toks = [int(streams[b][offsets[b] + s]) for b in range(B)]
        pos = [offsets[b] + s for b in range(B)]
        dec.forward_batch(toks, pos, out[s])
        want_att = check_att_every and s % check_att_every == 0
        for b in range(B):
            if want_att:
                refs[s, b], att = ref.forward(toks[b], pos[b], slot=b, want_att=True)
                dec.sync()
                for layer in range(wl.n_layers):
                    ga = dec.debug_attention(layer, slot=b)
                    assert ga.shape == (wl.n_heads, pos[b] + 1)
                    d = float(np.abs(ga - att[layer, :, : pos[b] + 1]).max())
                    assert d <= ATT_ABS, f"step {s} slot {b} layer {layer}: attention differs by {d:.3e}"
            else:
                refs[s, b] = ref.forward(toks[b], pos[b], slot=b)
    dec.sync()
    got = out.cpu().numpy()
    for b in range(B):
        check_logits(got[:, b], refs[:, b], f"{wl.name} B={B} slot {b}")
    return dec, got, w, streams


@pytest.mark.parametrize("B", [2, 3, 8])
def test_tiny_batched(B):
    wl = WORKLOADS["tiny"]
    offsets = [(b * 37) % 60 for b in range(B)]
    run_batched(wl, B, 24, offsets, flags=pkg.L2_FLAG_DEBUG, check_att_every=6)


def test_gqa_small_batched_staggered():
    wl = WORKLOADS["gqa_small"]
    B = 5
    offsets = [0, 17, 64, 100, 190]
    run_batched(wl, B, 20, offsets, flags=pkg.L2_FLAG_DEBUG, check_att_every=5)


def test_group_of_eight_batched_16():
    # 8 query heads per KV head, head_size 64 (the batched_1b grouping), 16 sequences
    wl = WORKLOADS["batched_1b"].replace(name="g8", dim=512, hidden_dim=1376, n_layers=2, n_heads=8,
                                         n_kv_heads=1, vocab_size=1000, seq_len=256, seed_override=91)
    B = 16
    offsets = [b * 256 // B for b in range(B)]
    run_batched(wl, B, 12, offsets, flags=pkg.L2_FLAG_DEBUG, check_att_every=4)


def test_group_of_four_batched():
    # 4 query heads per KV head, head_size 64: the row-per-lane attention with 2 heads per lane;
    # positions that end mid-way through a 16-row ring stage
    wl = WORKLOADS["batched_1b"].replace(name="g4", dim=512, hidden_dim=1376, n_layers=2, n_heads=8,
                                         n_kv_heads=2, vocab_size=1000, seq_len=256, seed_override=92)
    B = 6
    offsets = [0, 1, 15, 16, 33, 200]
    run_batched(wl, B, 10, offsets, flags=pkg.L2_FLAG_DEBUG, check_att_every=3)


def test_ragged_batched_64():
    wl = WORKLOADS["tiny"].replace(name="ragged64", dim=60, hidden_dim=92, n_layers=2, n_heads=5,
                                   n_kv_heads=2, vocab_size=301, seq_len=96, shared_wcls=False,
                                   seed_override=78, std_scale=(("wq", 8.0), ("wk", 8.0)))
    B = 64
    offsets = [(b * 3) % 80 for b in range(B)]
    run_batched(wl, B, 8, offsets)


def test_slot_results_match_batch_of_one():
    wl = WORKLOADS["gqa_small"]
    B = 4
    offsets = [3, 0, 9, 1]
    _, got, w, streams = run_batched(wl, B, 10, offsets)
    dev_w = pkg.to_device(w)
    for b in (0, 2):
        ref = oracle.Model(wl.config_tuple(), w)
        if offsets[b]:
            ref.decode(streams[b][: offsets[b]])
        one = pkg.Decoder(wl.config_tuple(), dev_w)
        one.kv_import(ref.key_cache[0][:, : offsets[b]], ref.value_cache[0][:, : offsets[b]])
        out = torch.empty((10, wl.vocab_size), device="cuda")
        for s in range(10):
            one.forward(int(streams[b][offsets[b] + s]), offsets[b] + s, out[s])
        one.sync()
        check_logits(got[:, b], out.cpu().numpy(), f"slot {b} vs batch of one")


def test_batched_is_deterministic_and_graph_matches_eager():
    wl = WORKLOADS["gqa_small"]
    w = pkg.to_device(synth.make_weights(wl))
    B = 6
    toks = [synth.token_stream(wl, b, 12) for b in range(B)]

    def run(flags):
        dec = pkg.Decoder(wl.config_tuple(), w, max_batch=B, flags=flags)
        out = torch.empty((12, B, wl.vocab_size), device="cuda")
        for s in range(12):
            dec.forward_batch([int(t[s]) for t in toks], [s] * B, out[s])
        dec.sync()
        return out.cpu().numpy()

    a = run(0)
    assert np.array_equal(a, run(0))
    assert np.array_equal(a, run(pkg.L2_FLAG_NO_GRAPH))
    assert np.array_equal(a, run(pkg.L2_FLAG_NO_PDL))


def test_batch_checks_and_slot_rewind():
    wl = WORKLOADS["tiny"]
    w = pkg.to_device(synth.make_weights(wl))
    dec = pkg.Decoder(wl.config_tuple(), w, max_batch=4)
    with pytest.raises(pkg.L2Error) as e:
        dec.forward_batch([1] * 5, [0] * 5)
    assert e.value.code == pkg.L2_EINVAL
    with pytest.raises(pkg.L2Error) as e:
        dec.forward_batch([1, 2], [0, 1])  # slot 1 has no row 0 yet
    assert e.value.code == pkg.L2_ESTATE
    dec.forward_batch([1, 2, 3], [0, 0, 0])
    dec.forward_batch([1, 2, 3], [1, 1, 1])
    dec.reset(1)
    assert [dec.position(b) for b in range(4)] == [2, 0, 2, 0]
    dec.forward_batch([4, 5, 6], [2, 0, 2])  # slot 1 restarts at position 0
    dec.sync()


def test_launch_op_of_a_batched_step():
    # l2_launch_op_batch reruns one kernel of the last step, whose rows it must match
    wl = WORKLOADS["tiny"]
    w_host = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w_host), max_batch=16)
    B = 16
    toks = [int(t) for t in synth.token_stream(wl, 9, B)]
    out = torch.empty((B, wl.vocab_size), device="cuda")
    dec.forward_batch(toks, [0] * B, out)
    for op in range(6):
        dec.launch_op(op, wl.n_layers - 1, 2, batch=B)
    dec.sync()
    with pytest.raises(pkg.L2Error) as e:
        dec.launch_op(3, 0, 1, batch=8)  # the last step had 16 rows
    assert e.value.code == pkg.L2_ESTATE
    with pytest.raises(pkg.L2Error) as e:
        dec.launch_op(3, 0, 1, batch=65)  # more rows than any step of the handle
    assert e.value.code == pkg.L2_EINVAL
    # a step after the standalone launches is still the oracle's
    ref = oracle.Model(wl.config_tuple(), w_host, n_slots=B)
    want = np.stack([ref.forward(toks[b], 0, slot=b) for b in range(B)])
    dec.forward_batch(toks, [0] * B, out)
    dec.sync()
    check_logits(out.cpu().numpy(), want, "batched step after l2_launch_op_batch")
    dec.close()
