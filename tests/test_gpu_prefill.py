"""Prefill (l2_prefill) against the oracle, token by token.

A prompt of T tokens at positions pos0.. of one slot is run as batched steps
of up to 64 rows (max_batch rows with L2_FLAG_DEBUG); every row's logits must equal (within the parity
bounds) the oracle's logits for that token at that position after the
tokens before it, i.e. the oracle's teacher-forced decode of the same
stream.  Covered: one chunk, several chunks with a ragged last one, a
one-token chunk (the batch-1 kernels writing a slot other than 0), a slot
other than 0 while slot 0 keeps decoding, 8 query heads per KV head, 64-row
chunks, the cache rows written, ordinary steps after a prefill, argument
checks, a one-sequence handle, ordinary steps after a prefill on a handle
running batch-1 steps as the persistent kernel, and shapes whose chunks run
the prompt-chunk attention kernel (head sizes 64 and 128).
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

G8 = WORKLOADS["batched_1b"].replace(name="g8p", dim=512, hidden_dim=1376, n_layers=2, n_heads=8, n_kv_heads=1,
                                     vocab_size=1000, seq_len=256, seed_override=93)


def run_plan(wl, max_batch, plan, slot=0, flags=0, then_steps=0):
    w = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=max_batch, flags=flags)
    ref = oracle.Model(wl.config_tuple(), w, n_slots=max_batch)
    toks = synth.token_stream(wl, slot, sum(plan) + then_steps)
    pos = 0
    for n in plan:
        out = torch.empty((n, wl.vocab_size), device="cuda")
        dec.prefill(toks[pos:pos + n], pos0=pos, slot=slot, out=out)
        dec.sync()
        want = ref.decode(toks[pos:pos + n], pos0=pos, slot=slot)
        check_logits(out.cpu().numpy(), want, f"{wl.name} prefill slot {slot} rows {pos}..{pos + n - 1}")
        pos += n
    assert dec.position(slot) == pos
    for layer in (0, wl.n_layers - 1):
        k, v = dec.kv_export(layer, n_pos=pos, slot=slot)
        # cache rows: 1e-4 relative to their magnitude (their scale grows with the model width)
        for got, want in ((k, ref.key_cache[slot][layer, :pos]), (v, ref.value_cache[slot][layer, :pos])):
            assert np.abs(got - want).max() <= 1e-4 * max(1.0, float(np.abs(want).max()))
    if then_steps:
        assert slot == 0
        out = torch.empty((then_steps, wl.vocab_size), device="cuda")
        for i in range(then_steps):
            dec.forward(int(toks[pos + i]), pos + i, out[i])
        dec.sync()
        check_logits(out.cpu().numpy(), ref.decode(toks[pos:pos + then_steps], pos0=pos, slot=0),
                     f"{wl.name} steps after prefill")
    return dec, ref


def test_prefill_several_chunks_then_decode():
    # 100 tokens: chunks of 64 and 36 rows on a handle of 2 sequences
    run_plan(WORKLOADS["gqa_small"], 2, [100], then_steps=5)


def test_prefill_on_a_one_sequence_handle_and_with_debug_export():
    run_plan(WORKLOADS["mid"], 1, [70, 3], then_steps=3)
    # with L2_FLAG_DEBUG the chunks are max_batch rows: 4 + 4 + 2
    run_plan(WORKLOADS["tiny"], 4, [10], flags=pkg.L2_FLAG_DEBUG, then_steps=2)


def test_prefill_in_pieces_and_a_single_token_in_slot_3():
    run_plan(WORKLOADS["tiny"], 8, [5, 1, 20, 1], slot=3)


def test_prefill_leaves_other_slots_alone():
    wl = WORKLOADS["tiny"]
    w = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w), max_batch=4)
    ref = oracle.Model(wl.config_tuple(), w, n_slots=4)
    s0 = synth.token_stream(wl, 0, 30)
    s2 = synth.token_stream(wl, 2, 12)
    out = torch.empty((30, wl.vocab_size), device="cuda")
    for i in range(15):
        dec.forward(int(s0[i]), i, out[i])
    dec.prefill(s2, pos0=0, slot=2)
    for i in range(15, 30):
        dec.forward(int(s0[i]), i, out[i])
    dec.sync()
    check_logits(out.cpu().numpy(), ref.decode(s0, slot=0), "slot 0 around a prefill of slot 2")
    assert dec.position(2) == 12 and dec.position(0) == 30


def test_prefill_group_of_eight():
    run_plan(G8, 16, [16, 9, 30])


def test_prefill_64_row_chunks():
    run_plan(WORKLOADS["mid"], 64, [64, 64, 10])


# Shapes whose 64-row chunks take the prompt-chunk attention kernel (attn_prefill.cu: at most two
# query heads per KV head and enough CTAs): 32 KV heads of 64, and 16 KV heads of 128 with two
# query heads each.  The ragged last chunk goes through the per-row kernel.
MHA64 = WORKLOADS["mid"].replace(name="mha64", dim=2048, hidden_dim=512, n_layers=2, n_heads=32, n_kv_heads=32,
                                 vocab_size=700, seq_len=256, seed_override=95)
GQA2_128 = WORKLOADS["mid"].replace(name="gqa2_128", dim=4096, hidden_dim=512, n_layers=2, n_heads=32, n_kv_heads=16,
                                    vocab_size=700, seq_len=192, seed_override=96)


@pytest.mark.parametrize("wl", [MHA64, GQA2_128], ids=["mha_hs64", "gqa2_hs128"])
def test_prefill_chunk_attention_kernel(wl):
    run_plan(wl, 1, [64, 64, 21], then_steps=3)


def test_prefill_then_persistent_steps():
    run_plan(WORKLOADS["tiny"], 1, [7, 3], flags=pkg.L2_FLAG_PERSIST, then_steps=4)


def test_prefill_argument_checks():
    wl = WORKLOADS["tiny"]
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(synth.make_weights(wl)), max_batch=4)
    toks = synth.token_stream(wl, 0, 8)
    with pytest.raises(pkg.L2Error) as e:
        dec.prefill(toks, pos0=3)  # rows 0..2 do not exist
    assert e.value.code == pkg.L2_ESTATE
    with pytest.raises(pkg.L2Error) as e:
        dec.prefill(toks, pos0=wl.seq_len - 4)
    assert e.value.code == pkg.L2_EINVAL
    with pytest.raises(pkg.L2Error) as e:
        dec.prefill(np.array([1, wl.vocab_size], np.int32))
    assert e.value.code == pkg.L2_EINVAL
    with pytest.raises(pkg.L2Error) as e:
        dec.prefill(toks, slot=4)
    assert e.value.code == pkg.L2_EINVAL
    assert dec.position(0) == 0  # nothing was enqueued
