"""l2_forward_static: the decode step for callers that cannot allocate device
memory once decoding has started (for instance a server whose device memory
all belongs to its own pool, or a loop that must not take the implicit
synchronisation of cudaMalloc/cudaFree).  It is called here through the C ABI
and must give the same logits as l2_forward, within the parity tolerance, on
consecutive calls; at positions where the attention kernel splits the cache
over several CTAs (so its partial results and tickets go through the static
array) it is also checked against the oracle.  This file is collected last on
purpose.
"""
import ctypes

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


def _static_step(dec, token, pos, out):
    lib = pkg.lib()
    rc = lib.l2_forward_static(dec.handle, int(token), int(pos), ctypes.c_void_p(out.data_ptr()))
    assert rc == pkg.L2_OK, lib.l2_last_error(dec.handle).decode()


def test_static_scratch_step_matches_forward_on_two_calls():
    wl = WORKLOADS["gqa_small"]
    w = pkg.to_device(synth.make_weights(wl))
    toks = synth.token_stream(wl, 0, 2)
    ref = pkg.Decoder(wl.config_tuple(), w)
    new = pkg.Decoder(wl.config_tuple(), w)
    out_ref = torch.empty((2, wl.vocab_size), device="cuda")
    out_new = torch.full((2, wl.vocab_size), float("nan"), device="cuda")
    for pos in range(2):
        ref.forward(int(toks[pos]), pos, out_ref[pos])
        _static_step(new, toks[pos], pos, out_new[pos])
    ref.sync()
    new.sync()
    a, b = out_ref.cpu().numpy(), out_new.cpu().numpy()
    for pos in range(2):
        check_logits(b[pos], a[pos], f"l2_forward_static call {pos}")
    ref.close()
    new.close()


# (workload, cache rows imported before the first step, steps).  At batch 1
# an attention CTA takes at least 128 positions and a KV head gets at most
# ceil(seq_len / 128) CTAs (fewer only if 152 SMs could not hold one per
# chunk, which these shapes do not reach): gqa_small at positions 200.. splits
# each head's cache over 2 CTAs, mid at 600.. over 5.  Each workload steps
# several times in a row, and mid runs after gqa_small has left its own
# partial results and tickets in the array.
MULTI_CHUNK = [("gqa_small", 200, 6), ("mid", 600, 4)]


def test_static_scratch_multi_chunk_matches_oracle_and_forward():
    for name, n0, steps in MULTI_CHUNK:
        wl = WORKLOADS[name]
        w_host = synth.make_weights(wl)
        w = pkg.to_device(w_host)
        k = synth.kv_rows(wl, 0, n0, "k")
        v = synth.kv_rows(wl, 0, n0, "v")
        toks = synth.token_stream(wl, 0, steps, start=n0)

        ref = oracle.Model(wl.config_tuple(), w_host)
        ref.key_cache[0][:, :n0] = k
        ref.value_cache[0][:, :n0] = v
        want = ref.decode(toks, pos0=n0)

        fwd = pkg.Decoder(wl.config_tuple(), w)
        new = pkg.Decoder(wl.config_tuple(), w)
        fwd.kv_import(k, v)
        new.kv_import(k, v)
        out_fwd = torch.empty((steps, wl.vocab_size), device="cuda")
        out_new = torch.full((steps, wl.vocab_size), float("nan"), device="cuda")
        for i, tok in enumerate(toks):
            fwd.forward(int(tok), n0 + i, out_fwd[i])
            _static_step(new, tok, n0 + i, out_new[i])
        fwd.sync()
        new.sync()
        got, base = out_new.cpu().numpy(), out_fwd.cpu().numpy()
        check_logits(got, want, f"{name} l2_forward_static against the oracle")
        check_logits(got, base.astype(np.float64), f"{name} l2_forward_static against l2_forward")
        assert new.position() == n0 + steps
        fwd.close()
        new.close()


def test_static_scratch_limit_is_enforced():
    # 32 heads of 128 on 4 KV heads with a 16384-position cache need more
    # attention scratch than the 131072 floats of the static array (on 152
    # SMs with one attention CTA per SM: 32 * 38 * 130 + 4 = 158084 floats).
    cfg = (4096, 16, 1, 32, 4, 16, 16384)
    wl = WORKLOADS["tiny"].replace(dim=4096, hidden_dim=16, n_layers=1, n_heads=32, n_kv_heads=4,
                                   vocab_size=16, seq_len=16384, shared_wcls=False)
    w = {k: torch.zeros(wl.shape(k), device="cuda") for k in wl.tensor_names()}
    dec = pkg.Decoder(cfg, w)
    lib = pkg.lib()
    rc = lib.l2_forward_static(dec.handle, 0, 0, None)
    assert rc == pkg.L2_EINVAL
    assert b"static array" in lib.l2_last_error(dec.handle)
    assert dec.position() == 0  # nothing was enqueued
    dec.close()
