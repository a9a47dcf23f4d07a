"""l2_forward_static: the decode step for callers that cannot allocate device
memory once decoding has started (for instance a server whose device memory
all belongs to its own pool, or a loop that must not take the implicit
synchronisation of cudaMalloc/cudaFree).  It is called here through the C ABI
and must give the same logits as l2_forward, within the parity tolerance, on
two calls in a row.  This file is collected last on purpose.
"""
import ctypes

import pytest

import synth
from synth import WORKLOADS
from tests.gpu_util import check_logits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402


def test_static_scratch_step_matches_forward_on_two_calls():
    wl = WORKLOADS["gqa_small"]
    w = pkg.to_device(synth.make_weights(wl))
    toks = synth.token_stream(wl, 0, 2)
    lib = pkg.lib()
    ref = pkg.Decoder(wl.config_tuple(), w)
    new = pkg.Decoder(wl.config_tuple(), w)
    out_ref = torch.empty((2, wl.vocab_size), device="cuda")
    out_new = torch.full((2, wl.vocab_size), float("nan"), device="cuda")
    for pos in range(2):
        ref.forward(int(toks[pos]), pos, out_ref[pos])
        rc = lib.l2_forward_static(new.handle, int(toks[pos]), pos,
                                   ctypes.c_void_p(out_new[pos].data_ptr()))
        assert rc == pkg.L2_OK, lib.l2_last_error(new.handle).decode()
    ref.sync()
    new.sync()
    a, b = out_ref.cpu().numpy(), out_new.cpu().numpy()
    for pos in range(2):
        check_logits(b[pos], a[pos], f"l2_forward_static call {pos}")
    ref.close()
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
