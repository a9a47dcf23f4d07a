"""Failure paths on the GPU, without faulting it.

- A bounded device-side wait that runs out: a kernel waits, with a 1 ms
  limit, on an mbarrier that nothing arrives on (the decode kernels' own wait
  routine), sets the device error word, waits for its bulk copy in flight and
  returns.  l2_sync must report L2_ETIMEOUT once and clear the word; the
  kernel also leaves the attention tickets counted, and the handle's next
  steps, at positions where attention merges several CTAs through those
  tickets, must still match the oracle.
- An injected CUDA graph instantiation failure: the step returns L2_ECUDA
  with nothing run and the position unchanged, the next call builds the graph
  and matches the oracle, and repeated failures leak no device memory.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import check_logits, gpu_decode

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402


def _prefix(wl, n0):
    return synth.kv_rows(wl, 0, n0, "k"), synth.kv_rows(wl, 0, n0, "v")


def test_wait_expiry_reports_timeout_and_handle_recovers():
    wl = WORKLOADS["gqa_small"]
    w_host = synth.make_weights(wl)
    n0, steps = 200, 4  # attention splits each head's 201+ positions over 2 CTAs
    k, v = _prefix(wl, n0)
    toks = synth.token_stream(wl, 0, steps, start=n0)
    ref = oracle.Model(wl.config_tuple(), w_host)
    ref.key_cache[0][:, :n0] = k
    ref.value_cache[0][:, :n0] = v
    want = ref.decode(toks, pos0=n0)

    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w_host))
    dec.kv_import(k, v)
    dec.sync()
    dec.debug_wait_timeout(1000)
    with pytest.raises(pkg.L2Error) as e:
        dec.sync()
    assert e.value.code == pkg.L2_ETIMEOUT
    assert "gave up" in str(e.value)
    dec.sync()  # the word was cleared
    got = gpu_decode(dec, toks, pos0=n0)
    check_logits(got, want, "steps after a wait expiry")
    dec.close()


def test_wait_expiry_argument_checks():
    wl = WORKLOADS["tiny"]
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(synth.make_weights(wl)))
    for bad in (0, -5, 2_000_001):
        with pytest.raises(pkg.L2Error) as e:
            dec.debug_wait_timeout(bad)
        assert e.value.code == pkg.L2_EINVAL
    dec.sync()
    dec.close()


def test_injected_graph_instantiate_failure():
    wl = WORKLOADS["tiny"]
    w_host = synth.make_weights(wl)
    w = pkg.to_device(w_host)
    toks = synth.token_stream(wl, 0, 6)
    want = oracle.Model(wl.config_tuple(), w_host).decode(toks)
    # batch-1 steps of tiny run as one kernel without a graph unless asked for the graph path
    dec = pkg.Decoder(wl.config_tuple(), w, flags=pkg.L2_FLAG_NO_ONE_CTA)
    pkg.fail_graph_at(1)
    with pytest.raises(pkg.L2Error) as e:
        dec.forward(int(toks[0]), 0)
    assert e.value.code == pkg.L2_ECUDA
    assert "injected" in str(e.value)
    assert dec.position() == 0
    got = gpu_decode(dec, toks)  # the graph is built again on this call
    check_logits(got, want, "steps after a failed graph instantiation")
    dec.close()

    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        d = pkg.Decoder(wl.config_tuple(), w, flags=pkg.L2_FLAG_NO_ONE_CTA)
        pkg.fail_graph_at(1)
        with pytest.raises(pkg.L2Error):
            d.forward(int(toks[0]), 0)
        d.close()
    pkg.fail_graph_at(0)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free0 - free1) < 64 << 20
