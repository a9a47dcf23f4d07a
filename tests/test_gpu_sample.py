"""The device sampler (l2_sample) against the sampler oracle, bit for bit.

Inputs are seeded synthetic logits (numpy generators in this file); for each
configuration both sides start from the same generator states and run
several rounds, and the sampled tokens and the advanced states must be equal
exactly (integer results).  Coverage: vocab sizes 1..49152 (the kernel's
limit), batches of 1..64, temperature 0 (argmax, no draw) and 0.3..1.7,
top-p off, 0.5, 0.9, 0.999 and a tiny topp, heavily tied logits, logits far
beyond the exponential's cut-off, equal logits (a closed form).

End to end: a greedy generation loop run on the GPU (decode step + device
argmax, the token of step t+1 read back from the device) reproduces the
oracle's own greedy generation, the two sequences compared token by token
while the oracle's top-two logit margin exceeds the logit tolerance.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.gpu_util import LOGIT_ABS

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402


def run_both(logits: np.ndarray, temperature: float, topp: float, states: np.ndarray, rounds: int):
    B, V = logits.shape
    dev_logits = torch.from_numpy(logits).cuda()
    dev_states = torch.from_numpy(states.view(np.int64).copy()).cuda()
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    ref_states = [int(s) for s in states]
    for rnd in range(rounds):
        pkg.sample(dev_logits, temperature, topp, dev_states, out)
        got = out.cpu().numpy()
        got_states = dev_states.cpu().numpy().view(np.uint64)
        for b in range(B):
            idx, ref_states[b], _, _ = oracle.sample(logits[b], temperature, topp, ref_states[b])
            assert got[b] == idx, (f"round {rnd} row {b}: device {got[b]} oracle {idx} "
                                   f"(V={V} T={temperature} topp={topp})")
            assert int(got_states[b]) == ref_states[b]
    return got


def seeded_states(B, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(1, 2**63, size=B, dtype=np.int64).astype(np.uint64) * np.uint64(2) + np.uint64(1))


@pytest.mark.parametrize("V", [1, 7, 512, 32000, 49152])
@pytest.mark.parametrize("temperature", [0.0, 0.3, 1.0, 1.7])
@pytest.mark.parametrize("topp", [0.0, 0.5, 0.9, 0.999])
def test_sampler_matches_oracle(V, temperature, topp):
    B = 3 if V >= 32000 else 8
    rng = np.random.default_rng(V * 131 + int(temperature * 10) * 7 + int(topp * 1000))
    logits = (rng.standard_normal((B, V)) * 2.5).astype(np.float32)
    run_both(logits, temperature, topp, seeded_states(B, V), rounds=4 if V >= 32000 else 10)


def test_batch_of_64_and_tied_logits():
    rng = np.random.default_rng(5)
    B, V = 64, 4096
    logits = np.round(rng.standard_normal((B, V)) * 2.0).astype(np.float32)  # values -6..6: heavy ties
    for topp in (0.0, 0.3, 0.8):
        run_both(logits, 1.0, topp, seeded_states(B, 9), rounds=3)
    run_both(logits, 0.0, 0.9, seeded_states(B, 10), rounds=1)


def test_extreme_logits_and_tiny_topp():
    rng = np.random.default_rng(6)
    B, V = 6, 32000
    logits = (rng.standard_normal((B, V)) * 40.0).astype(np.float32)  # most weights below the cut-off
    logits[1] = 0.0
    logits[2, :] = -1e4
    logits[2, 123] = 1e4
    for topp in (0.0, 1e-6, 0.5, 0.95):
        run_both(logits, 1.0, topp, seeded_states(B, 11), rounds=3)
        run_both(logits, 0.05, topp, seeded_states(B, 12), rounds=2)


def test_equal_logits_closed_form_on_device():
    B, V = 16, 32000
    states = seeded_states(B, 13)
    got = run_both(np.zeros((B, V), np.float32), 1.0, 0.0, states, rounds=1)
    for b in range(B):
        k24 = oracle.random_u32(int(states[b]))[0] >> 8
        assert got[b] == (k24 * V) >> 24


def test_greedy_generation_loop_on_device():
    wl = WORKLOADS["gqa_small"]
    w = synth.make_weights(wl)
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(w))
    ref = oracle.Model(wl.config_tuple(), w)
    st = torch.zeros(1, dtype=torch.int64, device="cuda") + 1
    out = torch.empty(wl.vocab_size, device="cuda")
    tok_dev = torch.empty(1, dtype=torch.int32, device="cuda")
    tok_gpu, tok_ref = 1, 1
    n = 48
    for pos in range(n):
        dec.forward(tok_gpu, pos, out)
        pkg.sample(out, 0.0, 0.0, st, tok_dev, stream=dec.stream)
        r = ref.forward(tok_ref, pos)
        top2 = np.sort(r)[-2:]
        tok_ref = int(np.argmax(r))
        dec.sync()
        tok_gpu = int(tok_dev.cpu()[0])
        if top2[1] - top2[0] > LOGIT_ABS:
            assert tok_gpu == tok_ref, f"pos {pos}: device {tok_gpu}, oracle {tok_ref}"
        else:  # a near tie: both continuations are valid; stop comparing
            break
    assert pos >= 8, "the generation ended in a near tie too early to be a test"


def test_device_resident_generation_loop():
    """forward (token read from device memory) -> l2_sample -> forward ...,
    with no host round trip inside the loop; greedy: the oracle's own greedy
    sequence (compared while its top-two margin exceeds the logit tolerance);
    temperature 0.8, top-p 0.9: the same tokens as the host-driven loop."""
    wl = WORKLOADS["gqa_small"]
    w = synth.make_weights(wl)
    dw = pkg.to_device(w)
    n = 40

    def device_loop(temperature, topp):
        dec = pkg.Decoder(wl.config_tuple(), dw)
        seq = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
        seq[0] = 1
        st = torch.tensor([0x9E3779B97F4A7C15 & (2**63 - 1)], dtype=torch.int64, device="cuda")
        out = torch.empty(wl.vocab_size, device="cuda")
        torch.cuda.synchronize()
        for pos in range(n):
            dec.forward_dev_tokens(seq[pos:pos + 1], pos, out)
            pkg.sample(out, temperature, topp, st, seq[pos + 1:pos + 2], stream=dec.stream)
        dec.sync()
        return seq.cpu().numpy()

    def host_loop(temperature, topp):
        dec = pkg.Decoder(wl.config_tuple(), dw)
        st = torch.tensor([0x9E3779B97F4A7C15 & (2**63 - 1)], dtype=torch.int64, device="cuda")
        out = torch.empty(wl.vocab_size, device="cuda")
        nxt = torch.empty(1, dtype=torch.int32, device="cuda")
        toks = [1]
        for pos in range(n):
            dec.forward(toks[-1], pos, out)
            pkg.sample(out, temperature, topp, st, nxt, stream=dec.stream)
            dec.sync()
            toks.append(int(nxt.cpu()[0]))
        return np.array(toks, np.int32)

    greedy = device_loop(0.0, 0.0)
    ref = oracle.Model(wl.config_tuple(), w)
    tok = 1
    for pos in range(n):
        r = ref.forward(tok, pos)
        top2 = np.sort(r)[-2:]
        tok = int(np.argmax(r))
        if top2[1] - top2[0] <= LOGIT_ABS:
            break
        assert greedy[pos + 1] == tok, f"pos {pos}: device {greedy[pos + 1]}, oracle {tok}"
    assert pos >= 8
    assert np.array_equal(device_loop(0.8, 0.9), host_loop(0.8, 0.9))


def test_out_of_range_device_token_is_reported():
    wl = WORKLOADS["tiny"]
    dec = pkg.Decoder(wl.config_tuple(), pkg.to_device(synth.make_weights(wl)))
    bad = torch.tensor([wl.vocab_size + 5], dtype=torch.int32, device="cuda")
    dec.forward_dev_tokens(bad, 0)
    with pytest.raises(pkg.L2Error) as e:
        dec.sync()
    assert e.value.code == pkg.L2_EDEVICE
    dec.sync()  # the error word was cleared
