"""Stand-ins for the CUDA pieces bench.py touches, so that its GPU arms can be
run on a machine without a GPU to check the JSON line they print.  Test
infrastructure only: the decoder here computes its logits with the oracle,
and nothing in the package ever imports this module.

Run as a script: installs the stand-ins, then runs bench.main(argv).
"""
import os
import sys
import time
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402
import llama_transformer_decode_gb300 as pkg  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402


class FakeDecoder:
    """The binding's Decoder API over the oracle, with the library's cache
    precondition (a step may not skip unwritten rows) enforced."""

    def __init__(self, config, weights, max_batch=1, stream=None, flags=0):
        self.m = oracle.Model(config, weights, n_slots=max_batch)
        self.n_layers = config[2]
        self.max_batch = max_batch
        self.written = [0] * max_batch

    def _step(self, tok, pos, slot):
        assert 0 <= pos <= self.written[slot], (slot, pos, self.written[slot])
        r = self.m.forward(int(tok), int(pos), slot=slot)
        self.written[slot] = pos + 1
        return r

    def reset(self, slot=-1):
        for b in (range(self.max_batch) if slot < 0 else [slot]):
            self.m.key_cache[b][:] = 0
            self.m.value_cache[b][:] = 0
            self.written[b] = 0

    def position(self, slot=0):
        return self.written[slot]

    def kv_import(self, k, v, slot=0):
        n = k.shape[1]
        self.m.key_cache[slot][:, :n] = k
        self.m.value_cache[slot][:, :n] = v
        self.written[slot] = n

    def forward(self, token, pos, out=None):
        r = self._step(token, pos, 0)
        if out is not None:
            out.copy_(torch.from_numpy(r))

    def forward_host(self, token, pos, out):
        out[...] = self._step(token, pos, 0)

    def forward_batch(self, tokens, pos, out=None):
        for b in range(len(tokens)):
            r = self._step(tokens[b], pos[b], b)
            if out is not None:
                out[b].copy_(torch.from_numpy(r))

    def prefill(self, tokens, pos0=0, slot=0, out=None):
        for i, t in enumerate(tokens):
            r = self._step(t, pos0 + i, slot)
            if out is not None:
                out[i].copy_(torch.from_numpy(r))

    def launch_op(self, op, layer=0, count=1, batch=1):
        pass

    def kernels_per_step(self, batch=1):
        return 5 * self.n_layers + 1 + (1 if batch >= bench.TC_MIN_BATCH else 0)

    def step_input_bytes(self):
        return 1232  # sizeof the step block (tokens, positions, slots, rows written, output, count, chunk plan)

    def sync(self):
        pass

    def close(self):
        pass


class _Event:
    def __init__(self, enable_timing=False):
        self.t = None

    def record(self, stream=None):
        self.t = time.perf_counter()

    def synchronize(self):
        pass

    def elapsed_time(self, other):
        return max(1e-3, (other.t - self.t) * 1000.0)


class _Stream:
    cuda_stream = 0

    def synchronize(self):
        pass


def install():
    torch.cuda.set_device = lambda d: None
    torch.cuda.get_device_properties = lambda d: types.SimpleNamespace(uuid="GPU-stand-in", multi_processor_count=152)
    torch.cuda.Stream = _Stream
    torch.cuda.Event = _Event
    torch.cuda.synchronize = lambda *a: None
    empty = torch.empty
    torch.empty = lambda *a, device=None, **k: empty(*a, **k)
    pkg._native.load = lambda *a, **k: None
    pkg.Decoder = FakeDecoder
    bench.load_weights_device = lambda wl, keep_host: (synth.make_weights(wl),
                                                       synth.make_weights(wl) if keep_host else None)


if __name__ == "__main__":
    install()
    sys.exit(bench.main(sys.argv[1:]))
