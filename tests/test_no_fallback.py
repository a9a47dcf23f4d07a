"""The product has no CPU path: the package never loads the oracle, refuses
host tensors, and raises when no GPU is present.  Host-only checks."""
import os
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import llama_transformer_decode_gb300 as pkg  # noqa: E402
import synth  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_package_import_does_not_load_the_oracle():
    code = ("import sys; import llama_transformer_decode_gb300 as p; p._native.load(); "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "False"


def test_package_sources_name_no_oracle_file():
    pkg_dir = os.path.join(ROOT, "llama_transformer_decode_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        if "_build" in dirpath or "__pycache__" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "l2_oracle" not in text and "sampler_oracle" not in text, f


def test_binding_refuses_host_tensors():
    with pytest.raises(ValueError):
        pkg._ptr(torch.zeros(4))
    with pytest.raises(TypeError):
        pkg._ptr(np.zeros(4, np.float32))


@pytest.mark.skipif(torch.cuda.is_available(), reason="a GPU is present")
def test_decoder_raises_without_a_gpu():
    wl = synth.WORKLOADS["tiny"]
    w = {k: torch.from_numpy(v) for k, v in synth.make_weights(wl).items()}
    with pytest.raises(Exception):
        pkg.Decoder(wl.config_tuple(), w)
    with pytest.raises(Exception):
        pkg.to_device(synth.make_weights(wl))
