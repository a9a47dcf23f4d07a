"""The bounds-checked build of the CUDA library (L2_DEBUG_BOUNDS=1).

In that build every index the kernels compute into the handle's buffers, and
every bulk copy's source range, is checked; a violation sets the device error
word and the access is skipped (nothing faults).  Run in a child process with
L2DECODE_BOUNDS_CHECKED=1 (tests/bounds_cases.py), the decode cases of every
instrumented kernel must report no violation (each case ends in l2_sync) and
give logits bitwise equal to the release build's in this process.  Negative
control: told that each KV cache holds fewer positions than a step reads, the
checked build must flag the step (l2_sync: L2_EDEVICE) and the release build
must not (it never reads the sizes).
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import llama_transformer_decode_gb300 as pkg  # noqa: E402
from tests import bounds_cases  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_results(tmp_path_factory):
    pkg._native.build(checked=True)
    out = tmp_path_factory.mktemp("bounds") / "checked.npz"
    env = dict(os.environ, L2DECODE_BOUNDS_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "tests.bounds_cases", str(out)], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-4000:]
    return dict(np.load(out))


def test_checked_build_is_loaded_in_the_child(checked_results):
    assert int(checked_results["_checked"][0]) == 1
    assert pkg.lib().l2_debug_bounds_checked() == 0  # this process: the release build


def test_checked_build_flags_nothing_and_matches_the_release_build_bitwise(checked_results):
    release = bounds_cases.run_cases()
    assert set(release) == {k for k in checked_results if not k.startswith("_")}
    for name, want in release.items():
        got = checked_results[name]
        assert np.isfinite(want).all(), name
        assert np.array_equal(got, want), f"{name}: the checked build differs from the release build"


def test_a_lowered_cache_size_is_flagged_only_by_the_checked_build(checked_results):
    assert int(checked_results["_limited_rc"][0]) == pkg.L2_EDEVICE
    assert bounds_cases.limited_cache_is_flagged() == pkg.L2_OK
