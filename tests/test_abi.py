"""The C-ABI library builds, loads, and exports every entry point that
include/l2.h declares.  Host-only checks: no kernel runs here."""
import ctypes
import os
import re

import pytest

import llama_transformer_decode_gb300 as pkg
from llama_transformer_decode_gb300 import _native

HEADER = os.path.join(_native.ROOT, "include", "l2.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(l2_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    try:
        return _native.load()
    except OSError as e:  # libcudart not loadable on this host
        pytest.skip(f"cannot load the CUDA runtime here: {e}")


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(_native.EXPORTS)


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_struct_layouts_match_header():
    assert ctypes.sizeof(_native.L2Config) == 7 * 4
    assert ctypes.sizeof(_native.L2Weights) == 12 * ctypes.sizeof(ctypes.c_void_p)
    text = open(HEADER).read()
    for field in _native.WEIGHT_FIELDS:
        assert re.search(r"\*%s;" % field, text), field


def test_create_rejects_bad_arguments_on_the_host(lib):
    cfg = _native.L2Config(64, 172, 5, 8, 4, 512, 512)
    w = _native.L2Weights()
    h = ctypes.c_void_p()
    assert lib.l2_create(None, ctypes.byref(w), 1, 0, None, ctypes.byref(h)) == pkg.L2_EINVAL
    assert lib.l2_create(ctypes.byref(cfg), ctypes.byref(w), 0, 0, None, ctypes.byref(h)) == pkg.L2_EINVAL
    assert lib.l2_create(ctypes.byref(cfg), ctypes.byref(w), 65, 0, None, ctypes.byref(h)) == pkg.L2_EINVAL
    assert b"max_batch" in lib.l2_last_error(None)
    assert lib.l2_create(ctypes.byref(cfg), ctypes.byref(w), 1, 0x100, None, ctypes.byref(h)) == pkg.L2_EINVAL
    for bad in [(64, 172, 5, 7, 4, 512, 512), (64, 172, 5, 8, 9, 512, 512), (64, 170, 5, 8, 4, 512, 512),
                (0, 172, 5, 8, 4, 512, 512), (544, 172, 5, 2, 2, 512, 512), (64, 172, 5, 16, 1, 512, 512)]:
        c = _native.L2Config(*bad)
        assert lib.l2_create(ctypes.byref(c), ctypes.byref(w), 1, 0, None, ctypes.byref(h)) == pkg.L2_EINVAL
    # a valid config with NULL weight pointers is refused before any device work
    assert lib.l2_create(ctypes.byref(cfg), ctypes.byref(w), 1, 0, None, ctypes.byref(h)) == pkg.L2_EINVAL
    assert b"NULL" in lib.l2_last_error(None)
    assert not h.value


def test_null_handle_calls_fail_cleanly(lib):
    toks = (ctypes.c_int * 2)(1, 2)
    pos = (ctypes.c_int * 2)(0, 0)
    host = (ctypes.c_float * 4)()
    hp = ctypes.cast(host, ctypes.c_void_p)
    assert lib.l2_forward(None, 0, 0, None) == pkg.L2_EINVAL
    assert lib.l2_forward_batch(None, 2, toks, pos, None) == pkg.L2_EINVAL
    assert lib.l2_forward_host(None, 0, 0, hp) == pkg.L2_EINVAL
    assert lib.l2_forward_static(None, 0, 0, None) == pkg.L2_EINVAL
    assert lib.l2_forward_dev_tokens(None, 2, None, pos, None) == pkg.L2_EINVAL
    assert lib.l2_prefill(None, 0, 2, toks, 0, None) == pkg.L2_EINVAL
    assert lib.l2_reset(None, 0) == pkg.L2_EINVAL
    assert lib.l2_sync(None) == pkg.L2_EINVAL
    assert lib.l2_position(None, 0) == pkg.L2_EINVAL
    assert lib.l2_kernels_per_step(None, 1) == pkg.L2_EINVAL
    assert lib.l2_debug_attention(None, 0, 0, hp) == pkg.L2_EINVAL
    assert lib.l2_kv_export(None, 0, 0, 1, hp, hp) == pkg.L2_EINVAL
    assert lib.l2_kv_import(None, 0, 1, hp, hp) == pkg.L2_EINVAL
    assert lib.l2_launch_op(None, 0, 0, 1) == pkg.L2_EINVAL
    assert lib.l2_logits(None) is None
    assert lib.l2_last_error(None) is not None  # the last l2_create failure on this thread, never NULL
    lib.l2_destroy(None)


def test_step_input_bytes_is_the_step_block(lib):
    # the bytes one step copies host -> device: its token, position and output-pointer block
    n = lib.l2_step_input_bytes()
    assert n > 0 and n % 8 == 0


def test_sample_rejects_bad_arguments_on_the_host(lib):
    f = ctypes.c_void_p
    buf = (ctypes.c_float * 16)()
    st = (ctypes.c_uint64 * 2)(1, 2)
    out = (ctypes.c_int * 2)()
    p, s, o = ctypes.cast(buf, f), ctypes.cast(st, f), ctypes.cast(out, f)
    assert lib.l2_sample(None, 1, 16, 1.0, 0.9, s, o, None) == pkg.L2_EINVAL
    assert b"NULL" in lib.l2_last_error(None)
    assert lib.l2_sample(p, 0, 16, 1.0, 0.9, s, o, None) == pkg.L2_EINVAL
    assert lib.l2_sample(p, 1, 0, 1.0, 0.9, s, o, None) == pkg.L2_EINVAL
    assert lib.l2_sample(p, 1, 49153, 1.0, 0.9, s, o, None) == pkg.L2_EINVAL
    assert b"vocab_size" in lib.l2_last_error(None)
    for t in (-1.0, float("inf"), float("nan")):
        assert lib.l2_sample(p, 1, 16, t, 0.9, s, o, None) == pkg.L2_EINVAL
    assert lib.l2_sample(p, 1, 16, 1.0, float("nan"), s, o, None) == pkg.L2_EINVAL
    # host memory is refused before any launch
    assert lib.l2_sample(p, 1, 16, 1.0, 0.9, s, o, None) == pkg.L2_EINVAL
    assert b"device memory" in lib.l2_last_error(None)
