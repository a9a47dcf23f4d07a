"""Build and load the CUDA library (``libl2decode.so``) behind the C ABI of
``include/l2.h``.  ctypes declarations only; no computation happens here."""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libl2decode.so")
# the bounds-checked build (every kernel index checked; see l2_debug_bounds_checked)
BUILD_CHECKED = os.path.join(BUILD, "checked")
LIB_CHECKED = os.path.join(BUILD, "libl2decode_checked.so")
SOURCES = ("gemv.cu", "gemv_batched.cu", "gemv_tc.cu", "attention.cu", "attn_prefill.cu", "step_kernel.cu", "step_cta.cu",
           "sample.cu", "l2_api.cu")
HEADERS = ("l2_device.cuh", "l2_params.h", "l2_kernels.h")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return "nvcc"


def _stale(lib: str | None = None) -> bool:
    lib = lib or LIB
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "l2.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile every CUDA source for sm_103a (in parallel) and link the shared
    library; checked=True builds the bounds-checked variant instead."""
    lib = LIB_CHECKED if checked else LIB
    if not force and not _stale(lib):
        return lib
    objdir = BUILD_CHECKED if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-DL2_DEBUG_BOUNDS=1"] if checked else []

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


class L2Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("dim", "hidden_dim", "n_layers", "n_heads", "n_kv_heads", "vocab_size", "seq_len")]


WEIGHT_FIELDS = ("token_embedding_table", "rms_att_weight", "rms_ffn_weight", "wq", "wk", "wv", "wo",
                 "w1", "w2", "w3", "rms_final_weight", "wcls")


class L2Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


EXPORTS = ("l2_create", "l2_reset", "l2_forward", "l2_forward_batch", "l2_forward_host", "l2_logits",
           "l2_position", "l2_debug_attention", "l2_kv_export", "l2_kv_import", "l2_sync",
           "l2_last_error", "l2_destroy", "l2_launch_op", "l2_kernels_per_step",
           "l2_step_input_bytes", "l2_forward_static", "l2_debug_fail_alloc_at", "l2_sample",
           "l2_forward_dev_tokens", "l2_prefill", "l2_debug_fail_graph_at", "l2_debug_wait_timeout",
           "l2_debug_bounds_checked", "l2_debug_limit_cache", "l2_launch_op_batch")

_lib = None


def declare(lib):
    vp, i, fp = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    ip = ctypes.POINTER(ctypes.c_int)
    lib.l2_create.argtypes = [ctypes.POINTER(L2Config), ctypes.POINTER(L2Weights), i, ctypes.c_uint, vp,
                              ctypes.POINTER(vp)]
    lib.l2_reset.argtypes = [vp, i]
    lib.l2_forward.argtypes = [vp, i, i, fp]
    lib.l2_forward_batch.argtypes = [vp, i, ip, ip, fp]
    lib.l2_forward_host.argtypes = [vp, i, i, fp]
    lib.l2_logits.argtypes = [vp]
    lib.l2_logits.restype = vp
    lib.l2_position.argtypes = [vp, i]
    lib.l2_debug_attention.argtypes = [vp, i, i, fp]
    lib.l2_kv_export.argtypes = [vp, i, i, i, fp, fp]
    lib.l2_kv_import.argtypes = [vp, i, i, fp, fp]
    lib.l2_sync.argtypes = [vp]
    lib.l2_last_error.argtypes = [vp]
    lib.l2_last_error.restype = ctypes.c_char_p
    lib.l2_destroy.argtypes = [vp]
    lib.l2_destroy.restype = None
    lib.l2_launch_op.argtypes = [vp, i, i, i]
    lib.l2_launch_op_batch.argtypes = [vp, i, i, i, i]
    lib.l2_kernels_per_step.argtypes = [vp, i]
    lib.l2_forward_static.argtypes = [vp, i, i, fp]
    lib.l2_step_input_bytes.argtypes = []
    lib.l2_step_input_bytes.restype = i
    lib.l2_debug_fail_alloc_at.argtypes = [i]
    lib.l2_debug_fail_alloc_at.restype = None
    lib.l2_sample.argtypes = [fp, i, i, ctypes.c_float, ctypes.c_float, vp, vp, vp]
    lib.l2_sample.restype = i
    lib.l2_forward_dev_tokens.argtypes = [vp, i, vp, ip, fp]
    lib.l2_forward_dev_tokens.restype = i
    lib.l2_prefill.argtypes = [vp, i, i, ip, i, fp]
    lib.l2_prefill.restype = i
    lib.l2_debug_fail_graph_at.argtypes = [i]
    lib.l2_debug_fail_graph_at.restype = None
    lib.l2_debug_wait_timeout.argtypes = [vp, i]
    lib.l2_debug_wait_timeout.restype = i
    lib.l2_debug_bounds_checked.argtypes = []
    lib.l2_debug_bounds_checked.restype = i
    lib.l2_debug_limit_cache.argtypes = [vp, ctypes.c_ulonglong]
    lib.l2_debug_limit_cache.restype = i
    for name in ("l2_create", "l2_reset", "l2_forward", "l2_forward_batch", "l2_forward_host",
                 "l2_position", "l2_debug_attention", "l2_kv_export", "l2_kv_import", "l2_sync",
                 "l2_launch_op", "l2_launch_op_batch", "l2_kernels_per_step", "l2_forward_static"):
        getattr(lib, name).restype = i
    return lib


def load(build_if_missing: bool = True):
    """The loaded CUDA library (the bounds-checked build when the environment
    sets L2DECODE_BOUNDS_CHECKED=1).  Raises if it is not built (and cannot be)."""
    global _lib
    if _lib is None:
        checked = os.environ.get("L2DECODE_BOUNDS_CHECKED") == "1"
        lib = LIB_CHECKED if checked else LIB
        if build_if_missing and _stale(lib):
            build(checked=checked)
        if not os.path.exists(lib):
            raise RuntimeError(f"CUDA library {lib} is missing; run build()")
        _lib = declare(ctypes.CDLL(lib))
    return _lib
