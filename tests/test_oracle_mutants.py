"""The pins have teeth: plant one plausible mistake at a time in a copy of the
oracle (on the CPU), rebuild it, and check that the pin battery rejects it.
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from tests.recompute import full_logits
from tests.test_oracle_pins import small_workload

SRC = os.path.join(os.path.dirname(oracle.__file__), "l2_oracle.c")

# (name, text in the oracle, replacement): each is a mistake a reader could make.
MUTANTS = [
    ("residual_after_wo_dropped", "x[i] = (float)((double)x[i] + (double)xb2[i]);", "x[i] = xb2[i];"),
    ("residual_after_w2_dropped", "x[i] = (float)((double)x[i] + (double)xb[i]);", "x[i] = xb[i];"),
    ("rope_sign_flipped", "vec[i] = (float)(v0 * fcr - v1 * fci);", "vec[i] = (float)(v0 * fcr + v1 * fci);"),
    ("rope_base_wrong", "pow(10000.0,", "pow(1000.0,"),
    ("rope_k_skipped", "oracle_rope(k, kv_dim, head_size, pos);", ";"),
    ("rope_freq_index_global", "int head_dim = i % head_size;", "int head_dim = i;"),
    ("gqa_map_modulo", "return (int)(((long long)h * (long long)n_kv_heads) / (long long)n_heads);",
     "return h % n_kv_heads;"),
    ("score_not_scaled", "s[t] = score / sqrt((double)head_size);", "s[t] = score;"),
    ("score_scaled_by_dim", "s[t] = score / sqrt((double)head_size);", "s[t] = score / sqrt((double)stride);"),
    ("attention_excludes_current", "for (int t = 0; t <= pos; t++) {\n        const float *k",
     "for (int t = 0; t < pos; t++) {\n        const float *k"),
    ("eps_dropped", "ss = ss / size + 1e-5;", "ss = ss / size;"),
    ("eps_outside_mean", "ss = ss / size + 1e-5;", "ss = (ss + 1e-5) / size;"),
    ("rmsnorm_weight_dropped", "o[j] = (float)((double)weight[j] * (inv * (double)x[j]));",
     "o[j] = (float)(inv * (double)x[j]);"),
    ("matmul_transposed", "const float *row = w + (size_t)i * (size_t)n;", "const float *row = w + i;"),
    ("silu_without_sigmoid", "val *= 1.0 / (1.0 + exp(-val));", ";"),
    ("ffn_w3_replaced_by_w1", "oracle_matmul(hb2, xb, w->w3 +", "oracle_matmul(hb2, xb, w->w1 +"),
    ("kv_layer_offset_dropped", "size_t loff = (size_t)l * seq * (size_t)kv_dim;", "size_t loff = 0;"),
    ("softmax_max_not_subtracted", "x[i] = exp(x[i] - max_val);", "x[i] = exp(x[i]);"),
    ("final_norm_skipped", "oracle_rmsnorm(x, x, w->rms_final_weight, dim);", ";"),
    ("ffn_norm_uses_att_weight", "oracle_rmsnorm(xb, x, w->rms_ffn_weight +", "oracle_rmsnorm(xb, x, w->rms_att_weight +"),
    ("swiglu_gate_on_w3", "double val = hb[i];\n            val *= 1.0 / (1.0 + exp(-val));\n            val *= (double)hb2[i];",
     "double val = hb2[i];\n            val *= 1.0 / (1.0 + exp(-val));\n            val *= (double)hb[i];"),
    ("silu_sign_flipped", "val *= 1.0 / (1.0 + exp(-val));", "val *= 1.0 / (1.0 + exp(val));"),
    ("v_read_from_key_cache", "value_cache + loff + (size_t)g * head_size, kv_dim",
     "key_cache + loff + (size_t)g * head_size, kv_dim"),
    ("query_head_offset_uses_kv_head", "q + (size_t)h * head_size,", "q + (size_t)g * head_size,"),
    ("kv_written_one_row_early", "float *k = key_cache + loff + (size_t)pos * kv_dim;",
     "float *k = key_cache + loff + (size_t)(pos > 0 ? pos - 1 : 0) * kv_dim;"),
    ("att_norm_layer_offset_dropped", "w->rms_att_weight + (size_t)l * dim", "w->rms_att_weight"),
    ("wq_layer_offset_dropped", "w->wq + (size_t)l * dim * dim", "w->wq"),
    ("classifier_uses_embedding", "oracle_matmul(logits, x, w->wcls, dim", "oracle_matmul(logits, x, w->token_embedding_table, dim"),
]


def battery(lib) -> list:
    """Names of the pin checks that fail for the oracle library ``lib``."""
    failed = []
    rng = np.random.default_rng(99)

    def check(name, fn):
        try:
            ok = bool(fn())
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    def recompute(H, KV):
        wl, w = small_workload(H, KV, sharp=2.5)
        toks = synth.token_stream(wl, 0, 12)
        inc = oracle.Model(wl.config_tuple(), w, lib=lib).decode(toks)
        ref = full_logits(wl.config_tuple(), w, toks)
        return np.isfinite(inc).all() and np.abs(inc - ref).max() <= 1e-5 * np.abs(ref).max()

    def rmsnorm_closed():
        x = rng.standard_normal(64).astype(np.float32) * 0.03
        o = oracle.rmsnorm(x, np.ones(64, np.float32), lib=lib).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2)
        w = rng.standard_normal(64).astype(np.float32)
        ratio = oracle.rmsnorm(x, w, lib=lib).astype(np.float64) / (w * x.astype(np.float64))
        return abs(np.mean(o * o) - ms / (ms + 1e-5)) < 1e-6 and np.allclose(ratio, ratio[0], rtol=1e-6)

    def softmax_closed():
        p = oracle.softmax([1000.0, 1001.0], lib=lib)
        return np.allclose(p, [1 / (1 + math.e), math.e / (1 + math.e)], rtol=1e-7)

    def matmul_brute():
        w = rng.standard_normal((7, 300)).astype(np.float32)
        x = rng.standard_normal(300).astype(np.float32)
        ref = w.astype(np.float64) @ x
        return np.allclose(oracle.matmul(w, x, lib=lib), ref, rtol=1e-6, atol=1e-6)

    def rope_complex():
        hs, pos = 48, 17
        v = rng.standard_normal(2 * hs).astype(np.float32)
        r = oracle.rope(v, hs, pos, lib=lib)
        z = v[0::2].astype(np.float64) + 1j * v[1::2]
        j = np.arange(hs) % (hs // 2)
        rot = z * np.exp(1j * pos * 10000.0 ** (-2.0 * j / hs))
        return np.allclose(r[0::2], rot.real, atol=1e-6) and np.allclose(r[1::2], rot.imag, atol=1e-6)

    check("recompute_gqa_6_4", lambda: recompute(6, 4))
    check("recompute_gqa_4_2", lambda: recompute(4, 2))
    check("rmsnorm_closed_form", rmsnorm_closed)
    check("softmax_closed_form", softmax_closed)
    check("matmul_bruteforce", matmul_brute)
    check("rope_complex", rope_complex)
    return failed


def test_unmutated_oracle_passes_battery():
    assert battery(oracle.load()) == []


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, find, repl):
    src = open(SRC).read()
    assert src.count(find) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(find, repl))
    lib = oracle.load(oracle.compile_oracle(str(mpath), str(tmp_path / "libmutant.so")))
    assert battery(lib), f"mutant {name} passed every pin"
