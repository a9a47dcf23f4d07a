"""Pins for the oracle: what the pages and the mathematics fix, checked on CPU.

Each test names the oracle function it pins and the property it uses.  None
of them re-types the oracle's own code: they use closed forms, invariants,
exact small-integer arithmetic, brute-force float64 products, and a second
formulation of the whole step (``tests/recompute.py``, the full causal
recompute of the R/Keras page).
"""
import math

import numpy as np
import pytest

import oracle
import synth
from synth import WORKLOADS
from tests.recompute import full_logits, rotary_tables, rotate_every_two

RNG = np.random.default_rng(1234)


def ulp_diff(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(a - b)


# ---------------------------------------------------------------- matmul ----

def test_matmul_small_integer_exact():
    # W (d=3, n=2) @ x (n,) -> (d,): integer operands make every result exact.
    w = np.array([[1, 2], [3, 4], [5, 6]], np.float32)
    x = np.array([1, -1], np.float32)
    assert oracle.matmul(w, x).tolist() == [-1.0, -1.0, -1.0]
    w = RNG.integers(-50, 50, size=(37, 53)).astype(np.float32)
    x = RNG.integers(-50, 50, size=53).astype(np.float32)
    exact = [sum(int(w[i, j]) * int(x[j]) for j in range(53)) for i in range(37)]
    assert oracle.matmul(w, x).tolist() == [float(e) for e in exact]


def test_matmul_matches_bruteforce_double():
    # Non-square so a transposed operand cannot pass; the oracle sums in double,
    # so it must equal the float64 product rounded once to fp32 (<= 1 ulp for
    # the order of the double sum).
    for d, n in [(1, 1), (7, 300), (300, 7), (129, 4096)]:
        w = RNG.standard_normal((d, n)).astype(np.float32)
        x = RNG.standard_normal(n).astype(np.float32)
        ref = (w.astype(np.float64) @ x.astype(np.float64)).astype(np.float32)
        assert ulp_diff(oracle.matmul(w, x), ref).max() <= 1


# --------------------------------------------------------------- rmsnorm ----

def test_rmsnorm_closed_forms():
    x = np.array([3.0, 4.0], np.float32)
    o = oracle.rmsnorm(x, np.ones(2, np.float32))
    inv = 1.0 / math.sqrt((9.0 + 16.0) / 2.0 + 1e-5)
    assert np.allclose(o, [3 * inv, 4 * inv], rtol=1e-7, atol=0)
    assert np.all(oracle.rmsnorm(x, np.zeros(2, np.float32)) == 0.0)
    for n in (1, 5, 64, 4096):
        x = RNG.standard_normal(n).astype(np.float32) * 0.03
        o = oracle.rmsnorm(x, np.ones(n, np.float32)).astype(np.float64)
        ms = np.mean(x.astype(np.float64) ** 2)
        assert abs(np.mean(o * o) - ms / (ms + 1e-5)) < 1e-6


def test_rmsnorm_weight_is_elementwise():
    n = 33
    x = RNG.standard_normal(n).astype(np.float32)
    w = RNG.standard_normal(n).astype(np.float32)
    ratio = oracle.rmsnorm(x, w).astype(np.float64) / (w.astype(np.float64) * x)
    assert np.allclose(ratio, ratio[0], rtol=1e-6)
    assert abs(ratio[0] - 1.0 / math.sqrt(np.mean(x.astype(np.float64) ** 2) + 1e-5)) < 1e-6 * ratio[0]


# --------------------------------------------------------------- softmax ----

def test_softmax_closed_forms():
    assert oracle.softmax([5.0]).tolist() == [1.0]
    p = oracle.softmax([0.0, math.log(2.0)])
    assert np.allclose(p, [1 / 3, 2 / 3], rtol=1e-7)
    assert np.all(oracle.softmax(np.full(10, 7.5)) == np.float32(0.1))
    p = oracle.softmax([1000.0, 1001.0])  # no overflow: the maximum is subtracted
    assert np.allclose(p, [1 / (1 + math.e), math.e / (1 + math.e)], rtol=1e-7)


def test_softmax_sum_and_shift_invariance():
    for n in (2, 17, 4096):
        # values on a 2^-10 grid, so that adding 10 is exact in fp32
        x = (np.round(RNG.standard_normal(n) * 3 * 1024) / 1024).astype(np.float32)
        p = oracle.softmax(x)
        assert abs(p.astype(np.float64).sum() - 1.0) <= n * 2.0 ** -24
        assert np.all(p > 0)
        assert ulp_diff(oracle.softmax(x + np.float32(10.0)), p).max() <= 1
        assert int(np.argmax(p)) == int(np.argmax(x))


# ------------------------------------------------------------------ RoPE ----

@pytest.mark.parametrize("hs", [2, 8, 48, 64, 128])
def test_rope_pos0_identity_bitwise(hs):
    v = RNG.standard_normal(3 * hs).astype(np.float32)
    assert np.array_equal(oracle.rope(v, hs, 0), v)


@pytest.mark.parametrize("hs,pos", [(8, 1), (48, 17), (64, 1023), (128, 4095)])
def test_rope_matches_complex_rotation_and_keeps_norm(hs, pos):
    v = RNG.standard_normal(2 * hs).astype(np.float32)
    r = oracle.rope(v, hs, pos)
    # (v0 + i v1) * exp(i theta_j), theta_j = pos * 10000^(-2j/hs), j the pair index in the head
    z = v.astype(np.float64)[0::2] + 1j * v.astype(np.float64)[1::2]
    j = np.arange(v.size // 2) % (hs // 2)
    rot = z * np.exp(1j * pos * 10000.0 ** (-2.0 * j / hs))
    assert np.allclose(r[0::2], rot.real, rtol=0, atol=2e-7 * np.abs(z).max())
    assert np.allclose(r[1::2], rot.imag, rtol=0, atol=2e-7 * np.abs(z).max())
    n_in = np.hypot(v[0::2].astype(np.float64), v[1::2])
    n_out = np.hypot(r[0::2].astype(np.float64), r[1::2])
    assert np.all(np.abs(n_out - n_in) <= 2 * np.spacing(n_in.astype(np.float32)))


def test_rope_matches_rotate_every_two_tables():
    # The R/Keras page's tensor form: x * cos + rotate_every_two(x) * sin.
    hs, T = 16, 40
    cos, sin = rotary_tables(T, hs)
    for pos in (0, 3, 39):
        v = RNG.standard_normal(hs).astype(np.float32)
        ref = v * cos[pos] + rotate_every_two(v.astype(np.float64)) * sin[pos]
        assert np.allclose(oracle.rope(v, hs, pos), ref, rtol=0, atol=1e-6)


def test_rope_scores_depend_only_on_relative_position():
    hs = 64
    q = RNG.standard_normal(hs).astype(np.float32)
    k = RNG.standard_normal(hs).astype(np.float32)
    base = float(np.dot(oracle.rope(q, hs, 10).astype(np.float64), oracle.rope(k, hs, 3)))
    for s in (1, 100, 1000):
        other = float(np.dot(oracle.rope(q, hs, 10 + s).astype(np.float64), oracle.rope(k, hs, 3 + s)))
        assert abs(other - base) < 1e-4
    far = float(np.dot(oracle.rope(q, hs, 20).astype(np.float64), oracle.rope(k, hs, 3)))
    assert abs(far - base) > 1e-3  # and it does depend on m - n


# ------------------------------------------------------------------- GQA ----

def test_kv_head_map():
    # Whole groups: equals the pages' h / kv_mul with kv_mul = n_heads / n_kv_heads.
    for H, KV in [(8, 4), (12, 12), (32, 32), (32, 4), (6, 1)]:
        assert [oracle.kv_head(h, H, KV) for h in range(H)] == [h // (H // KV) for h in range(H)]
    # 6 query heads on 4 KV heads (the walkthrough's own dim=288 example).
    assert [oracle.kv_head(h, 6, 4) for h in range(6)] == [0, 0, 1, 2, 2, 3]
    for H, KV in [(6, 4), (7, 3), (10, 4)]:
        g = [oracle.kv_head(h, H, KV) for h in range(H)]
        assert g == sorted(g) and set(g) == set(range(KV))
        sizes = np.bincount(g)
        assert sizes.max() - sizes.min() <= 1


def test_page_printed_kv_dim(tmp_path):
    # The walkthrough prints kv_dim = 288*4/6 = 192 for its example model.
    from tests.golden import read_golden
    g = read_golden("page_shapes.txt")
    dim, H, KV, kv_dim = (int(g[k]) for k in ("dim", "n_heads", "n_kv_heads", "kv_dim"))
    w = {k: np.zeros(s, np.float32) for k, s in
         {"emb": (2, dim), "rms_att": (1, dim), "rms_ffn": (1, dim), "wq": (1, dim, dim),
          "wk": (1, kv_dim, dim), "wv": (1, kv_dim, dim), "wo": (1, dim, dim), "w1": (1, 4, dim),
          "w2": (1, dim, 4), "w3": (1, 4, dim), "rms_final": (dim,), "wcls": (2, dim)}.items()}
    m = oracle.Model((dim, 4, 1, H, KV, 2, 3), w)
    assert m.kv_dim == kv_dim and m.key_cache[0].shape == (1, 3, kv_dim)
    m.forward(1, 0)  # a wrong kv_dim would index outside the (1, kv_dim, dim) wk slab


# ------------------------------------------------------------- attention ----

def test_attention_pos0_returns_v_exactly():
    hs = 48
    q = RNG.standard_normal(hs).astype(np.float32) * 10
    k = RNG.standard_normal((1, hs)).astype(np.float32)
    v = RNG.standard_normal((1, hs)).astype(np.float32)
    out, att = oracle.attention_head(q, k, v, 0)
    assert att.tolist() == [1.0] and np.array_equal(out, v[0])


def test_attention_matches_bruteforce():
    hs, T = 16, 50
    q = RNG.standard_normal(hs).astype(np.float32)
    k = RNG.standard_normal((T, hs)).astype(np.float32)
    v = RNG.standard_normal((T, hs)).astype(np.float32)
    for pos in (1, 9, T - 1):
        out, att = oracle.attention_head(q, k, v, pos)
        s = k[: pos + 1].astype(np.float64) @ q / math.sqrt(hs)
        p = np.exp(s - s.max())
        p /= p.sum()
        assert np.allclose(att, p, rtol=1e-12, atol=1e-15)
        assert abs(att.sum() - 1) < 1e-12
        assert np.allclose(out, p @ v[: pos + 1].astype(np.float64), rtol=0, atol=1e-6)
    # Equal keys: uniform weights, output is the mean of the value rows.
    k_eq = np.repeat(k[:1], T, axis=0)
    out, att = oracle.attention_head(q, k_eq, v, T - 1)
    assert np.allclose(att, 1.0 / T, rtol=1e-12)
    assert np.allclose(out, v.astype(np.float64).mean(axis=0), atol=1e-6)


# ------------------------------------------------------ whole decode step ----

def small_workload(H, KV, *, dim=24, hidden=40, L=2, V=50, S=24, seed=7, sharp=1.0):
    """A tiny model whose weights keep activations O(1) and attention sharp, so
    that every term of the step moves the logits visibly."""
    wl = WORKLOADS["tiny"].replace(name="pin", dim=dim, hidden_dim=hidden, n_layers=L, n_heads=H,
                                   n_kv_heads=KV, vocab_size=V, seq_len=S, shared_wcls=False,
                                   seed_override=seed, std=1.0 / math.sqrt(dim), rms_std=0.2,
                                   std_scale=(("wq", sharp), ("wk", sharp), ("emb", 3.0)))
    return wl, synth.make_weights(wl)


PIN_SHAPES = [(6, 4), (4, 2), (4, 4), (6, 1)]


@pytest.mark.parametrize("H,KV", PIN_SHAPES)
def test_incremental_decode_equals_full_causal_recompute(H, KV):
    wl, w = small_workload(H, KV, sharp=2.5)
    toks = synth.token_stream(wl, 0, 20)
    m = oracle.Model(wl.config_tuple(), w)
    inc = m.decode(toks)
    ref, probs = full_logits(wl.config_tuple(), w, toks, return_probs=True)
    scale = np.abs(ref).max()
    assert np.abs(inc - ref).max() <= 1e-5 * scale
    # attention probabilities of the last step, every layer and head
    m2 = oracle.Model(wl.config_tuple(), w)
    m2.decode(toks[:-1])
    _, att = m2.forward(int(toks[-1]), len(toks) - 1, want_att=True)
    T = len(toks)
    assert np.abs(att[:, :, :T] - probs[:, :, T - 1, :]).max() < 1e-6
    assert np.allclose(att[:, :, :T].astype(np.float64).sum(-1), 1.0, atol=T * 2.0 ** -24)
    # the attention is not near-uniform, so the test exercises the scores
    assert probs[:, :, T - 1, :].max() > 3.0 / T


def test_gqa_equals_replicated_mha_bitwise():
    H, KV = 6, 4
    wl, w = small_workload(H, KV, sharp=2.5)
    hs = wl.head_size
    g = [oracle.kv_head(h, H, KV) for h in range(H)]
    rows = np.concatenate([np.arange(gi * hs, (gi + 1) * hs) for gi in g])
    w_mha = dict(w)
    w_mha["wk"] = np.ascontiguousarray(w["wk"][:, rows, :])
    w_mha["wv"] = np.ascontiguousarray(w["wv"][:, rows, :])
    toks = synth.token_stream(wl, 0, 12)
    a = oracle.Model(wl.config_tuple(), w).decode(toks)
    cfg = list(wl.config_tuple())
    cfg[4] = H
    b = oracle.Model(tuple(cfg), w_mha).decode(toks)
    assert np.array_equal(a, b)


def test_zero_wo_w2_reduces_to_embedding_classifier():
    wl, w = small_workload(6, 4)
    w = dict(w)
    w["wo"] = np.zeros_like(w["wo"])
    w["w2"] = np.zeros_like(w["w2"])
    toks = synth.token_stream(wl, 0, 10)
    got = oracle.Model(wl.config_tuple(), w).decode(toks)
    e = w["emb"][toks].astype(np.float64)
    xn = e / np.sqrt(np.mean(e * e, axis=1, keepdims=True) + 1e-5) * w["rms_final"]
    ref = xn @ w["wcls"].astype(np.float64).T
    assert np.abs(got - ref).max() <= 1e-6 * np.abs(ref).max()


def test_pos0_attention_is_v_and_cache_rows_written():
    wl, w = small_workload(4, 2)
    m = oracle.Model(wl.config_tuple(), w)
    _, att = m.forward(3, 0, want_att=True)
    assert np.all(att[:, :, 0] == 1.0) and np.all(att[:, :, 1:] == 0.0)
    # K row at pos 0 is unrotated (theta = 0), V row is Wv @ rmsnorm(x)
    x = w["emb"][3]
    xb = oracle.rmsnorm(x, w["rms_att"][0])
    assert np.array_equal(m.key_cache[0][0, 0], oracle.matmul(w["wk"][0], xb))
    assert np.array_equal(m.value_cache[0][0, 0], oracle.matmul(w["wv"][0], xb))
    assert np.all(m.key_cache[0][:, 1:] == 0.0)


def test_decode_is_deterministic():
    wl, w = small_workload(6, 4)
    toks = synth.token_stream(wl, 0, 8)
    a = oracle.Model(wl.config_tuple(), w).decode(toks)
    b = oracle.Model(wl.config_tuple(), w).decode(toks)
    assert np.array_equal(a, b)


def test_rejects_out_of_range_arguments():
    wl, w = small_workload(4, 2)
    m = oracle.Model(wl.config_tuple(), w)
    for tok, pos in [(-1, 0), (wl.vocab_size, 0), (0, -1), (0, wl.seq_len)]:
        with pytest.raises(ValueError):
            m.forward(tok, pos)


def test_tiny_workload_recompute_prefix():
    # The tiny workload itself (shared classifier, 8 heads on 4 KV heads):
    # its first 16 teacher-forced steps against the full recompute.
    wl = WORKLOADS["tiny"]
    w = synth.make_weights(wl)
    assert w["wcls"] is w["emb"]
    toks = synth.token_stream(wl, 0, 16)
    inc = oracle.Model(wl.config_tuple(), w).decode(toks)
    ref = full_logits(wl.config_tuple(), w, toks)
    assert np.abs(inc - ref).max() <= 1e-5 * np.abs(ref).max()
