"""Pins of the bf16 rounding helper the bf16-weight tests feed to the oracle
(round to nearest, ties to even, as IEEE 754 defines it)."""
import numpy as np

from tests.bf16 import round_bf16, rounded_model


def f32(x):
    return np.float32(x)


def test_exact_bf16_values_are_kept():
    for v in (0.0, -0.0, 1.0, -2.5, 0.15625, 2.0 ** -100, 3.0 * 2.0 ** 50):
        assert round_bf16(np.array([v], np.float32))[0] == f32(v)


def test_ties_go_to_even_and_others_to_nearest():
    one = 1.0
    cases = [
        (one + 2.0 ** -8, one),                              # halfway, even neighbour is 1.0
        (one + 3 * 2.0 ** -8, one + 2.0 ** -6),              # halfway between odd 1+2^-7 and even 1+2^-6
        (-(one + 2.0 ** -8), -one),                          # sign-symmetric
        (one + 2.0 ** -8 + 2.0 ** -20, one + 2.0 ** -7),     # just above half: up
        (one + 2.0 ** -8 - 2.0 ** -20, one),                 # just below half: down
        (2.0 - 2.0 ** -9, 2.0),                              # carry into the next binade
    ]
    for x, want in cases:
        got = round_bf16(np.array([x], np.float32))[0]
        assert got == f32(want), (x, got, want)


def test_nearest_of_the_two_neighbours_on_random_data():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(20000) * 0.05).astype(np.float32)
    r = round_bf16(x)
    assert np.all(r.view(np.uint32) & 0xFFFF == 0)
    u = x.view(np.uint32)
    lo = (u & 0xFFFF0000).view(np.float32)                   # truncation (towards zero)
    hi = ((u & 0xFFFF0000) + 0x10000).view(np.float32)       # next bf16 away from zero
    d = np.abs(r.astype(np.float64) - x)
    assert np.all(d <= np.minimum(np.abs(lo.astype(np.float64) - x), np.abs(hi.astype(np.float64) - x)))


def test_rounded_model_leaves_embedding_and_gains():
    w = {k: np.linspace(-1, 1, 64, dtype=np.float32).reshape(8, 8) + 1e-4 for k in
         ("emb", "rms_att", "rms_ffn", "rms_final", "wq", "wk", "wv", "wo", "w1", "w2", "w3")}
    w["wcls"] = w["emb"]
    r = rounded_model(w)
    for k in ("emb", "rms_att", "rms_ffn", "rms_final"):
        assert r[k] is w[k]
    assert np.array_equal(r["wcls"], round_bf16(w["emb"])) and r["wcls"] is not r["emb"]
