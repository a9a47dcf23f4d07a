"""Pins of the sampler oracle (oracle/sampler_oracle.c) to facts outside it.

- The exponential: within 1 fp32 ulp of libm's double exp over (-87, 0].
- argmax: numpy's argmax (the first maximum) on random and tied inputs.
- The coin and multinomial draw: for equal logits every weight is exactly
  2^48, so the drawn index is floor(k * n / 2^24) for the coin k, a closed
  form; over many draws, frequencies match the softmax distribution
  computed in double by numpy (chi-square), at several temperatures.
- Top-p: the nucleus of hand-built distributions (which tokens can appear
  and in what ratio), ties resolved towards lower indices, a tiny topp
  keeping only the most probable token, topp outside (0, 1) meaning no
  nucleus.
- temperature 0: argmax of the logits and no draw from the generator.
- xorshift*: the walkthrough (§6 Sampler, random_u32()) prints the shifts
  and the multiplier; they are stored with that citation in
  tests/golden/sampler_constants.txt.  The oracle's state update, observed
  on the 64 basis states, is a 64 x 64 matrix over GF(2) that must equal the
  product of the three elementary matrices I + S built from the printed
  shifts; that matrix must have order exactly 2^64 - 1 (the generator visits
  every non-zero state), checked against the prime factors of 2^64 - 1; and
  the output, for states whose successor is 2^k (preimages taken with the
  printed matrix, not the oracle), must be the top 32 bits of the printed
  multiplier times 2^k, which fixes all 64 bits of the multiplier.  Linearity,
  injectivity, a non-zero orbit and chi-square uniformity are checked too.
"""
import math
import os
import subprocess

import numpy as np
import pytest

import oracle

M64 = (1 << 64) - 1


def draws(n, state=0x1234_5678_9ABC_DEF0):
    out = []
    for _ in range(n):
        v, state = oracle.random_u32(state)
        out.append(v)
    return np.array(out, dtype=np.uint64), state


def test_exp_within_one_ulp_of_libm():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.uniform(-86.99, 0.0, 20000), -rng.uniform(0.0, 1e-3, 2000),
                         np.array([0.0, -1e-30, -0.5, -1.0, -10.0, -86.9, -math.log(2.0)])]).astype(np.float32)
    for x in xs:
        got = oracle.sampler_exp(float(x))
        want = math.exp(float(x))
        assert abs(got - want) <= np.spacing(np.float32(want)), (x, got, want)
    assert oracle.sampler_exp(0.0) == 1.0
    assert oracle.sampler_exp(-87.0) == 0.0 and oracle.sampler_exp(-1000.0) == 0.0


def test_argmax_is_the_first_maximum():
    rng = np.random.default_rng(2)
    for n in (1, 2, 7, 512, 32000):
        v = rng.standard_normal(n).astype(np.float32)
        assert oracle.argmax(v) == int(np.argmax(v))
        v = np.round(v).astype(np.float32)  # many ties
        assert oracle.argmax(v) == int(np.argmax(v))


def test_xorshift_steps_are_linear_invertible_and_never_zero():
    rng = np.random.default_rng(3)

    def step(x):  # one xorshift* state update, observed through the oracle
        _, s = oracle.random_u32(x)
        return s

    for _ in range(200):
        a, b = (int(rng.integers(1, 1 << 63)) * 2 + 1) & M64, int(rng.integers(1, 1 << 62))
        assert step(a ^ b) == step(a) ^ step(b)  # linear over GF(2)
        assert step(a) != 0
    # invertibility: distinct states map to distinct states on a sample
    xs = {int(v) for v in rng.integers(1, 1 << 62, size=5000)}
    assert len({step(x) for x in xs}) == len(xs)


# ---- xorshift* pinned to the constants the walkthrough prints ----
# A linear map of GF(2)^64 is held as its 64 columns (the images of the basis
# states 1 << j, as Python ints); products use 8-bit lookup tables.

def _gf2_apply(cols, x):
    r, j = 0, 0
    while x:
        if x & 1:
            r ^= cols[j]
        x >>= 1
        j += 1
    return r


def _gf2_tables(cols):
    tabs = []
    for k in range(8):
        t = [0] * 256
        for v in range(1, 256):
            low = v & -v
            t[v] = t[v ^ low] ^ cols[8 * k + low.bit_length() - 1]
        tabs.append(t)
    return tabs


def _gf2_compose(f, g):
    """Columns of f o g."""
    tf = _gf2_tables(f)
    out = []
    for x in g:
        r = 0
        for k in range(8):
            r ^= tf[k][(x >> (8 * k)) & 255]
        out.append(r)
    return out


IDENTITY = [1 << j for j in range(64)]


def _gf2_pow(f, n):
    result, base = IDENTITY, f
    while n:
        if n & 1:
            result = _gf2_compose(base, result)
        base = _gf2_compose(base, base)
        n >>= 1
    return result


def _shift_matrix(k):
    """Columns of I + S where S shifts a state right by k (k > 0) or left by -k, mod 2^64."""
    cols = []
    for j in range(64):
        src = 1 << j
        shifted = (src >> k) if k > 0 else ((src << -k) & M64)
        cols.append(src ^ shifted)
    return cols


def golden_xorshift():
    from tests.golden import read_golden
    g = read_golden("sampler_constants.txt")
    r1, l1, r2 = int(g["shift_right_1"]), int(g["shift_left"]), int(g["shift_right_2"])
    # the page applies right r1, then left l1, then right r2
    m = _gf2_compose(_shift_matrix(r2), _gf2_compose(_shift_matrix(-l1), _shift_matrix(r1)))
    return m, int(g["multiplier"], 16), int(g["output_shift"])


# prime factors of 2^64 - 1 = (2^32 + 1)(2^16 + 1)(2^8 + 1)(2^4 + 1)(2^2 + 1)(2 + 1)
ORDER_PRIMES = (3, 5, 17, 257, 641, 65537, 6700417)


def _is_prime(n):
    return n > 1 and all(n % d for d in range(2, int(math.isqrt(n)) + 1))


def oracle_step_matrix(lib=None):
    return [oracle.random_u32(1 << j, lib)[1] for j in range(64)]


def test_xorshift_update_is_the_printed_recurrence():
    m, _, _ = golden_xorshift()
    assert oracle_step_matrix() == m


def test_xorshift_has_full_period():
    assert math.prod(ORDER_PRIMES) == M64 and all(_is_prime(p) for p in ORDER_PRIMES)
    m = oracle_step_matrix()
    assert _gf2_pow(m, M64) == IDENTITY
    for p in ORDER_PRIMES:
        assert _gf2_pow(m, M64 // p) != IDENTITY, p


def test_xorshift_output_is_the_printed_multiplier():
    m, mult, out_shift = golden_xorshift()
    inv = _gf2_pow(m, M64 - 1)  # m has order 2^64 - 1 (checked above), so this is its inverse
    for k in (0, 1, 7, 31, 32, 33, 63):
        target = 1 << k
        pre = _gf2_apply(inv, target)
        v, s = oracle.random_u32(pre)
        assert s == target
        assert v == ((target * mult) & M64) >> out_shift, k


def test_coin_is_uniform():
    v, _ = draws(65536)
    hist = np.bincount((v >> np.uint64(24)).astype(np.int64), minlength=256)
    exp = len(v) / 256
    chi2 = float(((hist - exp) ** 2 / exp).sum())
    assert chi2 < 360, chi2  # 255 dof: p ~ 1e-4 at 360


@pytest.mark.parametrize("n", [1, 3, 10, 32000])
def test_equal_logits_draw_the_closed_form_index(n):
    logits = np.zeros(n, np.float32)
    state = 0xDEADBEEF
    for _ in range(200):
        k24 = oracle.random_u32(state)[0] >> 8
        idx, state, total, r = oracle.sample(logits, 1.0, 0.0, state)
        assert total == n << 48
        assert idx == (k24 * n) >> 24


@pytest.mark.parametrize("temperature", [0.5, 1.0, 1.7])
def test_frequencies_follow_the_softmax(temperature):
    rng = np.random.default_rng(4)
    logits = rng.standard_normal(12).astype(np.float32) * 1.5
    p = np.exp((logits.astype(np.float64) - logits.max()) / temperature)
    p /= p.sum()
    state, counts, N = 42, np.zeros(12), 40000
    for _ in range(N):
        idx, state, _, _ = oracle.sample(logits, temperature, 0.0, state)
        counts[idx] += 1
    chi2 = float(((counts - N * p) ** 2 / (N * p)).sum())
    assert chi2 < 40, (chi2, counts, N * p)  # 11 dof: p ~ 1e-4 at 40


def test_top_p_nucleus_membership_and_ratio():
    probs = np.array([0.05, 0.5, 0.15, 0.3])  # sorted: 1 (0.5), 3 (0.3), 2 (0.15), 0 (0.05)
    logits = np.log(probs).astype(np.float32)
    for topp, members in ((0.6, {1, 3}), (0.85, {1, 3, 2}), (0.97, {0, 1, 2, 3}), (0.3, {1})):
        state, seen, counts = 7, set(), {}
        for _ in range(6000):
            idx, state, _, _ = oracle.sample(logits, 1.0, topp, state)
            seen.add(idx)
            counts[idx] = counts.get(idx, 0) + 1
        assert seen == members, (topp, seen)
    # within {1, 3} the odds are 5:3
    state, c = 9, {1: 0, 3: 0}
    for _ in range(16000):
        idx, state, _, _ = oracle.sample(logits, 1.0, 0.6, state)
        c[idx] += 1
    assert abs(c[1] / (c[1] + c[3]) - 0.625) < 0.015


def test_top_p_ties_prefer_lower_indices_and_degenerate_topp():
    logits = np.zeros(8, np.float32)  # all equal: the nucleus is the lowest indices
    state, seen = 11, set()
    for _ in range(4000):
        idx, state, total, _ = oracle.sample(logits, 1.0, 0.3, state)
        seen.add(idx)
        assert total == 3 << 48  # ceil(0.3 * 8) = 3 tokens
    assert seen == {0, 1, 2}
    # a tiny topp keeps the single most probable token
    logits = np.array([0.1, 2.0, 2.0, -1.0], np.float32)
    state = 5
    for _ in range(200):
        idx, state, _, _ = oracle.sample(logits, 1.0, 1e-6, state)
        assert idx == 1
    # topp outside (0, 1) is plain sampling over all tokens
    for topp in (0.0, 1.0, -0.5, 2.0):
        a = oracle.sample(logits, 1.0, topp, 99)
        b = oracle.sample(logits, 1.0, 0.0, 99)
        assert a == b


def test_temperature_zero_is_argmax_without_a_draw():
    rng = np.random.default_rng(6)
    logits = rng.standard_normal(1000).astype(np.float32)
    idx, state, _, _ = oracle.sample(logits, 0.0, 0.9, 1234)
    assert idx == int(np.argmax(logits)) and state == 1234


# ---- the pins have teeth: one planted mistake at a time in a copy of the
# sampler oracle (CPU only), rebuilt, must fail at least one quick check ----

SRC = os.path.join(os.path.dirname(oracle.__file__), "sampler_oracle.c")
MUTANTS = [
    ("coin_from_low_bits", "const uint32_t k24 = oracle_random_u32(state) >> 8;",
     "const uint32_t k24 = oracle_random_u32(state) & 0xFFFFFFu;"),
    ("temperature_ignored", "const float e = oracle_sampler_exp(logits[i] / temperature - m);",
     "const float e = oracle_sampler_exp(logits[i] - m);"),
    ("ties_prefer_higher_index", "return x->idx < y->idx ? -1 : (x->idx > y->idx);",
     "return x->idx > y->idx ? -1 : (x->idx < y->idx);"),
    ("nucleus_from_least_probable", "if (x->q != y->q) return x->q > y->q ? -1 : 1;",
     "if (x->q != y->q) return x->q < y->q ? -1 : 1;"),
    ("taylor_term_dropped", "float p = c7;\n    p = fmaf(p, r, c6);", "float p = c6;"),
    ("argmax_last_maximum", "if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;"),
    ("exp_reduction_low_part_dropped", "r = fmaf(-k, ln2_lo, r);", ";"),
    ("xorshift_first_shift_wrong", "*state ^= *state >> 12;", "*state ^= *state >> 13;"),
    ("xorshift_left_shift_wrong", "*state ^= *state << 25;", "*state ^= *state << 24;"),
    ("xorshift_last_shift_wrong", "*state ^= *state >> 27;", "*state ^= *state >> 26;"),
    ("xorshift_shift_direction_flipped", "*state ^= *state << 25;", "*state ^= *state >> 25;"),
    ("xorshift_steps_reordered", "*state ^= *state >> 12;\n    *state ^= *state << 25;",
     "*state ^= *state << 25;\n    *state ^= *state >> 12;"),
    ("xorshift_multiplier_digit_wrong", "0x2545F4914F6CDD1DULL", "0x2545F4914F6CDD1FULL"),
    ("xorshift_output_low_half", "return (uint32_t)((*state * 0x2545F4914F6CDD1DULL) >> 32);",
     "return (uint32_t)(*state * 0x2545F4914F6CDD1DULL);"),
]


_GOLD_INV = []


def golden_xorshift_inverse():
    """((printed update matrix, its inverse), multiplier, output shift), computed once."""
    if not _GOLD_INV:
        m, mult, out_shift = golden_xorshift()
        _GOLD_INV.append(((m, _gf2_pow(m, M64 - 1)), mult, out_shift))
    return _GOLD_INV[0]


def quick_battery(lib) -> list:
    failed = []

    def check(name, fn):
        try:
            ok = bool(fn())
        except Exception:
            ok = False
        if not ok:
            failed.append(name)

    def exp_ok():
        xs = np.linspace(-86.0, 0.0, 3001).astype(np.float32)
        return all(abs(oracle.sampler_exp(float(x), lib) - math.exp(float(x)))
                   <= np.spacing(np.float32(math.exp(float(x)))) for x in xs)

    def argmax_ok():
        v = np.array([1.0, 3.0, 3.0, 2.0], np.float32)
        return oracle.argmax(v, lib) == 1

    def closed_form_ok():
        state = 0xDEADBEEF
        for _ in range(50):
            k24 = oracle.random_u32(state, lib)[0] >> 8
            idx, state, _, _ = oracle.sample(np.zeros(10, np.float32), 1.0, 0.0, state, lib)
            if idx != (k24 * 10) >> 24:
                return False
        return True

    def temperature_ok():
        logits = np.array([0.0, 1.0, 2.0], np.float32)
        p = np.exp(logits / 0.5 - 4.0)
        p /= p.sum()
        state, c = 3, np.zeros(3)
        for _ in range(6000):
            idx, state, _, _ = oracle.sample(logits, 0.5, 0.0, state, lib)
            c[idx] += 1
        return float(((c - 6000 * p) ** 2 / (6000 * p)).sum()) < 20

    def topp_ok():
        probs = np.array([0.05, 0.5, 0.15, 0.3])
        state, seen = 7, set()
        for _ in range(3000):
            idx, state, _, _ = oracle.sample(np.log(probs).astype(np.float32), 1.0, 0.6, state, lib)
            seen.add(idx)
        if seen != {1, 3}:
            return False
        state, seen = 11, set()
        for _ in range(2000):
            idx, state, _, _ = oracle.sample(np.zeros(8, np.float32), 1.0, 0.3, state, lib)
            seen.add(idx)
        return seen == {0, 1, 2}

    def xorshift_ok():
        m, mult, out_shift = golden_xorshift_inverse()
        if oracle_step_matrix(lib) != m[0]:
            return False
        for k in (0, 32):
            v, s = oracle.random_u32(_gf2_apply(m[1], 1 << k), lib)
            if s != 1 << k or v != (((1 << k) * mult) & M64) >> out_shift:
                return False
        return True

    for name, fn in (("exp", exp_ok), ("argmax", argmax_ok), ("closed_form", closed_form_ok),
                     ("temperature", temperature_ok), ("topp", topp_ok), ("xorshift", xorshift_ok)):
        check(name, fn)
    return failed


def test_quick_battery_passes_on_the_oracle():
    assert quick_battery(oracle.load_sampler()) == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site of {name} not unique"
    mutated = tmp_path / f"{name}.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", str(mutated), "-o", str(so), "-lm"])
    assert quick_battery(oracle.load_sampler(str(so))), f"mutant {name} passed every pin"
