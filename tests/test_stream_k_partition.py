"""The tensor-core GEMV's stream-K work split, checked exhaustively on the CPU.

The kernel lays the (output tile, K stage) pairs of a launch out tile-major,
T = tiles * KT of them, and gives CTA c the range [c*T/G, (c+1)*T/G).  A
CTA's range is whole tiles plus at most a partial tile at each end; partial
tiles go to workspace slot 0 (the range's first segment) or 1 (its last),
each contributing CTA takes one ticket, and the last one adds the parts of
CTAs cta_of(t*KT) .. cta_of((t+1)*KT - 1) in that order.  Those integer
formulas are read here from the kernel source itself (so the test follows the
kernel) and checked for every shape class the host plans: every pair is
covered exactly once, cta_of inverts the ranges, the slot the merge reads is
the one the CTA wrote, the ticket count equals the contributing CTAs, and
the parts cover K once, in K order.
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "llama_transformer_decode_gb300", "csrc", "gemv_tc.cu")


def _c_to_py(expr: str) -> str:
    """A C integer expression over non-negative values -> Python."""
    e = re.sub(r"\((?:long long|int)\)", "", expr)
    e = e.replace("blockIdx.x", "c").replace("/", "//")
    return e


@pytest.fixture(scope="module")
def formulas():
    src = open(SRC).read()
    m = re.search(r"const long long s_begin = (.+?), s_end = (.+?);", src)
    assert m, "range formulas not found in the kernel"
    s_begin, s_end = (eval("lambda c, T, G: " + _c_to_py(g)) for g in m.groups())
    m = re.search(r"auto cta_of = \[&\]\(long long x\) \{ return (.+?); \};", src)
    assert m, "cta_of not found in the kernel"
    cta_of = eval("lambda x, T, G: " + _c_to_py(m.group(1)))
    m = re.search(r"k1 = \(int\)min\(\(long long\)KT, (.+?)\);", src)
    assert m, "segment end not found in the kernel"
    k1_rest = eval("lambda k0, s_end, sq: " + _c_to_py(m.group(1)))
    m = re.search(r"const int which = (.+?) \? 0 : 1;", src)
    assert m and m.group(1) == "sq == s_begin", "slot choice changed in the kernel"
    m = re.search(r"const int wh = (.+?) \? 0 : 1;", src)
    assert m, "merge slot formula not found in the kernel"
    wh = eval("lambda cc, T, G, t, KT: 0 if (" + _c_to_py(m.group(1)) + ") else 1")
    m = re.search(r"#define L2_TC_MIN_CTA_STAGES (\d+)", src)
    min_stages = int(m.group(1))
    assert re.search(r"std::min<long long>\(ctas, T / kMinCtaStages\)", src), "grid rule changed in the kernel"
    return dict(s_begin=s_begin, s_end=s_end, cta_of=cta_of, k1_rest=k1_rest, wh=wh, min_stages=min_stages)


def check_plan(f, ntiles: int, KT: int, ctas: int):
    T = ntiles * KT
    G = max(1, min(ctas, T // f["min_stages"]))
    assert 1 <= G <= min(ctas, T)
    seg_of = {}  # tile -> list of (cta, k0, k1, which)
    prev_end = 0
    for c in range(G):
        b, e = f["s_begin"](c, T, G), f["s_end"](c, T, G)
        assert b == prev_end and e > b, (ntiles, KT, ctas, c)
        if T >= f["min_stages"]:
            assert e - b >= f["min_stages"]
        prev_end = e
        assert f["cta_of"](b, T, G) == c and f["cta_of"](e - 1, T, G) == c
        parts = []
        sq = b
        while sq < e:  # the kernel's segment walk
            tile, k0 = divmod(sq, KT)
            k1 = min(KT, f["k1_rest"](k0, e, sq))
            which = 0 if sq == b else 1
            seg_of.setdefault(tile, []).append((c, k0, k1, which))
            if not (k0 == 0 and k1 == KT):
                parts.append(which)
            sq += k1 - k0
        # at most the first and the last segment are partial, one per workspace slot
        assert parts.count(0) <= 1 and parts.count(1) <= 1
    assert prev_end == T
    assert sorted(seg_of) == list(range(ntiles))
    for t, segs in seg_of.items():
        # the tile's K stages covered exactly once, in K order, by consecutive CTAs
        assert segs[0][1] == 0 and segs[-1][2] == KT
        for (c_a, _, k1a, _), (c_b, k0b, _, _) in zip(segs, segs[1:]):
            assert k1a == k0b and c_b == c_a + 1
        if len(segs) == 1:
            continue  # whole tile, finished by its CTA
        c0, c1 = f["cta_of"](t * KT, T, G), f["cta_of"]((t + 1) * KT - 1, T, G)
        assert [s[0] for s in segs] == list(range(c0, c1 + 1))  # tickets: c1 - c0 + 1 arrivals
        for cc, _, _, which in segs:
            assert f["wh"](cc, T, G, t, KT) == which  # the merge reads the slot the CTA wrote


SHAPES_T = list(range(1, 70)) + [88, 125, 250, 344, 1376, 1513]
SHAPES_KT = [1, 2, 3, 4, 5, 7, 8, 9, 16, 31, 32, 33, 64, 88, 172]


@pytest.mark.parametrize("ctas", [1, 2, 3, 76, 148, 152])
def test_stream_k_partition(formulas, ctas):
    for ntiles in SHAPES_T:
        for KT in SHAPES_KT:
            check_plan(formulas, ntiles, KT, ctas)


def test_model_shapes(formulas):
    # the launches of the benchmark workloads: (rows of the launch's tiles, row length)
    for dim, hidden, kv_dim, vocab in [(2048, 5632, 256, 32000), (4096, 11008, 4096, 32000),
                                       (768, 2048, 768, 32000), (288, 768, 192, 32000), (64, 172, 32, 512)]:
        launches = [(-(-dim // 128) + 2 * -(-kv_dim // 128), dim),  # QKV: tiles of Wq, Wk, Wv
                    (-(-dim // 128), dim), (-(-hidden // 64), dim), (-(-dim // 128), hidden),
                    (-(-vocab // 128), dim)]
        for ntiles, n in launches:
            check_plan(formulas, ntiles, -(-n // 64), 152)


@pytest.mark.parametrize("name", ["slot_strict", "cta_of_off_by_one", "segment_overruns", "range_rounding"])
def test_checker_rejects_plausible_mistakes(formulas, name):
    bad = dict(formulas)
    if name == "slot_strict":
        bad["wh"] = lambda cc, T, G, t, KT: 0 if cc * T // G > t * KT else 1
    elif name == "cta_of_off_by_one":
        bad["cta_of"] = lambda x, T, G: ((x + 1) * G + T - 1) // T
    elif name == "segment_overruns":
        bad["k1_rest"] = lambda k0, s_end, sq: k0 + (s_end - sq) + 1
    else:
        bad["s_end"] = lambda c, T, G: -(-(c + 1) * T // G)
    with pytest.raises(AssertionError):
        for ntiles in (3, 7, 40):
            for KT in (4, 9, 32):
                check_plan(bad, ntiles, KT, 152)
