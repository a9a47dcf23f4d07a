"""The tensor-core GEMV's work splits, checked exhaustively on the CPU.

Stream-K (plans with many tiles):

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

Cluster split (plans with fewer tiles than half the SMs): tile t's K stages
are split over the CS CTAs of cluster t as [KT r / CS, KT (r + 1) / CS), and
after the distributed-shared-memory reduction rank r finishes the tile's
rows (W1/W3: row pairs) [jlo, jhi); both are read from the source and must
cover their ranges exactly once, in rank order, with no empty part and even
row bounds (RoPE pairs stay in one CTA).
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
    mb = re.search(r"const long long s_begin = CS > 1 \? (.+?)\n\s*: (.+?);", src)
    me = re.search(r"const long long s_end = CS > 1 \? (.+?)\n\s*: (.+?);", src)
    assert mb and me, "range formulas not found in the kernel"
    s_begin, s_end = (eval("lambda c, T, G: " + _c_to_py(m.group(2))) for m in (mb, me))
    # the cluster split: CTA c of a grid of ntiles * CS, K stages per tile KT
    cs_begin, cs_end = (eval("lambda c, KT, CS: " + _c_to_py(m.group(1))) for m in (mb, me))
    m = re.search(r"const int jlo = (.+?);\n\s*const int jhi = rk \+ 1 == \(uint32_t\)CS \? kUnit : (.+?);", src)
    assert m, "row split of the cluster reduction not found in the kernel"
    row_lo, row_hi = (eval("lambda rk, CS, kUnit: " + _c_to_py(g).replace("~1LL", "~1")) for g in m.groups())
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
    return dict(s_begin=s_begin, s_end=s_end, cta_of=cta_of, k1_rest=k1_rest, wh=wh, min_stages=min_stages,
                cs_begin=cs_begin, cs_end=cs_end, row_lo=row_lo, row_hi=row_hi)


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


def check_cluster_plan(f, ntiles: int, KT: int, CS: int):
    """Cluster split: CTA c = tile * CS + rank covers stages [cs_begin, cs_end) of its
    tile; every tile's K stages exactly once, in rank order, none empty; and the
    ranks' output rows (rows of a tile, or W1/W3 row pairs) split [0, kUnit) into
    non-empty even-aligned slices in rank order."""
    for t in range(ntiles):
        prev = t * KT
        for rk in range(CS):
            c = t * CS + rk
            b, e = f["cs_begin"](c, KT, CS), f["cs_end"](c, KT, CS)
            assert b == prev and e > b, (ntiles, KT, CS, c)
            # the kernel's segment walk gives this CTA one segment, of tile t
            tile, k0 = divmod(b, KT)
            assert tile == t and min(KT, f["k1_rest"](k0, e, b)) == k0 + (e - b)
            prev = e
        assert prev == (t + 1) * KT
    for unit in (128, 64):
        prev = 0
        for rk in range(CS):
            lo = f["row_lo"](rk, CS, unit)
            hi = unit if rk + 1 == CS else f["row_hi"](rk, CS, unit)
            assert lo == prev and hi > lo and lo % 2 == 0 and hi % 2 == 0
            prev = hi
        assert prev == unit


@pytest.mark.parametrize("CS", [2, 3, 4, 5, 6, 7, 8])
def test_cluster_partition(formulas, CS):
    for ntiles in (1, 2, 16, 20, 32, 76):
        for KT in [k for k in SHAPES_KT if k >= CS]:  # the host keeps CS <= KT
            check_cluster_plan(formulas, ntiles, KT, CS)


def test_cluster_checker_rejects_a_rounding_mistake(formulas):
    bad = dict(formulas)
    bad["cs_end"] = lambda c, KT, CS: (c // CS) * KT + -(-KT * (c % CS + 1) // CS) + 1
    with pytest.raises(AssertionError):
        check_cluster_plan(bad, 3, 32, 6)
