"""The batch-1 GEMV's shared-memory layout of the input vector for bf16
weights, checked on the CPU.

A bf16 weight word w (8 weights, 16 bytes) of a row meets the input words 2w
and 2w + 1 (16 bytes each).  The kernel rearranges the input in place after
the RMSNorm: block kb of 32 weight words (M = min(32, nw - 32 kb) of them in
a row's last block) keeps its 2M input words as the even words, then the odd
ones.  The dot loop's lane l, starting at row word w0 = (a - rs) + l of a
chunk segment, then reads words 2 (w0 & ~31) + (w0 & 31) and M further on,
advancing 64 words per iteration.  The formulas are read from the kernel
source and simulated here: the rearrangement is a permutation of each
block's words, every lane reads exactly x[2w] and x[2w + 1] for its weight
word w at any segment start, and each group of 8 lanes (one shared-memory
wavefront of 16-byte loads) reads 8 distinct bank groups.  The same check
rejects the in-place layout the kernel had before (a 2-way conflict).
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "llama_transformer_decode_gb300", "csrc", "gemv.cu")


@pytest.fixture(scope="module")
def src():
    s = open(SRC).read()
    # the rearrangement (one warp per block) and the dot loop's reads, as the kernel states them
    for pat in (r"for \(int kb = warp; 32 \* kb < nw; kb \+= NW\) \{",
                r"const int M = min\(32, nw - 32 \* kb\);",
                r"e = xs\[64 \* kb \+ 2 \* lane\];",
                r"o = xs\[64 \* kb \+ 2 \* lane \+ 1\];",
                r"xs\[64 \* kb \+ lane\] = e;",
                r"xs\[64 \* kb \+ M \+ lane\] = o;",
                r"const int w0 = \(a - rs\) \+ lane;",
                r"int wb = w0 & ~31;",
                r"const float4 \*xr = xs \+ 2 \* wb \+ \(w0 & 31\);",
                r"const int M = min\(32, nw - wb\);",
                r"acc = dot_bf16x8\(reinterpret_cast<const uint4 \*>\(wr\)\[i\], xr\[0\], xr\[M\], acc\);",
                r"xr \+= 64;",
                r"wb \+= 32;"):
        assert re.search(pat, s), f"bf16 input layout changed in the kernel: {pat}"
    return s


def rearrange(x, nw):
    """The kernel's in-place rearrangement of one row's 2*nw input words."""
    out = list(x)
    for kb in range((nw + 31) // 32):
        M = min(32, nw - 32 * kb)
        e = [x[64 * kb + 2 * lane] for lane in range(M)]
        o = [x[64 * kb + 2 * lane + 1] for lane in range(M)]
        for lane in range(M):
            out[64 * kb + lane] = e[lane]
            out[64 * kb + M + lane] = o[lane]
    return out


def reads(nw, start, cnt):
    """(iteration, lane, word w, first index, second index) of every load of a
    segment of cnt weight words starting at row word `start`, as the dot loop
    issues them."""
    out = []
    for lane in range(32):
        w0 = start + lane
        wb = w0 & ~31
        xr = 2 * wb + (w0 & 31)
        for t, i in enumerate(range(lane, cnt, 32)):
            M = min(32, nw - wb)
            out.append((t, lane, start + i, xr, xr + M))
            xr += 64
            wb += 32
    return out


def conflict_free(loads):
    """Each iteration's 32 loads, in wavefronts of 8 lanes: distinct 16-byte
    word addresses modulo 8 (8 bank groups of 4 banks) within a wavefront."""
    by_iter = {}
    for t, lane, _, a, b in loads:
        by_iter.setdefault(t, {})[lane] = (a, b)
    for it in by_iter.values():
        for which in (0, 1):
            for g in range(4):
                addrs = [it[l][which] for l in range(8 * g, 8 * g + 8) if l in it]
                if len({a % 8 for a in addrs}) != len(addrs):
                    return False
    return True


NWS = [1, 6, 8, 31, 32, 33, 36, 64, 96, 172, 256, 512, 704, 1376]


@pytest.mark.parametrize("nw", NWS)
def test_rearrangement_is_a_permutation_and_reads_match(src, nw):
    x = list(range(2 * nw))
    xp = rearrange(x, nw)
    assert sorted(xp) == x  # nothing lost or duplicated, nothing written past the row
    for start in sorted({0, 1, 5, 31, 32, 33, nw // 2, max(0, nw - 33), max(0, nw - 1)}):
        if start >= nw:
            continue
        for cnt in sorted({1, 7, 32, 33, nw - start}):
            if cnt <= 0 or start + cnt > nw:
                continue
            for _, lane, w, a, b in reads(nw, start, cnt):
                assert 0 <= a < 2 * nw and 0 <= b < 2 * nw
                assert (xp[a], xp[b]) == (2 * w, 2 * w + 1), (nw, start, cnt, lane, w)


@pytest.mark.parametrize("nw", [32, 64, 512, 1376])
def test_full_blocks_conflict_free(src, nw):
    for start in (0, 5, 17, 32):
        assert conflict_free(reads(nw, start, nw - start)), (nw, start)


def test_in_place_layout_had_a_two_way_conflict():
    # the layout before: lane l read words 2 (start + l) and 2 (start + l) + 1 in place
    loads = [(0, lane, lane, 2 * lane, 2 * lane + 1) for lane in range(32)]
    assert not conflict_free(loads)


def test_checker_rejects_a_fixed_block_width():
    # a plausible mistake: the odd words always 32 apart, also in a row's last, shorter block
    def rearrange32(x, nw):
        out = list(x) + [None] * 64
        for kb in range((nw + 31) // 32):
            M = min(32, nw - 32 * kb)
            e = [x[64 * kb + 2 * lane] for lane in range(M)]
            o = [x[64 * kb + 2 * lane + 1] for lane in range(M)]
            for lane in range(M):
                out[64 * kb + lane] = e[lane]
                out[64 * kb + 32 + lane] = o[lane]
        return out
    for nw in (6, 36, 172):
        xp = rearrange32(list(range(2 * nw)), nw)
        bad = [(a, b, w) for _, _, w, a, b in reads(nw, 0, nw) if (xp[a], xp[b]) != (2 * w, 2 * w + 1)]
        assert bad, nw
