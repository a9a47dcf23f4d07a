"""Index arithmetic of the attention kernels, checked on the CPU.

The query heads a KV head serves, and the split of cache positions over
chunks (CTAs) and warps, are integer formulas in the kernel sources; they
are read from those sources here and checked for every head grouping up to
64 heads against the oracle's head map g(h) = floor(h * n_kv_heads / n_heads)
("run.c 逐行解讀" §4 forward() step 2e, with the grouping reading for
non-integer ratios), and for every position count of the benchmark contexts.
"""
import os
import re

import pytest

import oracle

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "llama_transformer_decode_gb300", "csrc")


def _src(name):
    return open(os.path.join(CSRC, name)).read()


def _c_to_py(expr: str) -> str:
    return re.sub(r"\((?:long long|int)\)", "", expr).replace("/", "//")


@pytest.fixture(scope="module")
def attn():
    src = _src("attention.cu")
    m = re.search(r"const int h0 = (.+?), h1 = (.+?);", src)
    assert m, "head range not found in the decode attention kernel"
    h0, h1 = (eval("lambda g, H, KV: " + _c_to_py(e)) for e in m.groups())
    m = re.search(r"const int max_group = (.+?);", src)
    max_group = eval("lambda n_heads, n_kv_heads: " + _c_to_py(m.group(1)))
    m = re.search(r"int n_active = p.capacity > 0 \? \(int\)p.step->nchunk\[b\] : (.+?);\n"
                  r"\s*if \(n_active > p.n_chunks\) n_active = p.n_chunks;\n"
                  r"\s*if \(n_active > P\) n_active = P;\n\s*if \(n_active < 1\) n_active = 1;", src)
    assert m, "chunk count not found in the decode attention kernel"
    # a step of one row: at least min_chunk positions per CTA (several rows: the host's plan)
    n_active = eval("lambda P, chunk: " + _c_to_py(m.group(1).replace("p.min_chunk", "chunk")))
    m = re.search(r"const int t0 = (.+?), t1 = (.+?);", src)
    t0, t1 = (eval("lambda c, P, n_active: " + _c_to_py(e)) for e in m.groups())
    m = re.search(r"const int wt0 = (.+?);\n\s*const int wt1 = (.+?);", src)
    wt0, wt1 = (eval("lambda t0, t1, rgi, NRG: " + _c_to_py(e)) for e in m.groups())
    return dict(h0=h0, h1=h1, max_group=max_group, n_active=n_active, t0=t0, t1=t1, wt0=wt0, wt1=wt1)


def test_heads_of_a_kv_head_are_the_oracle_groups(attn, oracle_lib):
    for H in range(1, 65):
        for KV in range(1, H + 1):
            covered = []
            for g in range(KV):
                a, b = attn["h0"](g, H, KV), attn["h1"](g, H, KV)
                assert 1 <= b - a <= attn["max_group"](H, KV)
                for h in range(a, b):
                    assert oracle.kv_head(h, H, KV, lib=oracle_lib) == g, (H, KV, h)
                covered += range(a, b)
            assert covered == list(range(H))


def test_persistent_step_kernel_uses_the_same_head_range():
    a = re.search(r"const int h0 = (.+?), h1 = (.+?);", _src("attention.cu")).groups()
    b = re.search(r"const int h0 = (.+?), h1 = (.+?);", _src("step_kernel.cu")).groups()
    assert a == b


def test_prompt_chunk_kernel_head_groups(oracle_lib):
    src = _src("attn_prefill.cu")
    assert re.search(r"const int h0 = g \* GQ;", src) and re.search(r"if \(n_heads % n_kv_heads\) return false;", src)
    for H in range(1, 65):
        for KV in range(1, H + 1):
            if H % KV:
                continue  # the prompt-chunk kernel is not used for these groupings
            GQ = H // KV
            for g in range(KV):
                for j in range(GQ):
                    assert oracle.kv_head(g * GQ + j, H, KV, lib=oracle_lib) == g


@pytest.mark.parametrize("n_chunks", [1, 2, 7, 16, 64, 152])
def test_positions_split_over_chunks_and_rings(attn, n_chunks):
    # rings per CTA: 8 (one warp per ring), 4 or 2 (two or four warps sharing a ring)
    for NRG in (8, 4, 2):
        for chunk in (1, 3, 32, 64, 100, 128):
            for P in list(range(1, 300)) + [1024, 2047, 2048, 4095, 4096]:
                n = max(1, min(attn["n_active"](P, chunk), n_chunks, P))
                assert 1 <= n <= P
                prev = 0
                for c in range(n):
                    a, b = attn["t0"](c, P, n), attn["t1"](c, P, n)
                    assert a == prev and b > a  # every joining CTA has positions
                    wprev = a
                    for r in range(NRG):
                        wa, wb = attn["wt0"](a, b, r, NRG), attn["wt1"](a, b, r, NRG)
                        assert wa == wprev and wb >= wa
                        wprev = wb
                    assert wprev == b
                    prev = b
                assert prev == P


def test_any_host_planned_chunk_count_splits_every_row(attn):
    # several rows: n_active comes from the host's plan (clamped to 1..min(n_chunks, P));
    # every count in that range must split the row's positions into non-empty chunks
    for P in list(range(1, 200)) + [1023, 2048]:
        for n in range(1, min(P, 40) + 1):
            ends = [attn["t1"](c, P, n) for c in range(n)]
            starts = [attn["t0"](c, P, n) for c in range(n)]
            assert starts[0] == 0 and ends[-1] == P
            assert all(b > a for a, b in zip(starts, ends)) and starts[1:] == ends[:-1]
