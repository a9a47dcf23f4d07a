// Causal grouped-query attention over the KV cache for one decode step,
// split across CTAs along the cache positions (flash-decoding).
//
// What it computes ("run.c 逐行解讀", §4 forward() step 2e; "run.c",
// transformer(), multihead attention): for every query head h with KV head
// g(h) = floor(h * n_kv_heads / n_heads),
//     s_t = q_h . K[t, g(h)] / sqrt(head_size),  t = 0..pos
//     a   = softmax(s)
//     out_h = sum_t a_t V[t, g(h)].
//
// How.  Grid (n_chunks, n_kv_heads, batch).  CTA (c, g, b) takes a contiguous
// slice of positions 0..pos of slot b and serves every query head of group g,
// so each K/V row is read from HBM once.  The cache layout is
// [slot][layer][kv_head][pos][head_size], so a slice is one contiguous range
// of K and one of V; each warp (with 8 query heads per KV head, each pair of
// warps) streams a sub-slice through its own ring of 1-D bulk async copies (TMA).  Lanes are grouped LP to a cache row (LP = the
// head size in 16-byte words, rounded up to a power of two); each group keeps
// an online softmax (running max m, sum l, un-normalised accumulator) per
// query head; with 4 or 8 query heads per KV head at head size 64 the
// row-per-lane layout (described at the kernel) splits rows, heads and
// dimensions over the lanes instead.  Groups, then warps, then CTAs are merged with the usual
// log-sum-exp rescaling; the CTA that arrives last on the group's ticket
// merges the chunks in chunk order and writes the output, so the result does
// not depend on CTA timing.  With a debug buffer the raw scores are stored and
// the last CTA turns them into probabilities exp(s_t - M) / L.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

// Launch shape (compile-time): warps per CTA, ring buffers per warp, K + V
// floats per ring buffer (a buffer holds stage_floats / (2 head_size) cache
// positions; K and V arrive as one copy each).
#ifndef L2_ATTN_WARPS
#define L2_ATTN_WARPS 8
#endif
#ifndef L2_ATTN_STAGES
#define L2_ATTN_STAGES 2
#endif
#ifndef L2_ATTN_STAGE_FLOATS
#define L2_ATTN_STAGE_FLOATS 2048
#endif

namespace l2 {

namespace {
constexpr int kNWA = L2_ATTN_WARPS;
constexpr int kAttStages = L2_ATTN_STAGES;
constexpr int kStageFloats = L2_ATTN_STAGE_FLOATS;
// Row-per-lane layout: ring buffers per ring (shared by the warps of a ring).
// Two stages measured faster than three on GB300 (batched_1b: 2.19 against
// 2.21 ms per step at 16 sequences, 3.59 against 3.60 ms at 64): less shared
// memory per CTA, more CTAs resident per SM.
#ifndef L2_ATTN_STAGES_RL
#define L2_ATTN_STAGES_RL 2
#endif
constexpr int kAttStagesRL = L2_ATTN_STAGES_RL;

// The WPR * 32 threads of one ring: named barrier 1 + ring (ids taken from
// constants, so the kernel reserves only the barriers it uses).  ring_sync_or
// gives every thread the OR of their flags; ring_sync is a plain barrier.
template <int ID, int NTH>
__device__ __forceinline__ bool bar_or_id(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID), "n"(NTH)
        : "memory");
    return r != 0;
}
template <int ID, int NTH>
__device__ __forceinline__ void bar_id(void) {
    asm volatile("bar.sync %0, %1;" ::"n"(ID), "n"(NTH) : "memory");
}
template <int NTH>
__device__ __forceinline__ bool ring_sync_or(bool v, int ring) {
    switch (ring) {
        case 0: return bar_or_id<1, NTH>(v);
        case 1: return bar_or_id<2, NTH>(v);
        case 2: return bar_or_id<3, NTH>(v);
        default: return bar_or_id<4, NTH>(v);
    }
}
template <int NTH>
__device__ __forceinline__ void ring_sync(int ring) {
    switch (ring) {
        case 0: bar_id<1, NTH>(); break;
        case 1: bar_id<2, NTH>(); break;
        case 2: bar_id<3, NTH>(); break;
        default: bar_id<4, NTH>(); break;
    }
}

__device__ __forceinline__ void merge_state(float &m, float &l, float4 &acc, float m2, float l2v, float4 acc2) {
    const float M = fmaxf(m, m2);
    if (M == -CUDART_INF_F) return;
    const float a = expf(m - M), b = expf(m2 - M);
    l = l * a + l2v * b;
    acc.x = acc.x * a + acc2.x * b;
    acc.y = acc.y * a + acc2.y * b;
    acc.z = acc.z * a + acc2.z * b;
    acc.w = acc.w * a + acc2.w * b;
    m = M;
}
}  // namespace

// RL = 1: the row-per-lane layout for 4 or 8 query heads per KV head at
// head size 64 (16 cache rows per ring stage).  Each warp serves 4 of the
// group's heads and keeps their query words in registers; with 8 heads two
// warps share a ring (two CTAs fit on an SM).  For the scores, lane (rg, dq)
// multiplies rows 4 rg .. 4 rg + 3 of the stage with the 4 heads over 8 of
// the 64 dimensions, and the 8 lanes of a row group add their partial sums up
// by exchanging halves (three shuffle rounds), leaving each (head, row) score
// in one lane.  The online softmax runs over the stage's 16 rows per head;
// the probabilities go through shared memory to the PV pass, where lane
// (hg, dg) accumulates two heads over 4 dimensions.  A cache row is read from
// shared memory twice per warp (scores, weighted sum), and no 16-byte load is
// a broadcast of one word to the whole warp: at 8 warps per SM the loop was
// bound by instruction latency, so the layout that halves the registers per
// thread (two CTAs per SM) is the one that pays.
template <int LP, int GQ, int RL>
__global__ void __launch_bounds__(kNWA * 32) attn_kernel(const AttnParams p) {
    constexpr int NT = kNWA * 32;
    constexpr int RPI = 32 / LP;        // cache rows a warp handles at once
    constexpr int WPR = RL ? GQ / 4 : 1;  // warps sharing one ring (row-per-lane: four heads per warp)
    constexpr int NRG = kNWA / WPR;     // rings per CTA (one softmax state per ring and head)
    constexpr int STG = RL ? kAttStagesRL : kAttStages;  // ring buffers per ring
    static_assert(WPR == 1 || NRG <= 4, "ring barriers are ids 1..4");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                      // [NRG][STG]
    int *flags = reinterpret_cast<int *>(smem + 8 * NRG * STG);        // [4]
    float *mrg = reinterpret_cast<float *>(smem + 8 * NRG * STG + 16); // [NRG][GQ][2]
    float *fin = mrg + NRG * GQ * 2;                                          // [GQ][2]
    const size_t hdr = (8 * NRG * STG + 16 + 4 * (NRG * GQ * 2 + GQ * 2) + 127) / 128 * 128;
    const int hs = p.head_size, hs4 = hs >> 2;
    float4 *ring = reinterpret_cast<float4 *>(smem + hdr);                     // [NRG][STG][stage]
    float4 *accs = ring + NRG * STG * (kStageFloats / 4);              // [NRG][GQ][hs4]
    float *pbuf = reinterpret_cast<float *>(accs + NRG * GQ * hs4);            // RL: [kNWA][4 heads][16 + 1]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // several rows: the host orders them, longest CTAs first
    const int c = blockIdx.x, g = blockIdx.y, b = p.capacity > 0 ? (int)p.step->row_order[blockIdx.z] : blockIdx.z;
    const int pos = p.step->pos[b];
    const int P = pos + 1;
    // CTAs of this (row, KV head): at least min_chunk positions each for a step of
    // one row; for several rows, the host's plan, which fits every row's CTAs
    // into the kernel's resident capacity at once
    int n_active = p.capacity > 0 ? (int)p.step->nchunk[b] : (P + p.min_chunk - 1) / p.min_chunk;
    if (n_active > p.n_chunks) n_active = p.n_chunks;
    if (n_active > P) n_active = P;
    if (n_active < 1) n_active = 1;
    // With a cluster and several chunks every CTA of the cluster takes part in the
    // merge (those past n_active with no positions); otherwise they have nothing to do.
    const bool in_cluster = p.cluster > 1 && n_active > 1;
    if (c >= n_active && !in_cluster) return;  // too few positions for this CTA to join

    const int H = p.n_heads, KV = p.n_kv_heads;
    const int h0 = (g * H + KV - 1) / KV, h1 = ((g + 1) * H + KV - 1) / KV;
    const int nq = h1 - h0;

    // (an idle cluster member, c >= n_active, gets the empty range [P, P))
    const int t0 = (int)((long long)min(c, n_active) * P / n_active), t1 = (int)((long long)min(c + 1, n_active) * P / n_active);
    const int rgi = warp / WPR, wsub = warp % WPR;  // this warp's ring, and its place in it
    const int wt0 = t0 + (int)((long long)(t1 - t0) * rgi / NRG);
    const int wt1 = t0 + (int)((long long)(t1 - t0) * (rgi + 1) / NRG);
    const int TP = kStageFloats / (2 * hs);  // positions per stage

    const size_t head_base = (((size_t)p.step->slot[b] * p.n_layers + p.layer) * KV + g) * (size_t)p.seq_len * hs;
    const float *kbase = p.kcache + head_base;
    const float *vbase = p.vcache + head_base;

    if (tid == 0) {
        for (int i = 0; i < NRG * STG; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        flags[0] = 0;  // a warp gave up waiting
        flags[1] = 0;  // this CTA merges the chunks
    }
    __syncthreads();

    uint64_t *wbars = bars + rgi * STG;
    float4 *wring = ring + (size_t)rgi * STG * (kStageFloats / 4);
    const bool producer = wsub == 0 && lane == 0;  // issues the ring's copies; every warp tracks them
    int ti = wt0;  // next position to request
    int n_issued = 0;
    auto issue = [&](int stage) {
        const int np = min(TP, wt1 - ti);
        if (producer) {
            const uint32_t bytes = (uint32_t)np * hs * 4u;
            float4 *dst = wring + (size_t)stage * (kStageFloats / 4);
            // rows outside the cache (bounds-checked build) are skipped; the barrier expects nothing
            const bool ok = in_bounds(head_base + (size_t)ti * hs, (size_t)np * hs, p.ext->cache, p.err);
            mbar_arrive_expect_tx(&wbars[stage], ok ? 2u * bytes : 0u);
            if (ok) {
                bulk_g2s_nohint(dst, kbase + (size_t)ti * hs, bytes, &wbars[stage]);
                bulk_g2s_nohint(dst + (size_t)TP * hs4, vbase + (size_t)ti * hs, bytes, &wbars[stage]);
            }
        }
        ti += np;
        ++n_issued;
    };
    // Rows before stable[b] (pos for an ordinary step, the chunk's first
    // position in a prefill) are not written during this step: fetch them
    // before the previous kernel (which writes the newer rows) has finished.
    const int stable = p.step->stable[b];
#pragma unroll 1
    for (int s = 0; s < STG && ti < wt1 && ti + min(TP, wt1 - ti) <= stable; ++s) issue(s);
    pdl_launch_dependents();
    pdl_wait();
#pragma unroll 1
    for (int s = n_issued; s < STG && ti < wt1; ++s) issue(s);

    bool ok = true;
    int k = 0;
    float *dbg = p.dbg ? p.dbg + (((size_t)b * p.n_layers + p.layer) * H + h0) * p.seq_len : nullptr;
    // the export's rows of this CTA's heads lie inside it (bounds-checked build), or it is not written
    if (dbg && !in_bounds((((size_t)b * p.n_layers + p.layer) * H + h0) * p.seq_len, (size_t)nq * p.seq_len,
                          p.ext->dbg, p.err))
        dbg = nullptr;
    if constexpr (RL == 1) {
        constexpr int TPR = 16;   // cache rows per ring stage (head size 64)
        constexpr int NHW = 4;    // query heads per warp (GQ / WPR)
        constexpr int RTH = WPR * 32;
        static_assert(GQ == NHW * WPR, "row-per-lane attention: 4 or 8 query heads per KV head");
        // Scores: lane (rg, dq) takes rows 4 rg .. 4 rg + 3 of the stage over dimensions
        // 4 dq .. 4 dq + 3 and 32 + 4 dq .. 32 + 4 dq + 3, for the warp's 4 heads (their
        // query words stay in registers), then the 8 lanes of the row group add up by
        // exchanging halves.  The lane's heads are numbered i ^ (dq >> 1) and its rows
        // r ^ 2 (dq & 1), so at every exchange a lane keeps the low half of its values and
        // sends the high half: it ends with head jw0 + (dq >> 1), rows r0, r0 + 1.
        const int rg = lane >> 3, dq = lane & 7, qh = dq >> 1, rb = 2 * (dq & 1);
        const int jw0 = wsub * NHW;          // the warp's first head of the group
        const int r0 = 4 * rg + rb;
        // PV: lane (hg, dg) accumulates heads jw0 + 2 hg, + 1 over dimensions 4 dg .. 4 dg + 3
        const int hg = lane >> 4, dg = lane & 15;
        float4 qa[NHW], qb[NHW];
#pragma unroll
        for (int i = 0; i < NHW; ++i) {
            const int j = jw0 + (i ^ qh);
            qa[i] = qb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            const size_t qi = (size_t)b * p.dim + (size_t)(h0 + j) * 64 + 4 * dq;
            if (j < nq && in_bounds(qi, 36, p.ext->q, p.err)) {
                qa[i] = *reinterpret_cast<const float4 *>(p.q + qi);
                qb[i] = *reinterpret_cast<const float4 *>(p.q + qi + 32);
            }
        }
        float *pT = pbuf + warp * (NHW * TPR + NHW);  // [head][row] probabilities of the stage, then [head] rescales
        float m = -CUDART_INF_F, l = 0.f;              // head jw0 + qh: running max and sum
        float4 acc[2];
        acc[0] = acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        int tc = wt0;
#pragma unroll 1
        for (; tc < wt1; ++k) {
            const int s = k % STG;
            const int np = min(TP, wt1 - tc);
            const bool got = mbar_wait(&wbars[s], (uint32_t)(k / STG) & 1u, p.err);
            // the ring's warps take one decision (the loop bounds are the ring's, so all get here)
            if (WPR > 1 ? ring_sync_or<RTH>(!got, rgi) : !got) {
                ok = false;
                break;
            }
            const float4 *K4 = wring + (size_t)s * (kStageFloats / 4);
            const float4 *V4 = K4 + TPR * 16;
            // partial scores w[i][r] over the lane's 8 dimensions (even and odd ones in the
            // two halves of packed fp32 FMAs)
            float w[NHW][4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int t = 4 * rg + (r ^ rb);
                const float4 ka = K4[t * 16 + dq], kb = K4[t * 16 + 8 + dq];
#pragma unroll
                for (int i = 0; i < NHW; ++i) {
                    float2 s2 = ffma2(make_float2(qa[i].x, qa[i].y), make_float2(ka.x, ka.y), make_float2(0.f, 0.f));
                    s2 = ffma2(make_float2(qa[i].z, qa[i].w), make_float2(ka.z, ka.w), s2);
                    s2 = ffma2(make_float2(qb[i].x, qb[i].y), make_float2(kb.x, kb.y), s2);
                    s2 = ffma2(make_float2(qb[i].z, qb[i].w), make_float2(kb.z, kb.w), s2);
                    w[i][r] = s2.x + s2.y;
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                w[0][r] += __shfl_xor_sync(0xffffffffu, w[2][r], 4);
                w[1][r] += __shfl_xor_sync(0xffffffffu, w[3][r], 4);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) w[0][r] += __shfl_xor_sync(0xffffffffu, w[1][r], 2);
            float sc[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) sc[r] = w[0][r] + __shfl_xor_sync(0xffffffffu, w[0][r + 2], 1);
            // head jw0 + qh, rows r0, r0 + 1: scale, mask, export
            const int hj = jw0 + qh;
            float mx = -CUDART_INF_F;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int t = r0 + r;
                sc[r] = t < np ? sc[r] * p.scale : -CUDART_INF_F;
                if (dbg && t < np && hj < nq) dbg[(size_t)hj * p.seq_len + tc + t] = sc[r];
                mx = fmaxf(mx, sc[r]);
            }
            // online softmax over the stage's rows: the 8 lanes of the head
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m, mx);  // finite: row 0 of the stage is valid
            const float corr = expf(m - mn);
            const float pe0 = expf(sc[0] - mn), pe1 = expf(sc[1] - mn);
            float ps = pe0 + pe1;
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 8);
            ps += __shfl_xor_sync(0xffffffffu, ps, 16);
            l = l * corr + ps;
            m = mn;
            *reinterpret_cast<float2 *>(pT + qh * TPR + r0) = make_float2(pe0, pe1);
            if (r0 == 0) pT[NHW * TPR + qh] = corr;
            __syncwarp();
            // PV: heads jw0 + 2 hg + j, dimensions 4 dg .. 4 dg + 3
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float cr = pT[NHW * TPR + 2 * hg + j];
                acc[j] = make_float4(acc[j].x * cr, acc[j].y * cr, acc[j].z * cr, acc[j].w * cr);
            }
#pragma unroll
            for (int tq = 0; tq < TPR / 4; ++tq) {
                if (4 * tq >= np) break;
                const float4 p0 = *reinterpret_cast<const float4 *>(pT + (2 * hg) * TPR + 4 * tq);
                const float4 p1 = *reinterpret_cast<const float4 *>(pT + (2 * hg + 1) * TPR + 4 * tq);
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int t = 4 * tq + r;
                    if (t >= np) break;  // rows past the slice hold stale data
                    const float4 v = V4[t * 16 + dg];
                    const float a = r == 0 ? p0.x : r == 1 ? p0.y : r == 2 ? p0.z : p0.w;
                    const float c = r == 0 ? p1.x : r == 1 ? p1.y : r == 2 ? p1.z : p1.w;
                    float2 lo = ffma2(make_float2(a, a), make_float2(v.x, v.y), make_float2(acc[0].x, acc[0].y));
                    float2 hi = ffma2(make_float2(a, a), make_float2(v.z, v.w), make_float2(acc[0].z, acc[0].w));
                    acc[0] = make_float4(lo.x, lo.y, hi.x, hi.y);
                    lo = ffma2(make_float2(c, c), make_float2(v.x, v.y), make_float2(acc[1].x, acc[1].y));
                    hi = ffma2(make_float2(c, c), make_float2(v.z, v.w), make_float2(acc[1].z, acc[1].w));
                    acc[1] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
            }
            __syncwarp();
            tc += np;
            if (WPR > 1) ring_sync<RTH>(rgi);  // the ring's warps are done with this buffer
            if (ti < wt1) {
                if (producer) fence_proxy_async_smem();
                issue(s);
            }
        }
        if (!ok) {
            for (int j = k + 1; j < n_issued; ++j)
                (void)mbar_wait(&wbars[j % STG], (uint32_t)(j / STG) & 1u, p.err);
            if (lane == 0) flags[0] = 1;
        }
        if (r0 == 0) {
            mrg[(rgi * GQ + jw0 + qh) * 2 + 0] = m;
            mrg[(rgi * GQ + jw0 + qh) * 2 + 1] = l;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) accs[(size_t)(rgi * GQ + jw0 + 2 * hg + j) * 16 + dg] = acc[j];
    } else {
        // A row's 16-byte words c4, c4 + LP, .. (WPL of them) go to the LP lanes of its
        // lane group: with one or two query heads per KV head a lane keeps several
        // words of q per head in registers, so a row's dot product ends in a short
        // shuffle tree (log2 LP levels) instead of one level per halving of 32 lanes.
        constexpr int WPL = GQ == 1 ? 4 : GQ == 2 ? 2 : 1;
        constexpr int PPG = WPL >= 4 ? 2 : 4;  // rows a lane group scores before one softmax update
        const int rg = lane / LP, c4 = lane % LP;
        float4 q4[GQ][WPL];
        float m[GQ], l[GQ];
        float4 acc[GQ][WPL];
#pragma unroll
        for (int j = 0; j < GQ; ++j) {
#pragma unroll
            for (int w = 0; w < WPL; ++w) {
                q4[j][w] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < nq && c4 + w * LP < hs4 &&
                    in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * (c4 + w * LP), 4, p.ext->q, p.err))
                    q4[j][w] = reinterpret_cast<const float4 *>(p.q + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[c4 + w * LP];
                acc[j][w] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            m[j] = -CUDART_INF_F;
            l[j] = 0.f;
        }
        int tc = wt0;
#pragma unroll 1
        for (; tc < wt1; ++k) {
            const int s = k % STG;
            const int np = min(TP, wt1 - tc);
            if (!mbar_wait(&wbars[s], (uint32_t)(k / STG) & 1u, p.err)) {
                ok = false;
                break;
            }
            const float4 *Ks = wring + (size_t)s * (kStageFloats / 4);
            const float4 *Vs = Ks + (size_t)TP * hs4;
            // Up to PPG rows per lane group at a time: all their scores first
            // (independent dot products and shuffles), then one online-softmax
            // update per head (one rescale per group of rows).
#pragma unroll 1
            for (int tt = 0; tt < np; tt += RPI * PPG) {
                float sc[PPG][GQ];
                float4 vv[PPG][WPL];
#pragma unroll
                for (int u = 0; u < PPG; ++u) {
                    const int tl = tt + u * RPI + rg;
                    const bool row_on = tl < np;
                    float4 kv[WPL];
#pragma unroll
                    for (int w = 0; w < WPL; ++w) {
                        kv[w] = make_float4(0.f, 0.f, 0.f, 0.f);
                        vv[u][w] = kv[w];
                        if (row_on && c4 + w * LP < hs4) {
                            kv[w] = Ks[tl * hs4 + c4 + w * LP];
                            vv[u][w] = Vs[tl * hs4 + c4 + w * LP];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < GQ; ++j) {
                        float d = 0.f;
#pragma unroll
                        for (int w = 0; w < WPL; ++w) d = dot4(q4[j][w], kv[w], d);
#pragma unroll
                        for (int o = LP / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                        sc[u][j] = row_on ? d * p.scale : -CUDART_INF_F;
                        if (dbg && row_on && c4 == 0 && j < nq) dbg[(size_t)j * p.seq_len + tc + tl] = sc[u][j];
                    }
                }
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    if (j >= nq) continue;
                    float mx = sc[0][j];
#pragma unroll
                    for (int u = 1; u < PPG; ++u) mx = fmaxf(mx, sc[u][j]);
                    const float mn = fmaxf(m[j], mx);
                    if (mn == -CUDART_INF_F) continue;  // no position of this group
                    const float corr = expf(m[j] - mn);
                    float pe[PPG];
                    float ps = 0.f;
#pragma unroll
                    for (int u = 0; u < PPG; ++u) {
                        pe[u] = expf(sc[u][j] - mn);
                        ps += pe[u];
                    }
#pragma unroll
                    for (int w = 0; w < WPL; ++w) {
                        float4 a = make_float4(acc[j][w].x * corr, acc[j][w].y * corr, acc[j][w].z * corr,
                                               acc[j][w].w * corr);
#pragma unroll
                        for (int u = 0; u < PPG; ++u) {
                            a.x = fmaf(pe[u], vv[u][w].x, a.x);
                            a.y = fmaf(pe[u], vv[u][w].y, a.y);
                            a.z = fmaf(pe[u], vv[u][w].z, a.z);
                            a.w = fmaf(pe[u], vv[u][w].w, a.w);
                        }
                        acc[j][w] = a;
                    }
                    l[j] = l[j] * corr + ps;
                    m[j] = mn;
                }
            }
            __syncwarp();
            tc += np;
            if (ti < wt1) {
                if (lane == 0) fence_proxy_async_smem();
                issue(s);
            }
        }
        if (!ok) {
            for (int j = k + 1; j < n_issued; ++j)
                (void)mbar_wait(&wbars[j % STG], (uint32_t)(j / STG) & 1u, p.err);
            if (lane == 0) flags[0] = 1;
        }

        // merge the row groups of the warp (lanes LP apart hold the same words)
#pragma unroll
        for (int o = LP; o < 32; o <<= 1) {
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m[j], o);
                const float l2v = __shfl_xor_sync(0xffffffffu, l[j], o);
                const float M = fmaxf(m[j], m2);
                const float fa = M == -CUDART_INF_F ? 0.f : expf(m[j] - M);
                const float fb = M == -CUDART_INF_F ? 0.f : expf(m2 - M);
#pragma unroll
                for (int w = 0; w < WPL; ++w) {
                    float4 a2;
                    a2.x = __shfl_xor_sync(0xffffffffu, acc[j][w].x, o);
                    a2.y = __shfl_xor_sync(0xffffffffu, acc[j][w].y, o);
                    a2.z = __shfl_xor_sync(0xffffffffu, acc[j][w].z, o);
                    a2.w = __shfl_xor_sync(0xffffffffu, acc[j][w].w, o);
                    if (M != -CUDART_INF_F)
                        acc[j][w] = make_float4(acc[j][w].x * fa + a2.x * fb, acc[j][w].y * fa + a2.y * fb,
                                                acc[j][w].z * fa + a2.z * fb, acc[j][w].w * fa + a2.w * fb);
                }
                if (M != -CUDART_INF_F) {
                    l[j] = l[j] * fa + l2v * fb;
                    m[j] = M;
                }
            }
        }
        if (lane < LP) {
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                if (lane == 0) {
                    mrg[(rgi * GQ + j) * 2 + 0] = m[j];
                    mrg[(rgi * GQ + j) * 2 + 1] = l[j];
                }
#pragma unroll
                for (int w = 0; w < WPL; ++w)
                    if (c4 + w * LP < hs4) accs[(size_t)(rgi * GQ + j) * hs4 + c4 + w * LP] = acc[j][w];
            }
        }
    }
    __syncthreads();
    // A CTA whose wait gave up (the error word is already set) publishes
    // nothing, but with several chunks it still takes its ticket below, so the
    // group's count completes and the last CTA resets it for the next launch.
    const bool gave_up = flags[0] != 0;

    // merge the warps in warp order and publish this CTA's partial
    const int NC = p.n_chunks;
    if (in_cluster) {
        // Thread-block cluster of the (row, KV head)'s n_chunks CTAs, rank = chunk: each
        // CTA leaves its partial (max, sum and accumulator per head, merged over its
        // rings) in its ring buffer (free now); after a cluster barrier rank 0 reads them
        // through distributed shared memory in chunk order and writes the output; a
        // second barrier keeps every partial alive until then.  No global workspace,
        // fence or ticket: those round trips took several microseconds per launch.
        float *cp = reinterpret_cast<float *>(ring);  // [GQ][2] (max, sum) in the first 64 bytes,
        float4 *ca = reinterpret_cast<float4 *>(cp + 16);  // then [GQ][hs] accumulators (16-byte aligned)
        static_assert(2 * GQ <= 16, "(max, sum) pairs fit 64 bytes");
        for (int idx = tid; idx < nq * hs4; idx += NT) {
            const int j = idx / hs4, w4 = idx % hs4;
            float mm = -CUDART_INF_F, ll = 0.f;
            float4 aa = make_float4(0.f, 0.f, 0.f, 0.f);
            if (!gave_up)
                for (int w = 0; w < NRG; ++w)
                    merge_state(mm, ll, aa, mrg[(w * GQ + j) * 2], mrg[(w * GQ + j) * 2 + 1],
                                accs[(size_t)(w * GQ + j) * hs4 + w4]);
            ca[(size_t)j * hs4 + w4] = aa;
            if (w4 == 0) {
                cp[2 * j] = mm;
                cp[2 * j + 1] = ll;
            }
        }
        cluster_sync_all();
        if (c == 0) {
            constexpr int kMaxCl = 8;
            for (int idx = tid; idx < nq * hs4; idx += NT) {
                const int j = idx / hs4, w4 = idx % hs4;
                float2 ml[kMaxCl];
                float4 a[kMaxCl];
#pragma unroll
                for (int r = 0; r < kMaxCl; ++r)
                    if (r < n_active) {
                        ml[r] = ld_dsmem2(dsmem_addr(cp + 2 * j, (uint32_t)r));
                        a[r] = ld_dsmem4(dsmem_addr(ca + (size_t)j * hs4 + w4, (uint32_t)r));
                    }
                float M = -CUDART_INF_F;
#pragma unroll
                for (int r = 0; r < kMaxCl; ++r)
                    if (r < n_active) M = fmaxf(M, ml[r].x);
                float L = 0.f;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int r = 0; r < kMaxCl; ++r)
                    if (r < n_active) {
                        const float e = expf(ml[r].x - M);
                        L += ml[r].y * e;
                        o.x += a[r].x * e;
                        o.y += a[r].y * e;
                        o.z += a[r].z * e;
                        o.w += a[r].w * e;
                    }
                const float inv = 1.0f / L;
                if (in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * w4, 4, p.ext->xb, p.err))
                    reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] =
                        make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                if (w4 == 0) {
                    fin[j * 2] = M;
                    fin[j * 2 + 1] = L;
                }
            }
            if (dbg) {
                __syncthreads();
                // the scores of every chunk (global, ordered before by the cluster barrier)
                for (int idx = tid; idx < nq * P; idx += NT) {
                    const int j = idx / P, t = idx % P;
                    float *cell = dbg + (size_t)j * p.seq_len + t;
                    *cell = expf(__ldcg(cell) - fin[j * 2]) / fin[j * 2 + 1];
                }
            }
        }
        cluster_sync_all();
        return;
    }
    if (n_active == 1) {
        if (gave_up) return;
        // The only chunk: normalise and write the output directly.
        for (int idx = tid; idx < nq * hs4; idx += NT) {
            const int j = idx / hs4, w4 = idx % hs4;
            float mm = -CUDART_INF_F, ll = 0.f;
            float4 aa = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = 0; w < NRG; ++w)
                merge_state(mm, ll, aa, mrg[(w * GQ + j) * 2], mrg[(w * GQ + j) * 2 + 1],
                            accs[(size_t)(w * GQ + j) * hs4 + w4]);
            const float inv = 1.0f / ll;
            if (in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * w4, 4, p.ext->xb, p.err))
                reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] =
                    make_float4(aa.x * inv, aa.y * inv, aa.z * inv, aa.w * inv);
            if (w4 == 0) {
                fin[j * 2] = mm;
                fin[j * 2 + 1] = ll;
            }
        }
        if (dbg) {
            __syncthreads();
            for (int idx = tid; idx < nq * P; idx += NT) {
                const int j = idx / P, t = idx % P;
                float *cell = dbg + (size_t)j * p.seq_len + t;
                *cell = expf(*cell - fin[j * 2]) / fin[j * 2 + 1];
            }
        }
        return;
    }
    for (int idx = tid; idx < (gave_up ? 0 : nq * hs4); idx += NT) {
        const int j = idx / hs4, w4 = idx % hs4;
        float mm = -CUDART_INF_F, ll = 0.f;
        float4 aa = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < NRG; ++w)
            merge_state(mm, ll, aa, mrg[(w * GQ + j) * 2], mrg[(w * GQ + j) * 2 + 1], accs[(size_t)(w * GQ + j) * hs4 + w4]);
        const size_t slot = ((size_t)b * H + h0 + j) * NC + c;
        if (!in_bounds(slot, 1, p.ext->ws_rows, p.err)) continue;
        reinterpret_cast<float4 *>(p.ws_acc + slot * hs)[w4] = aa;
        if (w4 == 0) {
            p.ws_ml[slot * 2 + 0] = mm;
            p.ws_ml[slot * 2 + 1] = ll;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        unsigned t = 0;
        if (in_bounds((size_t)b * KV + g, 1, p.ext->tickets, p.err)) t = atomicAdd(&p.tickets[b * KV + g], 1u);
        flags[1] = (t == (unsigned)(n_active - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!flags[1]) return;
    __threadfence();

    // last CTA of the group: merge the chunks in chunk order.  With up to kMrgRegs
    // chunks a thread loads every chunk's (max, sum) and accumulator words at once
    // (one round trip); with more, the (max, sum) pairs are staged in shared
    // memory first (the ring is free now: every copy has completed).
    if (!in_bounds(((size_t)b * H + h0 + nq - 1) * NC + n_active - 1, 1, p.ext->ws_rows, p.err)) return;
    constexpr int kMrgRegs = 8;
    if (n_active <= kMrgRegs) {
        for (int idx = tid; idx < nq * hs4; idx += NT) {
            const int j = idx / hs4, w4 = idx % hs4;
            const size_t sl0 = ((size_t)b * H + h0 + j) * NC;
            float2 ml[kMrgRegs];
            float4 a[kMrgRegs];
#pragma unroll
            for (int cc = 0; cc < kMrgRegs; ++cc) {
                if (cc < n_active) {
                    ml[cc] = __ldcg(reinterpret_cast<const float2 *>(p.ws_ml) + sl0 + cc);
                    a[cc] = __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + (sl0 + cc) * hs) + w4);
                }
            }
            float M = -CUDART_INF_F;
#pragma unroll
            for (int cc = 0; cc < kMrgRegs; ++cc)
                if (cc < n_active) M = fmaxf(M, ml[cc].x);
            float L = 0.f;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < kMrgRegs; ++cc) {
                if (cc < n_active) {
                    const float e = expf(ml[cc].x - M);
                    L += ml[cc].y * e;
                    o.x += a[cc].x * e;
                    o.y += a[cc].y * e;
                    o.z += a[cc].z * e;
                    o.w += a[cc].w * e;
                }
            }
            const float inv = 1.0f / L;
            o.x *= inv;
            o.y *= inv;
            o.z *= inv;
            o.w *= inv;
            if (in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * w4, 4, p.ext->xb, p.err))
                reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] = o;
            if (w4 == 0) {
                fin[j * 2] = M;
                fin[j * 2 + 1] = L;
            }
        }
        if (dbg) __syncthreads();
    } else {
        float *cml = reinterpret_cast<float *>(ring);  // [nq][n_active][2]
        for (int i = tid; i < nq * n_active; i += NT) {
            const size_t sl = ((size_t)b * H + h0 + i / n_active) * NC + i % n_active;
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.ws_ml + sl * 2));
            cml[2 * i] = ml.x;
            cml[2 * i + 1] = ml.y;
        }
        __syncthreads();
        if (tid < nq) {
            const float *c = cml + (size_t)tid * n_active * 2;
            float M = -CUDART_INF_F;
            for (int cc = 0; cc < n_active; ++cc) M = fmaxf(M, c[2 * cc]);
            float L = 0.f;
            for (int cc = 0; cc < n_active; ++cc) L += c[2 * cc + 1] * expf(c[2 * cc] - M);
            fin[tid * 2] = M;
            fin[tid * 2 + 1] = L;
        }
        __syncthreads();
        for (int i = tid; i < nq * n_active; i += NT) cml[2 * i] = expf(cml[2 * i] - fin[(i / n_active) * 2]);
        __syncthreads();
        for (int idx = tid; idx < nq * hs4; idx += NT) {
            const int j = idx / hs4, w4 = idx % hs4;
            const float inv = 1.0f / fin[j * 2 + 1];
            const float *e = cml + (size_t)j * n_active * 2;
            const float4 *src = reinterpret_cast<const float4 *>(p.ws_acc + ((size_t)b * H + h0 + j) * NC * hs) + w4;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
            for (int cc = 0; cc < n_active; ++cc) {
                const float4 a = __ldcg(src + (size_t)cc * hs4);
                o.x += a.x * e[2 * cc];
                o.y += a.y * e[2 * cc];
                o.z += a.z * e[2 * cc];
                o.w += a.w * e[2 * cc];
            }
            o.x *= inv;
            o.y *= inv;
            o.z *= inv;
            o.w *= inv;
            if (in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * w4, 4, p.ext->xb, p.err))
                reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] = o;
        }
    }
    if (dbg) {
        for (int idx = tid; idx < nq * P; idx += NT) {
            const int j = idx / P, t = idx % P;
            float *cell = dbg + (size_t)j * p.seq_len + t;
            *cell = expf(__ldcg(cell) - fin[j * 2]) / fin[j * 2 + 1];
        }
    }
    if (tid == 0 && in_bounds((size_t)b * KV + g, 1, p.ext->tickets, p.err)) p.tickets[b * KV + g] = 0u;
}

// ---------------------------------------------------------------- host side

namespace {
typedef void (*AttnFn)(const AttnParams);  // (the kernels take it as a grid constant)

template <int LP, int GQ>
AttnFn pick2() {
    return attn_kernel<LP, GQ, 0>;
}

template <int LP>
AttnFn pick1(int gq) {
    switch (gq) {
        case 1: return pick2<LP, 1>();
        case 2: return pick2<LP, 2>();
        case 4: return pick2<LP, 4>();
        case 8: return pick2<LP, 8>();
    }
    return nullptr;
}

AttnFn pick(int lp, int gq, int rl) {
    if (rl) {
        if (lp != 16) return nullptr;
        return gq == 8 ? attn_kernel<16, 8, 1> : gq == 4 ? attn_kernel<16, 4, 1> : nullptr;
    }
    switch (lp) {
        case 1: return pick1<1>(gq);
        case 2: return pick1<2>(gq);
        case 4: return pick1<4>(gq);
        case 8: return pick1<8>(gq);
        case 16: return pick1<16>(gq);
        case 32: return pick1<32>(gq);
    }
    return nullptr;
}

int pow2_at_least(int v) {
    int r = 1;
    while (r < v) r <<= 1;
    return r;
}
}  // namespace

AttnLaunch attn_plan(int head_size, int n_heads, int n_kv_heads) {
    AttnLaunch a{};
    const int hs4 = head_size / 4;
    const int max_group = (n_heads + n_kv_heads - 1) / n_kv_heads;
    a.gq = pow2_at_least(max_group);
    // lanes per cache row: the row's 16-byte words over WPL words per lane (WPL as in the kernel)
    const int wpl = a.gq == 1 ? 4 : a.gq == 2 ? 2 : 1;
    a.lp = pow2_at_least((hs4 + wpl - 1) / wpl);
#ifndef L2_ATTN_ROW_LANE
#define L2_ATTN_ROW_LANE 1
#endif
    a.rl = L2_ATTN_ROW_LANE && head_size == 64 && (a.gq == 4 || a.gq == 8) && kStageFloats == 2 * 16 * 64;
    a.threads = kNWA * 32;
    const int wpr = a.rl ? a.gq / 4 : 1, nrg = kNWA / wpr;  // warps per ring, rings per CTA (as in the kernel)
    const int stg = a.rl ? kAttStagesRL : kAttStages;
    const size_t hdr = (8 * nrg * stg + 16 + 4 * (nrg * a.gq * 2 + a.gq * 2) + 127) / 128 * 128;
    a.smem = hdr + (size_t)nrg * stg * kStageFloats * 4 + (size_t)nrg * a.gq * hs4 * 16;
    if (a.rl) a.smem += (size_t)kNWA * (16 + 1) * 4 * 4;  // probabilities [head][row] and rescales per warp
    // the last CTA stages (max, sum) of every chunk and head in its ring
    a.max_chunks = nrg * stg * kStageFloats / (2 * a.gq);
    a.ok = a.lp <= 32 && a.gq <= 8 && head_size % 4 == 0 && 2 * head_size <= kStageFloats;
    return a;
}

int attn_ctas_per_sm(const AttnLaunch &a) {
    int n = 0;
    AttnFn fn = pick(a.lp, a.gq, a.rl);
    if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, a.threads, a.smem) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n < 1 ? 1 : n;
}

bool attn_cluster_fits(const AttnLaunch &a, int n_chunks, int clusters) {
    AttnFn fn = pick(a.lp, a.gq, a.rl);
    if (!fn || n_chunks < 2 || n_chunks > 8) return false;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_chunks, clusters, 1);
    cfg.blockDim = dim3(a.threads);
    cfg.dynamicSmemBytes = a.smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)n_chunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n >= clusters;
}

cudaError_t attn_init() {
    static const int lps[] = {1, 2, 4, 8, 16, 32};
    static const int gqs[] = {1, 2, 4, 8};
    for (int lp : lps)
        for (int gq : gqs) {
            cudaError_t e = cudaFuncSetAttribute(pick(lp, gq, 0), cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
            if (e != cudaSuccess) return e;
        }
    for (int gq : {4, 8}) {
        cudaError_t e = cudaFuncSetAttribute(pick(16, gq, 1), cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_attn(const AttnLaunch &a, const AttnParams &p, int batch, cudaStream_t stream, bool pdl) {
    AttnFn fn = pick(a.lp, a.gq, a.rl);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_chunks, p.n_kv_heads, batch);
    cfg.blockDim = dim3(a.threads);
    cfg.dynamicSmemBytes = a.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)(p.cluster > 1 ? p.cluster : 1);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.cluster > 1 ? 2 : 1;
    void *args[] = {const_cast<AttnParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(fn), args);
}

}  // namespace l2
