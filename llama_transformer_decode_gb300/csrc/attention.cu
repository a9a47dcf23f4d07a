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
// of K and one of V; each warp streams a sub-slice through a private ring of
// 1-D bulk async copies (TMA).  Lanes are grouped LP to a cache row (LP = the
// head size in 16-byte words, rounded up to a power of two); each group keeps
// an online softmax (running max m, sum l, un-normalised accumulator) per
// query head; with 4 or 8 query heads per KV head at head size 64 the lanes
// take one cache row each instead (the row-per-lane layout, described at the
// kernel).  Groups, then warps, then CTAs are merged with the usual
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
// Row-per-lane layout: packed fp32 FMAs (two per instruction) for the scores and
// the weighted V sums.
#ifndef L2_ATTN_FFMA2
#define L2_ATTN_FFMA2 1
#endif
// Row-per-lane layout: two to four warps share a ring, so a CTA has fewer rings;
// deeper rings keep as many bytes in flight per SM.
constexpr int kAttStagesRL = 4;

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

// RL = 1: the row-per-lane layout for 4 or 8 query heads per KV head and
// head size 64 (16 cache rows per ring stage).  Two warps share each ring and
// split the group's query heads between them (so a CTA needs half the ring
// memory per warp and two CTAs fit on an SM).  Lane (t, half) of a warp
// scores row t for half of that warp's heads over the whole head (K chunks
// read in a lane-rotated order, conflict-free), the online softmax runs over
// the 16 rows with shuffles inside each half-warp (one exponential per row and
// head), and the probabilities go through shared memory to the PV pass, where
// lane l accumulates dimensions 2l, 2l+1 of the warp's heads.  Each cache row
// costs a few dozen instructions instead of one shuffle tree per head.
template <int LP, int GQ, int RL>
__global__ void __launch_bounds__(kNWA * 32) attn_kernel(const AttnParams p) {
    constexpr int NT = kNWA * 32;
    constexpr int RPI = 32 / LP;        // cache rows a warp handles at once
    constexpr int WPR = RL ? GQ / 2 : 1;  // warps sharing one ring (row-per-lane: two heads per warp)
    constexpr int NRG = kNWA / WPR;     // rings per CTA (one softmax state per ring and head)
    constexpr int STG = RL ? kAttStagesRL : kAttStages;  // ring buffers per ring
    static_assert(!RL || NRG <= 4, "ring barriers are ids 1..4");
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                      // [NRG][STG]
    int *flags = reinterpret_cast<int *>(smem + 8 * NRG * STG);        // [4]
    float *mrg = reinterpret_cast<float *>(smem + 8 * NRG * STG + 16); // [NRG][GQ][2]
    float *fin = mrg + NRG * GQ * 2;                                          // [GQ][2]
    const size_t hdr = (8 * NRG * STG + 16 + 4 * (NRG * GQ * 2 + GQ * 2) + 127) / 128 * 128;
    const int hs = p.head_size, hs4 = hs >> 2;
    float4 *ring = reinterpret_cast<float4 *>(smem + hdr);                     // [NRG][STG][stage]
    float4 *accs = ring + NRG * STG * (kStageFloats / 4);              // [NRG][GQ][hs4]
    float *qs = reinterpret_cast<float *>(accs + NRG * GQ * hs4);               // RL: [GQ][hs]
    float *pbuf = qs + GQ * hs;                                                 // RL: [kNWA][16 + 1][GQ / WPR]

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
    if (c >= n_active) return;  // too few positions for this CTA to join

    const int H = p.n_heads, KV = p.n_kv_heads;
    const int h0 = (g * H + KV - 1) / KV, h1 = ((g + 1) * H + KV - 1) / KV;
    const int nq = h1 - h0;

    const int t0 = (int)((long long)c * P / n_active), t1 = (int)((long long)(c + 1) * P / n_active);
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
        constexpr int TPR = 16;            // cache rows per ring stage (head size 64)
        constexpr int HS4 = 16;
        constexpr int HPW = GQ / WPR;      // heads per warp: 2
        constexpr int HPL = HPW / 2;       // heads per lane: 1 (one half-warp each)
        constexpr int RTH = WPR * 32;      // threads of one ring
        static_assert(HPL == 1, "row-per-lane attention: one head per half-warp");
        // the group's query vectors, shared by all warps
        for (int i = tid; i < GQ * 64; i += NT) {
            const int j = i / 64, d = i % 64;
            const size_t qi = (size_t)b * p.dim + (size_t)(h0 + j) * 64 + d;
            qs[i] = j < nq && in_bounds(qi, 1, p.ext->q, p.err) ? p.q[qi] : 0.f;
        }
        __syncthreads();
        const float4 *qs4 = reinterpret_cast<const float4 *>(qs);
        float *wp = pbuf + warp * (TPR + 1) * HPW;  // [TPR][HPW] probabilities, then [HPW] rescales
        const int t = lane & (TPR - 1), jh = lane / TPR;
        const int jw0 = wsub * HPW;                 // the warp's first head of the group
        // this lane's head's query vector in registers, its 16-byte chunks in the lane's
        // rotated order (chunk i of the loop below is chunk (i + t) % 16 of the head)
        float4 qr[HS4];
#pragma unroll
        for (int i = 0; i < HS4; ++i) qr[i] = qs4[(jw0 + jh) * HS4 + ((i + t) & (HS4 - 1))];
        float m[HPL], l[HPL];
        float acc[HPW][2];
#pragma unroll
        for (int jj = 0; jj < HPL; ++jj) {
            m[jj] = -CUDART_INF_F;
            l[jj] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < HPW; ++j) acc[j][0] = acc[j][1] = 0.f;
        int tc = wt0;
#pragma unroll 1
        for (; tc < wt1; ++k) {
            const int s = k % STG;
            const int np = min(TP, wt1 - tc);
            const bool got = mbar_wait(&wbars[s], (uint32_t)(k / STG) & 1u, p.err);
            // the ring's warps take one decision (the loop bounds are the ring's, so both get here)
            if (ring_sync_or<RTH>(!got, rgi)) {
                ok = false;
                break;
            }
            const float4 *Ks = wring + (size_t)s * (kStageFloats / 4);
            const float2 *Vs2 = reinterpret_cast<const float2 *>(Ks + (size_t)TP * HS4);
            // scores of row t for heads jw0 + jh*HPL.., the row's 16-byte chunks in rotated order
            const bool row_on = t < np;
            float sc[HPL];
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) sc[jj] = 0.f;
            if (row_on) {
                const float4 *Kr = Ks + t * HS4;
#if L2_ATTN_FFMA2
                // even and odd dimensions in the two halves of packed fp32 FMAs
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int i = 0; i < HS4; ++i) {
                    const float4 kv = Kr[(i + t) & (HS4 - 1)];
                    s2 = ffma2(make_float2(qr[i].x, qr[i].y), make_float2(kv.x, kv.y), s2);
                    s2 = ffma2(make_float2(qr[i].z, qr[i].w), make_float2(kv.z, kv.w), s2);
                }
                sc[0] = s2.x + s2.y;
#else
#pragma unroll
                for (int i = 0; i < HS4; ++i) sc[0] = dot4(qr[i], Kr[(i + t) & (HS4 - 1)], sc[0]);
#endif
            }
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) {
                const int hj = jw0 + jh * HPL + jj;
                sc[jj] = row_on ? sc[jj] * p.scale : -CUDART_INF_F;
                if (dbg && row_on && hj < nq) dbg[(size_t)hj * p.seq_len + tc + t] = sc[jj];
                // online softmax over the stage's rows (the 16 lanes of this half)
                float mx = sc[jj];
#pragma unroll
                for (int o = TPR / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = fmaxf(m[jj], mx);  // finite: row 0 of the stage is valid
                const float corr = expf(m[jj] - mn);
                const float pe = expf(sc[jj] - mn);
                float ps = pe;
#pragma unroll
                for (int o = TPR / 2; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                l[jj] = l[jj] * corr + ps;
                m[jj] = mn;
                wp[t * HPW + jh * HPL + jj] = pe;
                if (t == 0) wp[TPR * HPW + jh * HPL + jj] = corr;
            }
            __syncwarp();
            // PV: dimensions 2 lane, 2 lane + 1 of the warp's heads
#pragma unroll
            for (int j = 0; j < HPW; ++j) {
                const float cr = wp[TPR * HPW + j];
                acc[j][0] *= cr;
                acc[j][1] *= cr;
            }
#pragma unroll 4
            for (int tt = 0; tt < np; ++tt) {
                const float2 v = Vs2[tt * 32 + lane];
                const float2 pp = *reinterpret_cast<const float2 *>(wp + tt * HPW);  // the warp's two heads
#if L2_ATTN_FFMA2
                const float2 a0 = ffma2(make_float2(pp.x, pp.x), v, make_float2(acc[0][0], acc[0][1]));
                const float2 a1 = ffma2(make_float2(pp.y, pp.y), v, make_float2(acc[1][0], acc[1][1]));
                acc[0][0] = a0.x;
                acc[0][1] = a0.y;
                acc[1][0] = a1.x;
                acc[1][1] = a1.y;
#else
                acc[0][0] = fmaf(pp.x, v.x, acc[0][0]);
                acc[0][1] = fmaf(pp.x, v.y, acc[0][1]);
                acc[1][0] = fmaf(pp.y, v.x, acc[1][0]);
                acc[1][1] = fmaf(pp.y, v.y, acc[1][1]);
#endif
            }
            __syncwarp();
            tc += np;
            ring_sync<RTH>(rgi);  // both warps are done with this stage's buffer
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
        if (t == 0) {
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) {
                mrg[(rgi * GQ + jw0 + jh * HPL + jj) * 2 + 0] = m[jj];
                mrg[(rgi * GQ + jw0 + jh * HPL + jj) * 2 + 1] = l[jj];
            }
        }
        float *accf = reinterpret_cast<float *>(accs);
#pragma unroll
        for (int j = 0; j < HPW; ++j)
            *reinterpret_cast<float2 *>(accf + (size_t)(rgi * GQ + jw0 + j) * 64 + 2 * lane) =
                make_float2(acc[j][0], acc[j][1]);
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

    // last CTA of the group: merge the chunks in chunk order
    if (!in_bounds(((size_t)b * H + h0 + nq - 1) * NC + n_active - 1, 1, p.ext->ws_rows, p.err)) return;
    if (tid < nq) {
        const int j = tid;
        float M = -CUDART_INF_F;
        for (int cc = 0; cc < n_active; ++cc)
            M = fmaxf(M, __ldcg(p.ws_ml + (((size_t)b * H + h0 + j) * NC + cc) * 2));
        float L = 0.f;
        for (int cc = 0; cc < n_active; ++cc) {
            const size_t sl = ((size_t)b * H + h0 + j) * NC + cc;
            L += __ldcg(p.ws_ml + sl * 2 + 1) * expf(__ldcg(p.ws_ml + sl * 2) - M);
        }
        fin[j * 2] = M;
        fin[j * 2 + 1] = L;
    }
    __syncthreads();
    for (int idx = tid; idx < nq * hs4; idx += NT) {
        const int j = idx / hs4, w4 = idx % hs4;
        const float M = fin[j * 2], inv = 1.0f / fin[j * 2 + 1];
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cc = 0; cc < n_active; ++cc) {
            const size_t sl = ((size_t)b * H + h0 + j) * NC + cc;
            const float e = expf(__ldcg(p.ws_ml + sl * 2) - M);
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + sl * hs) + w4);
            o.x += a.x * e;
            o.y += a.y * e;
            o.z += a.z * e;
            o.w += a.w * e;
        }
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
        if (in_bounds((size_t)b * p.dim + (size_t)(h0 + j) * hs + 4 * w4, 4, p.ext->xb, p.err))
            reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] = o;
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
typedef void (*AttnFn)(const AttnParams);

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
    const int wpr = a.rl ? a.gq / 2 : 1, nrg = kNWA / wpr;  // warps per ring, rings per CTA (as in the kernel)
    const int stg = a.rl ? kAttStagesRL : kAttStages;
    const size_t hdr = (8 * nrg * stg + 16 + 4 * (nrg * a.gq * 2 + a.gq * 2) + 127) / 128 * 128;
    a.smem = hdr + (size_t)nrg * stg * kStageFloats * 4 + (size_t)nrg * a.gq * hs4 * 16;
    if (a.rl) a.smem += (size_t)a.gq * head_size * 4 + (size_t)kNWA * 17 * (a.gq / wpr) * 4;  // query vectors, probabilities
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<AttnParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(fn), args);
}

}  // namespace l2
