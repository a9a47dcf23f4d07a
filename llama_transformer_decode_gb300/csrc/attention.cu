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
constexpr int kPPG = 4;              // positions a lane group scores before one softmax update

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
// head size 64 (16 cache rows per ring stage).  Lane (t, half) scores row t
// for half of the group's heads over the whole head (K chunks read in a
// lane-rotated order, conflict-free), the online softmax runs over the 16
// rows with shuffles inside each half-warp (one exponential per row and
// head), and the probabilities go through shared memory to the PV pass,
// where lane l accumulates dimensions 2l, 2l+1 of every head.  Each cache row
// costs a few dozen instructions instead of one shuffle tree per head.
template <int LP, int GQ, int RL>
__global__ void __launch_bounds__(kNWA * 32) attn_kernel(const AttnParams p) {
    constexpr int NT = kNWA * 32;
    constexpr int RPI = 32 / LP;  // cache rows a warp handles at once
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);                      // [kNWA][kAttStages]
    int *flags = reinterpret_cast<int *>(smem + 8 * kNWA * kAttStages);        // [4]
    float *mrg = reinterpret_cast<float *>(smem + 8 * kNWA * kAttStages + 16); // [kNWA][GQ][2]
    float *fin = mrg + kNWA * GQ * 2;                                          // [GQ][2]
    const size_t hdr = (8 * kNWA * kAttStages + 16 + 4 * (kNWA * GQ * 2 + GQ * 2) + 127) / 128 * 128;
    const int hs = p.head_size, hs4 = hs >> 2;
    float4 *ring = reinterpret_cast<float4 *>(smem + hdr);                     // [kNWA][kAttStages][stage]
    float4 *accs = ring + kNWA * kAttStages * (kStageFloats / 4);              // [kNWA][GQ][hs4]
    float *qs = reinterpret_cast<float *>(accs + kNWA * GQ * hs4);               // RL: [GQ][hs]
    float *pbuf = qs + GQ * hs;                                                 // RL: [kNWA][16 + 1][GQ]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int pos = p.step->pos[b];
    const int P = pos + 1;
    int chunk = p.min_chunk;
    if (p.capacity > 0) {
        // spread the positions of every row over the resident CTAs (the host sums them)
        const long long total = p.step->attn_total;
        const long long per = (total * p.n_kv_heads + p.capacity - 1) / p.capacity;
        if (per > chunk) chunk = (int)per;
    }
    int n_active = (P + chunk - 1) / chunk;
    if (n_active > p.n_chunks) n_active = p.n_chunks;
    if (c >= n_active) return;  // too few positions for this CTA to join

    const int H = p.n_heads, KV = p.n_kv_heads;
    const int h0 = (g * H + KV - 1) / KV, h1 = ((g + 1) * H + KV - 1) / KV;
    const int nq = h1 - h0;

    const int t0 = (int)((long long)c * P / n_active), t1 = (int)((long long)(c + 1) * P / n_active);
    const int wt0 = t0 + (int)((long long)(t1 - t0) * warp / kNWA);
    const int wt1 = t0 + (int)((long long)(t1 - t0) * (warp + 1) / kNWA);
    const int TP = kStageFloats / (2 * hs);  // positions per stage

    const size_t head_base = (((size_t)p.step->slot[b] * p.n_layers + p.layer) * KV + g) * (size_t)p.seq_len * hs;
    const float *kbase = p.kcache + head_base;
    const float *vbase = p.vcache + head_base;

    if (tid == 0) {
        for (int i = 0; i < kNWA * kAttStages; ++i) mbar_init(&bars[i], 1);
        fence_barrier_init();
        flags[0] = 0;  // a warp gave up waiting
        flags[1] = 0;  // this CTA merges the chunks
    }
    __syncthreads();

    uint64_t *wbars = bars + warp * kAttStages;
    float4 *wring = ring + (size_t)warp * kAttStages * (kStageFloats / 4);
    int ti = wt0;  // next position to request
    int n_issued = 0;
    auto issue = [&](int stage) {
        const int np = min(TP, wt1 - ti);
        if (lane == 0) {
            const uint32_t bytes = (uint32_t)np * hs * 4u;
            float4 *dst = wring + (size_t)stage * (kStageFloats / 4);
            mbar_arrive_expect_tx(&wbars[stage], 2u * bytes);
            bulk_g2s_nohint(dst, kbase + (size_t)ti * hs, bytes, &wbars[stage]);
            bulk_g2s_nohint(dst + (size_t)TP * hs4, vbase + (size_t)ti * hs, bytes, &wbars[stage]);
        }
        ti += np;
        ++n_issued;
    };
    // Rows before stable[b] (pos for an ordinary step, the chunk's first
    // position in a prefill) are not written during this step: fetch them
    // before the previous kernel (which writes the newer rows) has finished.
    const int stable = p.step->stable[b];
#pragma unroll 1
    for (int s = 0; s < kAttStages && ti < wt1 && ti + min(TP, wt1 - ti) <= stable; ++s) issue(s);
    pdl_launch_dependents();
    pdl_wait();
#pragma unroll 1
    for (int s = n_issued; s < kAttStages && ti < wt1; ++s) issue(s);

    bool ok = true;
    int k = 0;
    float *dbg = p.dbg ? p.dbg + (((size_t)b * p.n_layers + p.layer) * H + h0) * p.seq_len : nullptr;
    if constexpr (RL == 1) {
        constexpr int TPR = 16;            // cache rows per ring stage (head size 64)
        constexpr int HS4 = 16;
        constexpr int HPL = GQ / 2;        // heads per lane
        // the group's query vectors, shared by all warps
        for (int i = tid; i < GQ * 64; i += NT) {
            const int j = i / 64, d = i % 64;
            qs[i] = j < nq ? p.q[(size_t)b * p.dim + (size_t)(h0 + j) * 64 + d] : 0.f;
        }
        __syncthreads();
        const float4 *qs4 = reinterpret_cast<const float4 *>(qs);
        float *wp = pbuf + warp * (TPR + 1) * GQ;  // [TPR][GQ] probabilities, then [GQ] rescales
        const int t = lane & (TPR - 1), jh = lane / TPR;
        float m[HPL], l[HPL];
        float acc[GQ][2];
#pragma unroll
        for (int jj = 0; jj < HPL; ++jj) {
            m[jj] = -CUDART_INF_F;
            l[jj] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < GQ; ++j) acc[j][0] = acc[j][1] = 0.f;
        int tc = wt0;
#pragma unroll 1
        for (; tc < wt1; ++k) {
            const int s = k % kAttStages;
            const int np = min(TP, wt1 - tc);
            if (!mbar_wait(&wbars[s], (uint32_t)(k / kAttStages) & 1u, p.err)) {
                ok = false;
                break;
            }
            const float4 *Ks = wring + (size_t)s * (kStageFloats / 4);
            const float2 *Vs2 = reinterpret_cast<const float2 *>(Ks + (size_t)TP * HS4);
            // scores of row t for heads jh*HPL.., the row's 16-byte chunks in rotated order
            const bool row_on = t < np;
            float sc[HPL];
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) sc[jj] = 0.f;
            if (row_on) {
                const float4 *Kr = Ks + t * HS4;
#pragma unroll
                for (int i = 0; i < HS4; ++i) {
                    const int ch = (i + t) & (HS4 - 1);
                    const float4 kv = Kr[ch];
#pragma unroll
                    for (int jj = 0; jj < HPL; ++jj) sc[jj] = dot4(qs4[(jh * HPL + jj) * HS4 + ch], kv, sc[jj]);
                }
            }
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) {
                sc[jj] = row_on ? sc[jj] * p.scale : -CUDART_INF_F;
                if (dbg && row_on && jh * HPL + jj < nq) dbg[(size_t)(jh * HPL + jj) * p.seq_len + tc + t] = sc[jj];
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
                wp[t * GQ + jh * HPL + jj] = pe;
                if (t == 0) wp[TPR * GQ + jh * HPL + jj] = corr;
            }
            __syncwarp();
            // PV: dimensions 2 lane, 2 lane + 1 of every head
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                const float c = wp[TPR * GQ + j];
                acc[j][0] *= c;
                acc[j][1] *= c;
            }
#pragma unroll 4
            for (int tt = 0; tt < np; ++tt) {
                const float2 v = Vs2[tt * 32 + lane];
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    const float pj = wp[tt * GQ + j];
                    acc[j][0] = fmaf(pj, v.x, acc[j][0]);
                    acc[j][1] = fmaf(pj, v.y, acc[j][1]);
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
                (void)mbar_wait(&wbars[j % kAttStages], (uint32_t)(j / kAttStages) & 1u, p.err);
            if (lane == 0) flags[0] = 1;
        }
        if (t == 0) {
#pragma unroll
            for (int jj = 0; jj < HPL; ++jj) {
                mrg[(warp * GQ + jh * HPL + jj) * 2 + 0] = m[jj];
                mrg[(warp * GQ + jh * HPL + jj) * 2 + 1] = l[jj];
            }
        }
        float *accf = reinterpret_cast<float *>(accs);
#pragma unroll
        for (int j = 0; j < GQ; ++j)
            *reinterpret_cast<float2 *>(accf + (size_t)(warp * GQ + j) * 64 + 2 * lane) = make_float2(acc[j][0], acc[j][1]);
    } else {
        // query vectors of the group, one 16-byte word per lane and head
        const int rg = lane / LP, c4 = lane % LP;
        const bool lane_on = c4 < hs4;
        float4 q4[GQ];
        float m[GQ], l[GQ];
        float4 acc[GQ];
    #pragma unroll
        for (int j = 0; j < GQ; ++j) {
            q4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < nq && lane_on)
                q4[j] = reinterpret_cast<const float4 *>(p.q + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[c4];
            m[j] = -CUDART_INF_F;
            l[j] = 0.f;
            acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        int tc = wt0;
    #pragma unroll 1
        for (; tc < wt1; ++k) {
            const int s = k % kAttStages;
            const int np = min(TP, wt1 - tc);
            if (!mbar_wait(&wbars[s], (uint32_t)(k / kAttStages) & 1u, p.err)) {
                ok = false;
                break;
            }
            const float4 *Ks = wring + (size_t)s * (kStageFloats / 4);
            const float4 *Vs = Ks + (size_t)TP * hs4;
    #pragma unroll 1
            // Up to kPPG positions per lane group at a time: all their scores
            // first (independent dot products and shuffles), then one online-
            // softmax update per head (one rescale per group of positions).
            for (int tt = 0; tt < np; tt += RPI * kPPG) {
                float sc[kPPG][GQ];
                float4 vv[kPPG];
    #pragma unroll
                for (int u = 0; u < kPPG; ++u) {
                    const int tl = tt + u * RPI + rg;
                    const bool row_on = tl < np;
                    float4 kv = make_float4(0.f, 0.f, 0.f, 0.f);
                    vv[u] = kv;
                    if (row_on && lane_on) {
                        kv = Ks[tl * hs4 + c4];
                        vv[u] = Vs[tl * hs4 + c4];
                    }
    #pragma unroll
                    for (int j = 0; j < GQ; ++j) {
                        float d = dot4(q4[j], kv, 0.f);
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
                    for (int u = 1; u < kPPG; ++u) mx = fmaxf(mx, sc[u][j]);
                    const float mn = fmaxf(m[j], mx);
                    if (mn == -CUDART_INF_F) continue;  // no position of this group
                    const float corr = expf(m[j] - mn);
                    float ps = 0.f;
                    float4 a = make_float4(acc[j].x * corr, acc[j].y * corr, acc[j].z * corr, acc[j].w * corr);
    #pragma unroll
                    for (int u = 0; u < kPPG; ++u) {
                        const float pe = expf(sc[u][j] - mn);
                        ps += pe;
                        a.x = fmaf(pe, vv[u].x, a.x);
                        a.y = fmaf(pe, vv[u].y, a.y);
                        a.z = fmaf(pe, vv[u].z, a.z);
                        a.w = fmaf(pe, vv[u].w, a.w);
                    }
                    l[j] = l[j] * corr + ps;
                    acc[j] = a;
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
                (void)mbar_wait(&wbars[j % kAttStages], (uint32_t)(j / kAttStages) & 1u, p.err);
            if (lane == 0) flags[0] = 1;
        }

        // merge the row groups of the warp (lanes LP apart share a column word)
    #pragma unroll
        for (int o = LP; o < 32; o <<= 1) {
    #pragma unroll
            for (int j = 0; j < GQ; ++j) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m[j], o);
                const float l2v = __shfl_xor_sync(0xffffffffu, l[j], o);
                float4 a2;
                a2.x = __shfl_xor_sync(0xffffffffu, acc[j].x, o);
                a2.y = __shfl_xor_sync(0xffffffffu, acc[j].y, o);
                a2.z = __shfl_xor_sync(0xffffffffu, acc[j].z, o);
                a2.w = __shfl_xor_sync(0xffffffffu, acc[j].w, o);
                merge_state(m[j], l[j], acc[j], m2, l2v, a2);
            }
        }
        if (lane < LP) {
    #pragma unroll
            for (int j = 0; j < GQ; ++j) {
                if (lane == 0) {
                    mrg[(warp * GQ + j) * 2 + 0] = m[j];
                    mrg[(warp * GQ + j) * 2 + 1] = l[j];
                }
                if (lane_on) accs[(size_t)(warp * GQ + j) * hs4 + c4] = acc[j];
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
            for (int w = 0; w < kNWA; ++w)
                merge_state(mm, ll, aa, mrg[(w * GQ + j) * 2], mrg[(w * GQ + j) * 2 + 1],
                            accs[(size_t)(w * GQ + j) * hs4 + w4]);
            const float inv = 1.0f / ll;
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
        for (int w = 0; w < kNWA; ++w)
            merge_state(mm, ll, aa, mrg[(w * GQ + j) * 2], mrg[(w * GQ + j) * 2 + 1], accs[(size_t)(w * GQ + j) * hs4 + w4]);
        const size_t slot = ((size_t)b * H + h0 + j) * NC + c;
        reinterpret_cast<float4 *>(p.ws_acc + slot * hs)[w4] = aa;
        if (w4 == 0) {
            p.ws_ml[slot * 2 + 0] = mm;
            p.ws_ml[slot * 2 + 1] = ll;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const unsigned t = atomicAdd(&p.tickets[b * KV + g], 1u);
        flags[1] = (t == (unsigned)(n_active - 1)) ? 1 : 0;
    }
    __syncthreads();
    if (!flags[1]) return;
    __threadfence();

    // last CTA of the group: merge the chunks in chunk order
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
        reinterpret_cast<float4 *>(p.out + (size_t)b * p.dim + (size_t)(h0 + j) * hs)[w4] = o;
    }
    if (dbg) {
        for (int idx = tid; idx < nq * P; idx += NT) {
            const int j = idx / P, t = idx % P;
            float *cell = dbg + (size_t)j * p.seq_len + t;
            *cell = expf(__ldcg(cell) - fin[j * 2]) / fin[j * 2 + 1];
        }
    }
    if (tid == 0) p.tickets[b * KV + g] = 0u;
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
    a.lp = pow2_at_least(hs4);
    a.gq = pow2_at_least(max_group);
#ifndef L2_ATTN_ROW_LANE
#define L2_ATTN_ROW_LANE 1
#endif
    a.rl = L2_ATTN_ROW_LANE && head_size == 64 && (a.gq == 4 || a.gq == 8) && kStageFloats == 2 * 16 * 64;
    a.threads = kNWA * 32;
    const size_t hdr = (8 * kNWA * kAttStages + 16 + 4 * (kNWA * a.gq * 2 + a.gq * 2) + 127) / 128 * 128;
    a.smem = hdr + (size_t)kNWA * kAttStages * kStageFloats * 4 + (size_t)kNWA * a.gq * hs4 * 16;
    if (a.rl) a.smem += (size_t)a.gq * head_size * 4 + (size_t)kNWA * 17 * a.gq * 4;  // query vectors, probabilities
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
