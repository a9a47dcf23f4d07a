// The whole batch-1 decode step of a small model in one thread block.
//
// What it computes: llama2.c's forward(token, pos) ("run.c 逐行解讀", §4
// forward(), steps 1-3; "run.c", transformer()): the embedding row, then per
// layer RMSNorm, the Q/K/V matmuls, RoPE, K and V written into the cache at
// pos, causal attention of every query head h over cache rows 0..pos of KV
// head g(h) = floor(h * n_kv_heads / n_heads), the output matmul and residual,
// RMSNorm, W1/W3 with SwiGLU, W2 and residual; then the final RMSNorm and the
// classifier.
//
// Why one block.  For a model whose weights sit in L2 (a few MB), the step
// launched as one kernel per matrix product is bound by the cost of each
// kernel boundary (about 3.7 us each, 5 per layer), not by bytes.  Here the
// phases are separated by __syncthreads instead: the activations (x, the
// normalised x, q, the attention output, the hidden vector) and the attention
// scores live in shared memory with every RMSNorm gain (loaded once), and 32
// warps read the weights straight from L2 with 16-byte loads.  A matrix
// product gives each output row to a group of G lanes (G the smallest power
// of two covering the row's 16-byte words, at most 32), so short rows still
// keep every lane busy; each group reduces its row by shuffles and one lane
// writes the result.  With head size <= 16 the attention of a head (scores,
// softmax, weighted V sum) runs inside one warp, lanes over positions, with no
// block barrier until all heads are done; larger heads take three block-wide
// phases.  Each phase costs about one L2 round trip and one barrier (0.3-2 us
// per phase measured on GB300), which is what bounds the step.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kCT = 1024;      // threads
constexpr int kCW = kCT / 32;  // warps
static_assert(kCW == 32, "cta_sum adds one partial per lane of a warp");

__host__ __device__ constexpr int align4(int n) { return (n + 3) & ~3; }

// Shared-memory layout (floats, every region 16-byte aligned).
struct CtaLayout {
    int gain, x, xn, q, att, kn, vn, hb, sc, part, red, total;
    __host__ __device__ CtaLayout(int dim, int hidden, int kv_dim, int n_heads, int seq_len, int n_layers) {
        gain = 0;                                  // every RMSNorm gain: [layer][att, ffn], final
        x = gain + align4((2 * n_layers + 1) * dim);
        xn = x + align4(dim);
        q = xn + align4(dim);
        att = q + align4(dim);
        kn = att + align4(dim);
        vn = kn + align4(kv_dim);
        hb = vn + align4(kv_dim);
        sc = hb + align4(hidden);                   // scores [n_heads][pos + 1]
        part = sc + align4(n_heads * seq_len);      // weighted-V partial sums
        red = part + align4(dim > kCT ? dim : kCT);  // one float per warp
        total = red + kCW;
    }
};

// Sum over the block, the same value in every thread: the warps' partials are
// added by one shuffle tree (the same order in every warp).
__device__ __forceinline__ float cta_sum(float v, float *red) {
    v = warp_sum(v);
    __syncthreads();  // red is free
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    return warp_sum(red[threadIdx.x & 31]);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// out = gain * (x / rms(x)), the RMSNorm of "run.c" rmsnorm() (eps 1e-5); gain in shared memory.
__device__ void cta_rmsnorm(const float *x, const float *gain, float *out, int n, float *red) {
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += kCT) ss = fmaf(x[i], x[i], ss);
    const float inv = 1.0f / sqrtf(cta_sum(ss, red) / (float)n + 1e-5f);
    for (int i = threadIdx.x; i < n; i += kCT) out[i] = gain[i] * (inv * x[i]);
    __syncthreads();
}

// Rows 0..R-1 of NM matrices of row length n (a multiple of 4) times v (shared
// memory): row(m, r) gives row r of matrix m, out(r, y) receives the NM dot
// products of row r (called by one lane per row).  The caller synchronises.
template <int NM, typename RowFn, typename OutFn>
__device__ void cta_gemv(int n, int R, const float *v, RowFn row, OutFn out) {
    const int n4 = n >> 2;
    const int G = n4 >= 32 ? 32 : n4 >= 16 ? 16 : n4 >= 8 ? 8 : n4 >= 4 ? 4 : n4 >= 2 ? 2 : 1;
    const int RPW = 32 / G;  // rows a warp takes at once
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane / G, gl = lane - sub * G;
    const float4 *v4 = reinterpret_cast<const float4 *>(v);
#pragma unroll 2
    for (int r0 = warp * RPW; r0 < R; r0 += kCW * RPW) {
        const int r = r0 + sub;
        float acc[NM];
#pragma unroll
        for (int m = 0; m < NM; ++m) acc[m] = 0.f;
        if (r < R) {
            const float4 *w4[NM];
#pragma unroll
            for (int m = 0; m < NM; ++m) w4[m] = reinterpret_cast<const float4 *>(row(m, r));
            for (int i = gl; i < n4; i += G) {
                const float4 x = v4[i];
#pragma unroll
                for (int m = 0; m < NM; ++m) acc[m] = dot4(__ldg(w4[m] + i), x, acc[m]);
            }
        }
        for (int o = G >> 1; o > 0; o >>= 1)
#pragma unroll
            for (int m = 0; m < NM; ++m) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
        if (gl == 0 && r < R) out(r, acc);
    }
}

}  // namespace

__global__ void __launch_bounds__(kCT, 1) l2dec_step_cta_kernel(const CtaStepParams p) {
    extern __shared__ __align__(16) float sm[];
    const int dim = p.dim, hidden = p.hidden_dim, kvd = p.kv_dim, hs = p.head_size, H = p.n_heads, KV = p.n_kv_heads;
    const int S = p.seq_len, half = hs >> 1;
    const CtaLayout ly(dim, hidden, kvd, H, S, p.n_layers);
    float *gains = sm + ly.gain;
    float *x = sm + ly.x, *xn = sm + ly.xn, *q = sm + ly.q, *att = sm + ly.att, *kn = sm + ly.kn, *vn = sm + ly.vn;
    float *hb = sm + ly.hb, *sc = sm + ly.sc, *part = sm + ly.part, *red = sm + ly.red;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int token = p.step->token[0], pos = p.step->pos[0], P = pos + 1;
    const float2 *rr = p.rope + (size_t)pos * half;

    // step 1: x = the token's embedding row; every RMSNorm gain into shared memory
    {
        const size_t e0 = (size_t)token * dim;
        const bool ok = in_bounds(e0, (size_t)dim, p.ext->emb, p.err);
        for (int i = tid; i < dim; i += kCT) x[i] = ok ? p.emb[e0 + i] : 0.f;
        const int ld = p.n_layers * dim;
        for (int i = tid; i < 2 * ld + dim; i += kCT) {
            const int l = i / (2 * dim), r = i - l * 2 * dim;
            gains[i] = i >= 2 * ld ? __ldg(p.rms_final + (i - 2 * ld))
                                   : __ldg((r < dim ? p.rms_att : p.rms_ffn) + (size_t)l * dim + (r < dim ? r : r - dim));
        }
    }
    __syncthreads();

    for (int l = 0; l < p.n_layers; ++l) {
        // 2a: attention RMSNorm
        cta_rmsnorm(x, gains + (size_t)l * 2 * dim, xn, dim, red);

        // 2b-2c: q, k, v = Wq xn, Wk xn, Wv xn (rows of the three matrices stacked)
        const float *wq = p.wq + (size_t)l * dim * dim, *wk = p.wk + (size_t)l * kvd * dim,
                    *wv = p.wv + (size_t)l * kvd * dim;
        const float *wo = p.wo + (size_t)l * dim * dim;
        const float *w1 = p.w1 + (size_t)l * hidden * dim, *w3 = p.w3 + (size_t)l * hidden * dim;
        const float *w2 = p.w2 + (size_t)l * dim * hidden;
        cta_gemv<1>(
            dim, dim + 2 * kvd, xn,
            [&](int, int r) {
                return r < dim ? wq + (size_t)r * dim : r < dim + kvd ? wk + (size_t)(r - dim) * dim
                                                                       : wv + (size_t)(r - dim - kvd) * dim;
            },
            [&](int r, const float *y) {
                if (r < dim) q[r] = y[0];
                else if (r < dim + kvd) kn[r - dim] = y[0];
                else vn[r - dim - kvd] = y[0];
            });
        __syncthreads();

        // 2d: RoPE on the pairs of q and k; k and v into the cache row at pos
        const size_t lbase = (size_t)l * KV * S;  // this layer's first row (slot 0)
        for (int e = tid; e < (dim >> 1) + kvd; e += kCT) {
            if (e < (dim >> 1)) {
                const int v = 2 * e;
                const float2 cs = rr[(v % hs) >> 1];
                const float y0 = q[v], y1 = q[v + 1];
                q[v] = y0 * cs.x - y1 * cs.y;
                q[v + 1] = y0 * cs.y + y1 * cs.x;
            } else {
                const int c = 2 * (e - (dim >> 1));  // 0 .. 2 kv_dim: K pairs, then V pairs
                const bool is_k = c < kvd;
                const int cc = is_k ? c : c - kvd, g = cc / hs, d = cc % hs;
                const size_t idx = ((lbase + (size_t)g * S) + pos) * hs + d;
                if (!in_bounds(idx, 2, p.ext->cache, p.err)) continue;
                if (is_k) {
                    const float2 cs = rr[d >> 1];
                    const float y0 = kn[cc], y1 = kn[cc + 1];
                    p.kcache[idx] = y0 * cs.x - y1 * cs.y;
                    p.kcache[idx + 1] = y0 * cs.y + y1 * cs.x;
                } else {
                    p.vcache[idx] = vn[cc];
                    p.vcache[idx + 1] = vn[cc + 1];
                }
            }
        }
        __syncthreads();

        // 2e: attention of head h over cache rows t <= pos of KV head g(h): scores
        // q_h . K[t] / sqrt(head_size), softmax (subtract the maximum, exponentiate, divide
        // by the sum), out_h = sum_t p_t V[t].  The row at pos was just written by this
        // block: the cache is read through L2.
        const int hs4 = hs >> 2;
        if (hs <= 16) {
            // one warp per head, no block barrier inside: lanes take positions lane, lane + 32, ..
            for (int h = warp; h < H; h += kCW) {
                const int g = (int)((long long)h * KV / H);
                const size_t r0 = (lbase + (size_t)g * S) * hs;  // the head's cache row 0
                const bool okc = in_bounds(r0, (size_t)P * hs, p.ext->cache, p.err);
                const float4 *k4 = reinterpret_cast<const float4 *>(p.kcache + r0);
                const float4 *v4 = reinterpret_cast<const float4 *>(p.vcache + r0);
                const float4 *q4 = reinterpret_cast<const float4 *>(q + h * hs);
                float *s = sc + h * P;
                float mx = -CUDART_INF_F;
                for (int t = lane; t < P; t += 32) {
                    float d = 0.f;
                    if (okc)
                        for (int i = 0; i < hs4; ++i) d = dot4(__ldcg(k4 + (size_t)t * hs4 + i), q4[i], d);
                    d *= p.scale;
                    s[t] = d;
                    mx = fmaxf(mx, d);
                }
                mx = warp_max(mx);
                float sum = 0.f;
                for (int t = lane; t < P; t += 32) {
                    const float ex = expf(s[t] - mx);
                    s[t] = ex;
                    sum += ex;
                }
                sum = warp_sum(sum);
                float *dbg = p.dbg ? p.dbg + ((size_t)l * H + h) * S : nullptr;
                if (dbg && !in_bounds(((size_t)l * H + h) * S, (size_t)P, p.ext->dbg, p.err)) dbg = nullptr;
                float4 acc[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int t = lane; t < P; t += 32) {
                    const float pr = s[t] / sum;
                    if (dbg) dbg[t] = pr;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (i < hs4 && okc) {
                            const float4 v = __ldcg(v4 + (size_t)t * hs4 + i);
                            acc[i] = make_float4(fmaf(pr, v.x, acc[i].x), fmaf(pr, v.y, acc[i].y), fmaf(pr, v.z, acc[i].z),
                                                 fmaf(pr, v.w, acc[i].w));
                        }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < hs4) {
                        const float4 a = make_float4(warp_sum(acc[i].x), warp_sum(acc[i].y), warp_sum(acc[i].z),
                                                     warp_sum(acc[i].w));
                        if (lane == 0) reinterpret_cast<float4 *>(att + h * hs)[i] = a;
                    }
            }
            __syncthreads();
        } else {
            // scores, softmax and the weighted V sum as three block-wide phases
            for (int e = tid; e < H * P; e += kCT) {
                const int h = e / P, t = e - h * P;
                const int g = (int)((long long)h * KV / H);
                const size_t k0 = ((lbase + (size_t)g * S) + t) * hs;
                float d = 0.f;
                if (in_bounds(k0, (size_t)hs, p.ext->cache, p.err)) {
                    const float4 *k4 = reinterpret_cast<const float4 *>(p.kcache + k0);
                    const float4 *q4 = reinterpret_cast<const float4 *>(q + h * hs);
                    for (int i = 0; i < hs4; ++i) d = dot4(__ldcg(k4 + i), q4[i], d);
                }
                sc[h * P + t] = d * p.scale;
            }
            __syncthreads();
            // softmax over t per head: subtract the maximum, exponentiate, divide by the sum
            for (int h = warp; h < H; h += kCW) {
                float *s = sc + h * P;
                float mx = -CUDART_INF_F;
                for (int t = lane; t < P; t += 32) mx = fmaxf(mx, s[t]);
                mx = warp_max(mx);
                float sum = 0.f;
                for (int t = lane; t < P; t += 32) {
                    const float ex = expf(s[t] - mx);
                    s[t] = ex;
                    sum += ex;
                }
                sum = warp_sum(sum);
                float *dbg = p.dbg ? p.dbg + ((size_t)l * H + h) * S : nullptr;
                if (dbg && !in_bounds(((size_t)l * H + h) * S, (size_t)P, p.ext->dbg, p.err)) dbg = nullptr;
                for (int t = lane; t < P; t += 32) {
                    const float pr = s[t] / sum;
                    s[t] = pr;
                    if (dbg) dbg[t] = pr;
                }
            }
            __syncthreads();
            // out[h][d] = sum_t p[h][t] V[t, g(h)][d]: NP threads per output element split t
            const int NP = dim >= kCT ? 1 : kCT / dim;
            for (int e = tid; e < dim * NP; e += kCT) {
                const int i = e % dim, sp = e / dim;
                const int h = i / hs, d = i - h * hs, g = (int)((long long)h * KV / H);
                const size_t v0 = (lbase + (size_t)g * S) * hs + d;
                const float *ph = sc + h * P;
                float a = 0.f;
                if (in_bounds(v0 + (size_t)pos * hs, 1, p.ext->cache, p.err)) {
#pragma unroll 4
                    for (int t = sp; t < P; t += NP) a = fmaf(ph[t], __ldcg(p.vcache + v0 + (size_t)t * hs), a);
                }
                part[sp * dim + i] = a;
            }
            __syncthreads();
            for (int i = tid; i < dim; i += kCT) {
                float a = 0.f;
                for (int sp = 0; sp < NP; ++sp) a += part[sp * dim + i];
                att[i] = a;
            }
            __syncthreads();
        }

        // 2f: x += Wo att
        cta_gemv<1>(
            dim, dim, att, [&](int, int r) { return wo + (size_t)r * dim; }, [&](int r, const float *y) { x[r] += y[0]; });
        __syncthreads();

        // 2g: FFN RMSNorm, hb = silu(W1 xn) * (W3 xn)
        cta_rmsnorm(x, gains + (size_t)l * 2 * dim + dim, xn, dim, red);
        cta_gemv<2>(
            dim, hidden, xn, [&](int m, int r) { return (m ? w3 : w1) + (size_t)r * dim; },
            [&](int r, const float *y) { hb[r] = y[0] / (1.0f + expf(-y[0])) * y[1]; });
        __syncthreads();

        // 2h: x += W2 hb
        cta_gemv<1>(
            hidden, dim, hb, [&](int, int r) { return w2 + (size_t)r * hidden; },
            [&](int r, const float *y) { x[r] += y[0]; });
        __syncthreads();
    }

    // step 3: final RMSNorm and the classifier
    cta_rmsnorm(x, gains + (size_t)p.n_layers * 2 * dim, xn, dim, red);
    float *user = p.step->logits_out;
    cta_gemv<1>(
        dim, p.vocab, xn, [&](int, int r) { return p.wcls + (size_t)r * dim; },
        [&](int r, const float *y) {
            p.logits[r] = y[0];
            if (user) user[r] = y[0];
        });
    for (int i = tid; i < dim; i += kCT) p.x[i] = x[i];
}

size_t step_cta_smem(int dim, int hidden, int kv_dim, int n_heads, int seq_len, int n_layers) {
    return (size_t)CtaLayout(dim, hidden, kv_dim, n_heads, seq_len, n_layers).total * sizeof(float);
}

cudaError_t step_cta_init() {
    return cudaFuncSetAttribute(l2dec_step_cta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t launch_step_cta(const CtaStepParams &p, size_t smem, cudaStream_t stream) {
    l2dec_step_cta_kernel<<<1, kCT, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace l2
