// Fused streaming matrix-vector kernels of the decode step (batch 1).
//
// Every weight matmul of llama2.c's forward step ("run.c", matmul(): W (d,n)
// @ x (n,) -> (d,), rows split across threads) is one launch of l2dec_matvec_kernel,
// with the neighbouring elementwise work fused in:
//   GEMV_QKV   rmsnorm(x) -> Wq|Wk|Wv -> RoPE -> q, and K/V rows written into
//              the cache (walkthrough §4 forward() steps 2a-2d)
//   GEMV_RESID x += W v for Wo (step 2f) and W2 (step 2h)
//   GEMV_W13   rmsnorm(x) -> W1, W3 -> hb = silu(h1) * h3 (steps 2g-2h)
//   GEMV_CLS   rmsnorm(x) -> logits = Wcls x (step 3)
//
// Design.  The kernel is HBM-bound (0.5 flop per weight byte), so it is built
// around moving the weights at full bandwidth:
//   - the grid is one CTA per SM; CTA c owns a contiguous, balanced range of
//     output rows, i.e. one contiguous range of weight memory per matrix;
//   - that range is split evenly, at 16-byte granularity and regardless of row
//     boundaries, across the CTA's warps;
//   - each warp streams its range through a private ring of shared-memory
//     buffers filled by 1-D bulk async copies (TMA) completing on mbarriers,
//     so several KB per warp are always in flight;
//   - lanes read 16-byte words of the weights and of the input vector (held in
//     shared memory) and accumulate with FMAs; a row finished by one warp is
//     reduced with shuffles, and a row shared by neighbouring warps is summed
//     from their partials in warp order, so results are deterministic;
//   - the weight copies for the first stages are issued before
//     griddepcontrol.wait, so under programmatic dependent launch they overlap
//     the tail of the previous kernel.
// Weights are fp32 (WT = 0, 4 per 16-byte word) or bf16 (WT = 1, a handle
// created with L2_FLAG_BF16_WEIGHTS: 8 per word, each widened exactly to
// fp32 -- a bf16 value is the top half of an fp32 -- and multiplied into the
// fp32 input vector with fp32 accumulation); everything else is fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

// Launch shapes (compile-time): warps per CTA, ring buffers per warp, 16-byte
// words per buffer.  A plan takes the first shape whose shared memory (ring +
// input vector) fits: A, else B (for long rows such as W2's), else C.
// Measured on GB300 (7B shape): 8 KB copies reach ~6 TB/s where 2 KB copies
// with the same bytes in flight stay near 3.7 TB/s, so the per-copy cost sets
// the rate; and a pure read stream of 8 KB copies reaches ~7.3 TB/s, so the
// compute between a buffer's arrival and its refill matters.  With three or
// more stages (L2_GEMV_ISSUE_AHEAD) a warp therefore refills the buffer it
// finished in the previous iteration as soon as its wait returns, keeping
// stages - 1 copies in flight while it computes.  L2_GEMV_FENCE adds a
// generic->async proxy fence before a buffer is refilled (not needed: the
// warp's reads of the buffer have completed when it issues the refill).
#ifndef L2_GEMV_WARPS
#define L2_GEMV_WARPS 8
#endif
#ifndef L2_GEMV_STAGES
#define L2_GEMV_STAGES 3
#endif
#ifndef L2_GEMV_CHUNK_WORDS
#define L2_GEMV_CHUNK_WORDS 512
#endif
#ifndef L2_GEMV_WARPS_B
#define L2_GEMV_WARPS_B 7
#endif
#ifndef L2_GEMV_STAGES_B
#define L2_GEMV_STAGES_B 3
#endif
#ifndef L2_GEMV_CHUNK_WORDS_B
#define L2_GEMV_CHUNK_WORDS_B 512
#endif
#ifndef L2_GEMV_ISSUE_AHEAD
#define L2_GEMV_ISSUE_AHEAD 1
#endif
#ifndef L2_GEMV_FENCE
#define L2_GEMV_FENCE 0
#endif
// With issue-ahead, request every ring buffer before griddepcontrol.wait (all
// STAGES chunks, not STAGES - 1): the buffer the steady state keeps free for
// the next refill is free at the start too, so one more chunk of this
// kernel's weights streams while the previous kernel drains.
#ifndef L2_GEMV_PREISSUE_ALL
#define L2_GEMV_PREISSUE_ALL 0
#endif

namespace l2 {

namespace {

struct Piece {
    const float4 *src;  // first weight word of the piece
    long long f0;       // offset of the piece in the CTA's word stream
    int rows;           // whole rows of n floats
    int yoff;           // local output index of the piece's first row
    long long off;      // its first word's offset in the layer's matrix (bounds checks)
    long long words;    // that matrix's words (bounds checks)
};

template <int NW, int STAGES>
struct GemvFixed {
    uint64_t bars[NW * STAGES];
    float head_val[NW];
    float tail_val[NW];
    int head_row[NW];
    int tail_row[NW];
    float red[NW];
    float scalar;
    int npieces;
    int failed;
    Piece pieces[3];
};

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

template <int NW, int STAGES>
__host__ __device__ constexpr size_t fixed_bytes() {
    return align_up(sizeof(GemvFixed<NW, STAGES>), 128);
}

__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

// 8 bf16 weights (in memory order: low half of w.x first) times 8 fp32
// inputs: four independent pairs, added as a tree, so the chain a word adds to
// the running sum is one addition (the word carries twice the fp32 products).
__device__ __forceinline__ float dot_bf16x8(uint4 w, float4 x0, float4 x1, float acc) {
    const float p0 = fmaf(__uint_as_float(w.x & 0xffff0000u), x0.y, __uint_as_float(w.x << 16) * x0.x);
    const float p1 = fmaf(__uint_as_float(w.y & 0xffff0000u), x0.w, __uint_as_float(w.y << 16) * x0.z);
    const float p2 = fmaf(__uint_as_float(w.z & 0xffff0000u), x1.y, __uint_as_float(w.z << 16) * x1.x);
    const float p3 = fmaf(__uint_as_float(w.w & 0xffff0000u), x1.w, __uint_as_float(w.w << 16) * x1.z);
    return acc + ((p0 + p1) + (p2 + p3));
}

}  // namespace

template <int NW, int STAGES, int CH4, int MODE, int WT>
__global__ void __launch_bounds__(NW * 32, 1) l2dec_matvec_kernel(const GemvParams p) {
    constexpr int NT = NW * 32;
    extern __shared__ __align__(128) unsigned char smem[];
    auto &fx = *reinterpret_cast<GemvFixed<NW, STAGES> *>(smem);
    float4 *ring = reinterpret_cast<float4 *>(smem + fixed_bytes<NW, STAGES>());
    const int n4 = p.n >> 2;             // input vector: 16-byte words
    const int nw = WT ? p.n >> 3 : n4;   // weight row: 16-byte words
    // the first weight word of row `row` of a matrix
    auto row_ptr = [&](const float *mat, size_t row) {
        return WT ? reinterpret_cast<const float4 *>(reinterpret_cast<const unsigned short *>(mat) + row * p.n)
                  : reinterpret_cast<const float4 *>(mat + row * p.n);
    };
    float4 *xs = ring + NW * STAGES * CH4;
    float *ys = reinterpret_cast<float *>(xs + n4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- this CTA's rows: a balanced share of the units ----
    const long long u0 = (long long)blockIdx.x * p.total_units / gridDim.x;
    const long long u1 = (long long)(blockIdx.x + 1) * p.total_units / gridDim.x;
    const int vr0 = (int)(u0 * p.unit_rows);
    const int R = (int)((u1 - u0) * p.unit_rows);

    if (tid == 0) {
        int np = 0;
        long long f = 0;
        if (R > 0) {
            if (MODE == GEMV_QKV) {
                const float *mats[3] = {p.mat0, p.mat1, p.mat2};
                const int rws[3] = {p.rows0, p.rows1, p.rows2};
                int b0 = 0;
                for (int m = 0; m < 3; ++m) {
                    int lo = max(vr0, b0), hi = min(vr0 + R, b0 + rws[m]);
                    if (lo < hi) {
                        fx.pieces[np] = {row_ptr(mats[m], (size_t)(lo - b0)), f, hi - lo, lo - vr0,
                                         (long long)(lo - b0) * nw, (long long)rws[m] * nw};
                        f += (long long)(hi - lo) * nw;
                        ++np;
                    }
                    b0 += rws[m];
                }
            } else if (MODE == GEMV_W13) {
                const long long mw = (long long)p.total_units * p.unit_rows * nw;
                fx.pieces[0] = {row_ptr(p.mat0, (size_t)vr0), 0, R, 0, (long long)vr0 * nw, mw};
                fx.pieces[1] = {row_ptr(p.mat1, (size_t)vr0), (long long)R * nw, R, R, (long long)vr0 * nw, mw};
                np = 2;
            } else {
                fx.pieces[0] = {row_ptr(p.mat0, (size_t)vr0), 0, R, 0, (long long)vr0 * nw,
                                (long long)p.total_units * p.unit_rows * nw};
                np = 1;
            }
        }
        fx.npieces = np;
        fx.failed = 0;
        for (int i = 0; i < NW * STAGES; ++i) mbar_init(&fx.bars[i], 1);
        fence_barrier_init();
    }
    if (lane == 0) {
        fx.head_row[warp] = -1;
        fx.tail_row[warp] = -1;
    }
    __syncthreads();

    const int np = fx.npieces;
    long long F = 0;
    for (int i = 0; i < np; ++i) F += (long long)fx.pieces[i].rows * nw;
    // Warp ranges start on 128-byte boundaries of the stream (whole cache lines
    // whenever the pieces themselves start on one).
    const long long fb = (F * warp / NW) & ~7LL;
    const long long fe = warp == NW - 1 ? F : (F * (warp + 1) / NW) & ~7LL;

    // The chunk that starts at word f of the stream: its piece and length.
    auto chunk_at = [&](long long f, int &pi, int &len) {
        pi = 0;
        while (pi + 1 < np && f >= fx.pieces[pi + 1].f0) ++pi;
        const long long pend = fx.pieces[pi].f0 + (long long)fx.pieces[pi].rows * nw;
        long long l = fe - f;
        if (pend - f < l) l = pend - f;
        if (l > CH4) l = CH4;
        len = (int)l;
    };

    const uint64_t pol = policy_evict_first();
    const bool hint = p.evict_first != 0;
    uint64_t *bars = &fx.bars[warp * STAGES];
    float4 *wring = ring + (size_t)warp * STAGES * CH4;
    long long fi = fb;  // next word to request
    int n_issued = 0;   // chunks requested so far
    auto issue = [&](int stage) {
        int pi, len;
        chunk_at(fi, pi, len);
        if (lane == 0) {
            const Piece &pc = fx.pieces[pi];
            // a copy outside its matrix (bounds-checked build) is skipped; the barrier expects nothing
            const bool ok = in_bounds((size_t)(pc.off + (fi - pc.f0)), (size_t)len, (size_t)pc.words, p.err) &&
                            len <= CH4;
            mbar_arrive_expect_tx(&bars[stage], ok ? (uint32_t)len * 16u : 0u);
            if (ok && hint)
                bulk_g2s(wring + (size_t)stage * CH4, pc.src + (fi - pc.f0), (uint32_t)len * 16u, &bars[stage], pol);
            else if (ok)
                bulk_g2s_nohint(wring + (size_t)stage * CH4, pc.src + (fi - pc.f0), (uint32_t)len * 16u, &bars[stage]);
        }
        fi += len;
        ++n_issued;
    };

    // Weights do not depend on the previous kernel: start streaming them now.
    constexpr bool AHEAD = L2_GEMV_ISSUE_AHEAD && STAGES >= 3;
    constexpr int PRE = AHEAD && !L2_GEMV_PREISSUE_ALL ? STAGES - 1 : STAGES;
#pragma unroll 1
    for (int s = 0; s < PRE && fi < fe; ++s) issue(s);

    pdl_launch_dependents();
    pdl_wait();

    // ---- input vector into shared memory (with RMSNorm where the mode has one) ----
    if (MODE == GEMV_RESID) {
        const float4 *in4 = reinterpret_cast<const float4 *>(p.in_vec);
        for (int i = tid; i < n4; i += NT) xs[i] = in4[i];
    } else {
        const float *src = p.x;
        if (MODE == GEMV_QKV && p.layer == 0) {
            const size_t row = (size_t)p.step->token[0] * p.dim;
            src = in_bounds(row, (size_t)p.dim, p.ext->emb, p.err) ? p.emb + row : p.emb;
        }
        const float4 *s4 = reinterpret_cast<const float4 *>(src);
        float ss = 0.f;
        for (int i = tid; i < n4; i += NT) {
            float4 v = s4[i];
            xs[i] = v;
            ss = fmaf(v.x, v.x, ss);
            ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss);
            ss = fmaf(v.w, v.w, ss);
        }
        if (MODE == GEMV_QKV && p.layer == 0 && blockIdx.x == 0) {
            float4 *x4 = reinterpret_cast<float4 *>(p.x);
            for (int i = tid; i < n4; i += NT) x4[i] = s4[i];
        }
        ss = warp_sum(ss);
        if (lane == 0) fx.red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
            float t = 0.f;
            for (int w = 0; w < NW; ++w) t += fx.red[w];
            fx.scalar = 1.0f / sqrtf(t / (float)p.n + 1e-5f);
        }
        __syncthreads();
        const float inv = fx.scalar;
        const float4 *g4 = reinterpret_cast<const float4 *>(p.norm_w);
        for (int i = tid; i < n4; i += NT) {
            float4 v = xs[i], g = g4[i];
            xs[i] = make_float4(g.x * (inv * v.x), g.y * (inv * v.y), g.z * (inv * v.z), g.w * (inv * v.w));
        }
    }
    __syncthreads();
    if (WT) {
        // A bf16 weight word (8 weights) meets two input words, 2w and 2w + 1.  Read in
        // place, lane l's pair sits 32 bytes from lane l+1's, so every load of the input
        // took two shared-memory wavefronts per 8 lanes (a 2-way bank conflict).  Each
        // block of 32 weight words (M < 32 in a row's last block) therefore keeps its 2M
        // input words as [even words | odd words]: the lanes read consecutive words.
        for (int kb = warp; 32 * kb < nw; kb += NW) {
            const int M = min(32, nw - 32 * kb);
            float4 e = make_float4(0.f, 0.f, 0.f, 0.f), o = e;
            if (lane < M) {
                e = xs[64 * kb + 2 * lane];
                o = xs[64 * kb + 2 * lane + 1];
            }
            __syncwarp();
            if (lane < M) {
                xs[64 * kb + lane] = e;
                xs[64 * kb + M + lane] = o;
            }
        }
        __syncthreads();
    }

    // ---- stream this warp's weight words ----
    float acc = 0.f;
    bool started = false;  // this warp began the current row at its first word
    bool pending = false;  // acc holds words of a row not yet deposited
    int cur_row = -1;
    long long fc = fb;
    // Row walk state within the current piece: row r spans local words [rs, re).
    int cpi = -1, r = 0, rs = 0, re = 0;
    bool ok = true;
    int k = 0;
#pragma unroll 1
    for (; fc < fe; ++k) {
        const int s = k % STAGES;
        int pi, len;
        chunk_at(fc, pi, len);
        if (!mbar_wait(&bars[s], (uint32_t)(k / STAGES) & 1u, p.err)) {
            ok = false;
            break;
        }
        // chunk k + STAGES - 1 goes into the buffer finished in iteration k - 1
        // (at k = 0 it may already be in flight: every buffer was requested up front)
        if (AHEAD && fi < fe && n_issued == k + STAGES - 1) issue((k + STAGES - 1) % STAGES);
        const Piece &pc = fx.pieces[pi];
        const float4 *buf = wring + (size_t)s * CH4;
        const int lf = (int)(fc - pc.f0), lend = lf + len;
        if (pi != cpi) {
            cpi = pi;
            r = lf / nw;
            rs = r * nw;
            re = rs + nw;
        }
        int a = lf;
        while (a < lend) {
            if (a == re) {
                ++r;
                rs = re;
                re += nw;
            }
            const int b = lend < re ? lend : re;
            if (a == rs) started = true;
            cur_row = pc.yoff + r;
            const float4 *wr = buf + (a - lf);
            const int cnt = b - a;
            if (WT) {
                // the input words of row word w: block w / 32 at 64 (w / 32), its M words
                // apart; lane l's word advances by one block per iteration
                const int w0 = (a - rs) + lane;
                int wb = w0 & ~31;
                const float4 *xr = xs + 2 * wb + (w0 & 31);
#pragma unroll 4
                for (int i = lane; i < cnt; i += 32) {
                    const int M = min(32, nw - wb);
                    acc = dot_bf16x8(reinterpret_cast<const uint4 *>(wr)[i], xr[0], xr[M], acc);
                    xr += 64;
                    wb += 32;
                }
            } else {
                const float4 *xr = xs + (a - rs);
#pragma unroll 4
                for (int i = lane; i < cnt; i += 32) acc = dot4(wr[i], xr[i], acc);
            }
            pending = true;
            if (b == re) {
                const float v = warp_sum(acc);
                if (lane == 0) {
                    if (started) {
                        ys[cur_row] = v;
                    } else {
                        fx.head_row[warp] = cur_row;
                        fx.head_val[warp] = v;
                    }
                }
                acc = 0.f;
                pending = false;
                started = true;
            }
            a = b;
        }
        __syncwarp();
        fc += len;
        if (!AHEAD && fi < fe) {
#if L2_GEMV_FENCE
            if (lane == 0) fence_proxy_async_smem();
#endif
            issue(s);
        }
    }
    if (!ok) {
        // Let the copies still in flight land before the CTA's memory is released;
        // the CTA then skips its epilogue (the host sees the device error word).
        for (int j = k + 1; j < n_issued; ++j) (void)mbar_wait(&bars[j % STAGES], (uint32_t)(j / STAGES) & 1u, p.err);
        if (lane == 0) fx.failed = 1;
        pending = false;
    }
    if (pending) {
        const float v = warp_sum(acc);
        if (lane == 0) {
            if (started) {
                fx.tail_row[warp] = cur_row;
                fx.tail_val[warp] = v;
            } else {
                fx.head_row[warp] = cur_row;
                fx.head_val[warp] = v;
            }
        }
    }
    __syncthreads();
    if (fx.failed) return;
    if (tid == 0) {
        for (int w = 0; w < NW; ++w) {
            if (fx.head_row[w] >= 0) ys[fx.head_row[w]] += fx.head_val[w];
            if (fx.tail_row[w] >= 0) ys[fx.tail_row[w]] = fx.tail_val[w];
        }
    }
    __syncthreads();

    // ---- epilogue ----
    if (MODE == GEMV_QKV) {
        const int pos = p.step->pos[0];
        const int hs = p.head_size, half = hs >> 1;
        const float2 *rr = p.rope + (size_t)pos * half;
        for (int i = tid; i < (R >> 1); i += NT) {
            const int j = 2 * i, v = vr0 + j;
            const float y0 = ys[j], y1 = ys[j + 1];
            if (v < p.dim) {
                if (!in_bounds((size_t)pos * half + ((v % hs) >> 1), 1, p.ext->rope, p.err) ||
                    !in_bounds((size_t)v, 2, p.ext->q, p.err))
                    continue;
                const float2 cs = rr[(v % hs) >> 1];
                p.q[v] = y0 * cs.x - y1 * cs.y;
                p.q[v + 1] = y0 * cs.y + y1 * cs.x;
            } else {
                const bool is_k = v < p.dim + p.kv_dim;
                const int c = is_k ? v - p.dim : v - p.dim - p.kv_dim;
                const int g = c / hs, d = c % hs;
                const size_t idx =
                    ((((size_t)p.step->slot[0] * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + pos) * hs + d;
                if (!in_bounds(idx, 2, p.ext->cache, p.err) ||
                    !in_bounds((size_t)pos * half + (d >> 1), 1, p.ext->rope, p.err))
                    continue;
                if (is_k) {
                    const float2 cs = rr[d >> 1];
                    p.kcache[idx] = y0 * cs.x - y1 * cs.y;
                    p.kcache[idx + 1] = y0 * cs.y + y1 * cs.x;
                } else {
                    p.vcache[idx] = y0;
                    p.vcache[idx + 1] = y1;
                }
            }
        }
    } else if (MODE == GEMV_RESID) {
        for (int j = tid; j < R; j += NT)
            if (in_bounds((size_t)vr0 + j, 1, p.ext->x, p.err)) p.x[vr0 + j] += ys[j];
    } else if (MODE == GEMV_W13) {
        for (int j = tid; j < R; j += NT)
            if (in_bounds((size_t)vr0 + j, 1, p.ext->hb, p.err)) p.hb[vr0 + j] = silu(ys[j]) * ys[R + j];
    } else {
        float *user = p.step->logits_out;
        for (int j = tid; j < R; j += NT) {
            if (!in_bounds((size_t)vr0 + j, 1, p.ext->logits, p.err)) continue;
            p.logits[vr0 + j] = ys[j];
            if (user) user[vr0 + j] = ys[j];
        }
    }
}

// ---------------------------------------------------------------- host side

__global__ void f32_to_bf16_kernel(const float *src, unsigned short *dst, size_t n) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(src[i]);
        dst[i] = *reinterpret_cast<const unsigned short *>(&b);
    }
}

cudaError_t convert_to_bf16(const float *src, unsigned short *dst, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    f32_to_bf16_kernel<<<1024, 256, 0, stream>>>(src, dst, n);
    return cudaGetLastError();
}


namespace {
struct Shape {
    int nw, stages, ch4;
};
constexpr Shape kShapes[kGemvShapes] = {{L2_GEMV_WARPS, L2_GEMV_STAGES, L2_GEMV_CHUNK_WORDS},
                                        {L2_GEMV_WARPS_B, L2_GEMV_STAGES_B, L2_GEMV_CHUNK_WORDS_B},
                                        {8, 2, 512}};

template <int S, int MODE, int WT>
void *kernel_ptr() {
    return reinterpret_cast<void *>(l2dec_matvec_kernel<kShapes[S].nw, kShapes[S].stages, kShapes[S].ch4, MODE, WT>);
}

template <int S, int WT>
void *kernel_for(int mode) {
    switch (mode) {
        case GEMV_QKV: return kernel_ptr<S, GEMV_QKV, WT>();
        case GEMV_RESID: return kernel_ptr<S, GEMV_RESID, WT>();
        case GEMV_W13: return kernel_ptr<S, GEMV_W13, WT>();
        case GEMV_CLS: return kernel_ptr<S, GEMV_CLS, WT>();
    }
    return nullptr;
}

template <int WT>
void *kernel_for(int shape, int mode) {
    switch (shape) {
        case 0: return kernel_for<0, WT>(mode);
        case 1: return kernel_for<1, WT>(mode);
        case 2: return kernel_for<2, WT>(mode);
    }
    return nullptr;
}

void *kernel_for(int shape, int mode, int wt) { return wt ? kernel_for<1>(shape, mode) : kernel_for<0>(shape, mode); }

template <int S>
size_t fixed_of() {
    return fixed_bytes<kShapes[S].nw, kShapes[S].stages>();
}

size_t fixed_of(int shape) {
    switch (shape) {
        case 0: return fixed_of<0>();
        case 1: return fixed_of<1>();
        default: return fixed_of<2>();
    }
}
}  // namespace

int gemv_threads(int shape) { return kShapes[shape].nw * 32; }

size_t gemv_smem_bytes(int shape, int n, int ymax) {
    const Shape &sh = kShapes[shape];
    return fixed_of(shape) + (size_t)sh.nw * sh.stages * sh.ch4 * 16 + (size_t)n * 4 + align_up((size_t)ymax * 4, 16);
}

int gemv_pick_shape(int n, int ymax, size_t *smem) {
    for (int sh = 0; sh < kGemvShapes; ++sh) {
        *smem = gemv_smem_bytes(sh, n, ymax);
        if (*smem <= 227 * 1024) return sh;
    }
    return -1;
}

cudaError_t gemv_init() {
    for (int wt = 0; wt < 2; ++wt)
        for (int sh = 0; sh < kGemvShapes; ++sh)
            for (int mode = GEMV_QKV; mode <= GEMV_CLS; ++mode) {
                cudaError_t e = cudaFuncSetAttribute(kernel_for(sh, mode, wt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     227 * 1024);
                if (e != cudaSuccess) return e;
            }
    return cudaSuccess;
}

cudaError_t launch_gemv(int mode, int shape, const GemvParams &p, int grid, size_t smem, cudaStream_t stream,
                        bool pdl, int wt) {
    if (shape < 0 || shape >= kGemvShapes) return cudaErrorInvalidValue;
    void *fn = kernel_for(shape, mode, wt);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(gemv_threads(shape));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<GemvParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace l2
