// The whole decode step for one sequence in one persistent launch.
//
// What it computes is llama2.c's forward() for one token ("run.c",
// transformer(); "run.c 逐行解讀" §4 forward(), steps 1-3): per layer,
// rmsnorm -> Wq|Wk|Wv -> RoPE -> K/V rows into the cache -> causal GQA
// attention -> Wo + residual -> rmsnorm -> W1, W3 -> SwiGLU -> W2 + residual;
// then the final rmsnorm and the classifier.  The arithmetic per output is
// the same as the per-matmul kernels' (gemv.cu, attention.cu); what differs
// is how the step is scheduled on the GPU.
//
// Why one launch.  At batch 1 the step streams every weight once and is
// bound by HBM bandwidth.  A separate launch per matmul pays, at each of the
// 5 L + 1 boundaries, for the previous kernel's drain and the next one's ramp
// (measured on GB300: a pure read kernel of n bytes takes ~6.5 us + n / 7.4
// TB/s back to back), and programmatic dependent launch hides only part of
// it because a CTA of the next kernel cannot become resident while the
// previous one holds the SM's shared memory.
//
// How.  A cooperative launch of one CTA per SM runs the step's phases
//   QKV(l), ATT(l), WO(l), W13(l), W2(l) for every layer l, then CLS,
// with a grid-wide barrier after each phase but the last (the next phase
// reads what every CTA wrote).  Every warp owns a ring of shared-memory
// buffers fed by 1-D bulk async copies (TMA) and consumes ONE continuous
// stream of copies across the whole step: its share of the QKV weights,
// then its share of the cache rows its attention item needs, then its share
// of Wo, and so on.  A buffer is refilled as soon as it is consumed, with
// the next copy of the stream whatever phase it belongs to; weights never
// depend on the step's activations and cache rows before pos were written by
// earlier steps, so while a CTA waits at a barrier its ring is already
// filling with the next phase's data and HBM keeps streaming.  The cache row
// at pos, written during this step, is read with plain loads after the
// barrier.  Activations written by other CTAs (x, xb, q, hb, the new cache
// row, attention partials) are read with ld.global.cg (L2), never from L1.
//
// Work split per phase: GEMV phases give CTA c a balanced contiguous range of
// output rows (pairs for QKV, so RoPE stays local) and split its weight words
// evenly across the warps, as in gemv.cu; the attention phase gives CTA c at
// most one item (KV head g, a chunk of its positions), split across the
// warps, with partials merged by the last CTA of the head (attention.cu).
//
// Measured on GB300 it is slower than the default graph of per-matmul
// kernels with programmatic dependent launch (7B shape: 213 against 233
// steps/s at positions 3..400; tiny shape: 6.2 k against 9.8 k): each phase
// boundary here is a chain of L2 round trips (barrier arrival and polling,
// the input vector, the epilogue's loads and stores) of about 4-6 us, more
// than the ~4 us a hardware-resolved kernel boundary costs, and the streaming
// between boundaries is no faster.  It is kept as an option (L2_FLAG_PERSIST).
//
// Every wait is bounded: a copy or a barrier that does not complete within
// about two seconds sets L2_DEV_ERR_TIMEOUT; the CTA then waits (bounded)
// for its own copies in flight and returns, and the other CTAs time out at
// their next barrier and do the same.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

// Launch shape: warps per CTA (compile-time); the ring (buffers per warp and
// their size) is chosen by the host to fill the shared memory the largest
// phase leaves free: the deeper the ring, the more of the next phase is in
// flight while a barrier resolves.
#ifndef L2_STEP_WARPS
#define L2_STEP_WARPS 8
#endif

namespace l2 {

namespace {

constexpr int kNW = L2_STEP_WARPS;
constexpr int kMaxStages = 4;
constexpr int kNT = kNW * 32;
constexpr int kPPG = 4;  // cache positions a lane group scores before one softmax update

enum Phase : int { PH_QKV = 0, PH_ATT = 1, PH_WO = 2, PH_W13 = 3, PH_W2 = 4, PH_CLS = 5 };

struct Piece {
    const float4 *src;  // first weight word of the piece
    long long f0;       // offset of the piece in the CTA's word stream
    int rows;           // whole rows of n floats
    int yoff;           // local output index of the piece's first row
};

// One warp's share of one phase of the step's copy stream.
struct Seg {
    int kind, layer;
    // GEMV phases: the CTA's output rows [vr0, vr0 + R) are up to three pieces
    // of weight memory laid end to end; this warp streams words [b, e).
    int np, n4, vr0, R;
    Piece pc[3];
    // attention: this CTA's item (KV head g, chunk c of n_active) and this
    // warp's positions [wt0, wt1); ring rows are [b, e) = [wt0, min(wt1, pos)).
    int g, c, n_active, wt0, wt1;
    const float *kb, *vb;
    long long b, e;
};

struct Fixed {
    uint64_t bars[kNW * kMaxStages];
    float head_val[kNW];
    float tail_val[kNW];
    int head_row[kNW];
    int tail_row[kNW];
    float red[kNW];
    float scalar;
    int abort;  // a wait of this CTA gave up
    int last;   // this CTA merges the attention chunks of its head
};

__host__ __device__ constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
constexpr size_t kFixedBytes = align_up(sizeof(Fixed), 128);

__device__ __forceinline__ float silu(float v) { return v / (1.0f + expf(-v)); }

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The phase at index ph of the step (5 per layer, then the classifier).
__device__ __forceinline__ void phase_of(const StepKParams &p, int ph, int &kind, int &layer) {
    if (ph >= 5 * p.n_layers) {
        kind = PH_CLS;
        layer = 0;
    } else {
        kind = ph % 5;
        layer = ph / 5;
    }
}

// Attention chunks in use at this position: enough that each takes at least
// min_chunk positions, at most n_chunks.
__device__ __forceinline__ int active_chunks(const StepKParams &p, int P) {
    int n = (P + p.min_chunk - 1) / p.min_chunk;
    return n < p.n_chunks ? n : p.n_chunks;
}

// This warp's share of phase ph.
__device__ void make_seg(const StepKParams &p, int ph, int pos, int warp, Seg &s) {
    phase_of(p, ph, s.kind, s.layer);
    s.np = 0;
    s.b = s.e = 0;
    s.R = 0;
    s.vr0 = 0;
    s.g = -1;
    const size_t l = (size_t)s.layer;
    const int G = gridDim.x, cta = blockIdx.x;
    if (s.kind == PH_ATT) {
        const int P = pos + 1;
        const int na = active_chunks(p, P);
        s.n_active = na;
        if (cta >= na * p.n_kv_heads) return;
        s.g = cta / na;
        s.c = cta % na;
        const int t0 = (int)((long long)s.c * P / na), t1 = (int)((long long)(s.c + 1) * P / na);
        s.wt0 = t0 + (int)((long long)(t1 - t0) * warp / kNW);
        s.wt1 = t0 + (int)((long long)(t1 - t0) * (warp + 1) / kNW);
        const size_t head_base = ((l * p.n_kv_heads + s.g) * (size_t)p.seq_len) * p.head_size;
        s.kb = p.kcache + head_base;
        s.vb = p.vcache + head_base;
        s.b = s.wt0;
        s.e = s.wt1 < pos ? s.wt1 : pos;
        if (s.e < s.b) s.e = s.b;
        return;
    }
    // GEMV geometry of the phase
    int n, unit_rows, units;
    const float *m0, *m1 = nullptr, *m2 = nullptr;
    switch (s.kind) {
        case PH_QKV:
            n = p.dim;
            unit_rows = 2;
            units = (p.dim + 2 * p.kv_dim) / 2;
            m0 = p.wq + l * p.dim * p.dim;
            m1 = p.wk + l * p.kv_dim * p.dim;
            m2 = p.wv + l * p.kv_dim * p.dim;
            break;
        case PH_WO:
            n = p.dim;
            unit_rows = 1;
            units = p.dim;
            m0 = p.wo + l * p.dim * p.dim;
            break;
        case PH_W13:
            n = p.dim;
            unit_rows = 1;
            units = p.hidden_dim;
            m0 = p.w1 + l * p.hidden_dim * p.dim;
            m1 = p.w3 + l * p.hidden_dim * p.dim;
            break;
        case PH_W2:
            n = p.hidden_dim;
            unit_rows = 1;
            units = p.dim;
            m0 = p.w2 + l * p.dim * p.hidden_dim;
            break;
        default:
            n = p.dim;
            unit_rows = 1;
            units = p.vocab;
            m0 = p.wcls;
            break;
    }
    const int n4 = n >> 2;
    s.n4 = n4;
    const long long u0 = (long long)cta * units / G, u1 = (long long)(cta + 1) * units / G;
    s.vr0 = (int)(u0 * unit_rows);
    s.R = (int)((u1 - u0) * unit_rows);
    if (s.R <= 0) return;
    long long F = 0;
    if (s.kind == PH_QKV) {
        // three pieces (Wq, Wk, Wv rows), any of them possibly empty
        auto cut = [&](const float *mat, int b0, int rows) {
            const int lo = max(s.vr0, b0), hi = max(lo, min(s.vr0 + s.R, b0 + rows));
            Piece pc = {reinterpret_cast<const float4 *>(mat + (size_t)(lo - b0) * n), F, hi - lo, lo - s.vr0};
            F += (long long)(hi - lo) * n4;
            return pc;
        };
        s.pc[0] = cut(m0, 0, p.dim);
        s.pc[1] = cut(m1, p.dim, p.kv_dim);
        s.pc[2] = cut(m2, p.dim + p.kv_dim, p.kv_dim);
        s.np = 3;
    } else {
        s.pc[0] = {reinterpret_cast<const float4 *>(m0 + (size_t)s.vr0 * n), 0, s.R, 0};
        s.np = 1;
        F = (long long)s.R * n4;
        if (s.kind == PH_W13) {
            s.pc[1] = {reinterpret_cast<const float4 *>(m1 + (size_t)s.vr0 * n), F, s.R, s.R};
            s.np = 2;
            F *= 2;
        }
    }
    // warp shares start on 128-byte boundaries of the stream
    s.b = (F * warp / kNW) & ~7LL;
    s.e = warp == kNW - 1 ? F : (F * (warp + 1) / kNW) & ~7LL;
}

// Piece i of a segment (by value, so the pieces stay in registers).
__device__ __forceinline__ Piece piece(const Seg &s, int i) {
    Piece r = s.pc[0];
    if (i == 1) r = s.pc[1];
    if (i == 2) r = s.pc[2];
    return r;
}

// The GEMV copy that starts at word f of a segment: its piece and length (at
// most ch4 words).  (Piece offsets never decrease; an empty piece shares its
// successor's.)
__device__ __forceinline__ void locate(const Seg &s, long long f, int ch4, int &pi, int &len) {
    pi = 0;
    if (s.np > 1 && f >= s.pc[1].f0) pi = 1;
    if (s.np > 2 && f >= s.pc[2].f0) pi = 2;
    const Piece pc = piece(s, pi);
    const long long pend = pc.f0 + (long long)pc.rows * s.n4;
    long long l = s.e - f;
    if (pend - f < l) l = pend - f;
    if (l > ch4) l = ch4;
    len = (int)l;
}

}  // namespace

template <int GQ>
__global__ void __launch_bounds__(kNT, 1) step_kernel(const StepKParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    Fixed &fx = *reinterpret_cast<Fixed *>(smem);
    const int S = p.stages, CH4 = p.ch4;
    float4 *ring = reinterpret_cast<float4 *>(smem + kFixedBytes);
    unsigned char *uni = smem + kFixedBytes + (size_t)kNW * S * CH4 * 16;  // phase-dependent region
    float4 *xs = reinterpret_cast<float4 *>(uni);          // GEMV input vector
    float *ys = reinterpret_cast<float *>(uni) + p.xs_floats;
    const int hs = p.head_size, hs4 = hs >> 2;
    float4 *accs = reinterpret_cast<float4 *>(uni);  // attention: [kNW][GQ][hs4]
    float *mrg = reinterpret_cast<float *>(accs + kNW * GQ * hs4);  // [kNW][GQ][2]
    float *fin = mrg + kNW * GQ * 2;                                 // [GQ][2]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x;
    const int pos = p.step->pos[0];
    const int NPH = 5 * p.n_layers + 1;
    const int TP = CH4 * 4 / (2 * hs);  // cache positions per ring buffer

    if (tid == 0) {
        for (int i = 0; i < kNW * S; ++i) mbar_init(&fx.bars[i], 1);
        fence_barrier_init();
        fx.abort = 0;
    }
    if (lane == 0) {
        fx.head_row[warp] = -1;
        fx.tail_row[warp] = -1;
    }
    __syncthreads();

    uint64_t *bars = &fx.bars[warp * S];
    float4 *wring = ring + (size_t)warp * S * CH4;
    const uint64_t pol = policy_evict_first();
    const bool hint = p.evict_first != 0;

    // ---- the issue side of this warp's stream ----
    // Copy j of the stream uses buffer j mod S and completes phase floor(j / S)
    // mod 2 of that buffer's mbarrier; the counters below track both.
    long long n_iss = 0, n_con = 0;   // copies issued / consumed
    int st_iss = 0, st_con = 0;       // their buffers
    uint32_t con_par = 0;             // bit s: parity of buffer s's next completion
    int iph = 0;                     // phase of the next copy to issue (NPH: none left)
    Seg is;
    make_seg(p, 0, pos, warp, is);
    long long icur = is.b;
    auto advance = [&]() {
        while (iph < NPH && icur >= is.e) {
            if (++iph < NPH) {
                make_seg(p, iph, pos, warp, is);
                icur = is.b;
            }
        }
    };
    advance();
    auto pump = [&]() {
        while (n_iss - n_con < S && iph < NPH) {
            const int st = st_iss;
            st_iss = st_iss + 1 == S ? 0 : st_iss + 1;
            float4 *dst = wring + (size_t)st * CH4;
            if (is.kind == PH_ATT) {
                const long long np = min((long long)TP, is.e - icur);
                if (lane == 0) {
                    const uint32_t bytes = (uint32_t)np * hs * 4u;
                    mbar_arrive_expect_tx(&bars[st], 2u * bytes);
                    bulk_g2s_nohint(dst, is.kb + (size_t)icur * hs, bytes, &bars[st]);
                    bulk_g2s_nohint(dst + (size_t)TP * hs4, is.vb + (size_t)icur * hs, bytes, &bars[st]);
                }
                icur += np;
            } else {
                int pi, len;
                locate(is, icur, CH4, pi, len);
                if (lane == 0) {
                    const Piece pc = piece(is, pi);
                    mbar_arrive_expect_tx(&bars[st], (uint32_t)len * 16u);
                    if (hint)
                        bulk_g2s(dst, pc.src + (icur - pc.f0), (uint32_t)len * 16u, &bars[st], pol);
                    else
                        bulk_g2s_nohint(dst, pc.src + (icur - pc.f0), (uint32_t)len * 16u, &bars[st]);
                }
                icur += len;
            }
            ++n_iss;
            advance();
        }
    };
    // Waits for the next copy of the stream; false if it gave up.
    auto take = [&]() -> const float4 * {
        const int st = st_con;
        if (!mbar_wait(&bars[st], (con_par >> st) & 1u, p.err)) return nullptr;
        return wring + (size_t)st * CH4;
    };
    auto release = [&]() {
        __syncwarp();
        con_par ^= 1u << st_con;
        st_con = st_con + 1 == S ? 0 : st_con + 1;
        ++n_con;
        pump();
    };
    pump();

    // Leaves after a failed wait: every copy still in flight lands first.
    auto drain = [&]() {
        int st = st_con;
        uint32_t par = con_par;
        for (long long j = n_con; j < n_iss; ++j) {
            (void)mbar_wait(&bars[st], (par >> st) & 1u, p.err);
            par ^= 1u << st;
            st = st + 1 == S ? 0 : st + 1;
        }
    };
    // Grid-wide barrier number k of the step; false if this CTA must stop.
    auto grid_sync = [&](int k) -> bool {
        __syncthreads();
        if (tid == 0 && !fx.abort) {
            // release this CTA's writes (ordered before by the CTA barrier), arrive
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(&p.step->sync_count) : "memory");
            const unsigned target = (unsigned)(k + 1) * (unsigned)G;
            if (ld_acquire_gpu(&p.step->sync_count) < target) {
                const uint64_t t0 = globaltimer_ns();
                for (uint32_t i = 1;; ++i) {
                    if (ld_acquire_gpu(&p.step->sync_count) >= target) break;
                    if ((i & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
                        atomicOr(p.err, L2_DEV_ERR_TIMEOUT);
                        fx.abort = 1;
                        break;
                    }
                }
            }
        }
        __syncthreads();
        return !fx.abort;
    };

    int nbar = 0;
    for (int ph = 0; ph < NPH; ++ph) {
        Seg cs;
        make_seg(p, ph, pos, warp, cs);
        bool ok = true;
        if (cs.kind != PH_ATT) {
            // ---- GEMV phase: input vector into shared memory ----
            // RMSNorm phases keep g * x in shared memory and scale each row's
            // dot product by 1/rms at the end: one CTA barrier instead of three.
            const int n4 = cs.n4;
            const bool norm = cs.kind == PH_QKV || cs.kind == PH_W13 || cs.kind == PH_CLS;
            if (lane == 0) {
                fx.head_row[warp] = -1;
                fx.tail_row[warp] = -1;
            }
            if (!norm) {
                const float4 *in4 = reinterpret_cast<const float4 *>(cs.kind == PH_WO ? p.xb : p.hb);
                for (int i = tid; i < n4; i += kNT) xs[i] = __ldcg(in4 + i);
            } else {
                const float *src = p.x;
                const bool from_emb = cs.kind == PH_QKV && cs.layer == 0;
                if (from_emb) src = p.emb + (size_t)p.step->token[0] * p.dim;
                const float4 *s4 = reinterpret_cast<const float4 *>(src);
                const float *gw = cs.kind == PH_QKV ? p.rms_att + (size_t)cs.layer * p.dim
                                  : cs.kind == PH_W13 ? p.rms_ffn + (size_t)cs.layer * p.dim
                                                      : p.rms_final;
                const float4 *g4 = reinterpret_cast<const float4 *>(gw);
                float ss = 0.f;
                for (int i = tid; i < n4; i += kNT) {
                    const float4 v = from_emb ? s4[i] : __ldcg(s4 + i), g = g4[i];
                    xs[i] = make_float4(g.x * v.x, g.y * v.y, g.z * v.z, g.w * v.w);
                    ss = fmaf(v.x, v.x, ss);
                    ss = fmaf(v.y, v.y, ss);
                    ss = fmaf(v.z, v.z, ss);
                    ss = fmaf(v.w, v.w, ss);
                }
                if (from_emb && blockIdx.x == 0) {
                    float4 *x4 = reinterpret_cast<float4 *>(p.x);
                    for (int i = tid; i < n4; i += kNT) x4[i] = s4[i];
                }
                ss = warp_sum(ss);
                if (lane == 0) fx.red[warp] = ss;
            }
            __syncthreads();
            float inv = 1.f;
            if (norm) {
                float t = 0.f;
                for (int w = 0; w < kNW; ++w) t += fx.red[w];
                inv = 1.0f / sqrtf(t / (float)p.dim + 1e-5f);
            }

            // ---- stream this warp's weight words ----
            float acc = 0.f;
            bool started = false, pending = false;
            int cur_row = -1, cpi = -1, r = 0, rs = 0, re = 0;
#pragma unroll 1
            for (long long fc = cs.b; fc < cs.e;) {
                int pi, len;
                locate(cs, fc, CH4, pi, len);
                const float4 *buf = take();
                if (!buf) {
                    ok = false;
                    break;
                }
                const Piece pc = piece(cs, pi);
                const int lf = (int)(fc - pc.f0), lend = lf + len;
                if (pi != cpi) {
                    cpi = pi;
                    r = lf / n4;
                    rs = r * n4;
                    re = rs + n4;
                }
                int a = lf;
                while (a < lend) {
                    if (a == re) {
                        ++r;
                        rs = re;
                        re += n4;
                    }
                    const int b = lend < re ? lend : re;
                    if (a == rs) started = true;
                    cur_row = pc.yoff + r;
                    const float4 *wr = buf + (a - lf);
                    const float4 *xr = xs + (a - rs);
                    const int cnt = b - a;
#pragma unroll 4
                    for (int i = lane; i < cnt; i += 32) acc = dot4(wr[i], xr[i], acc);
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
                fc += len;
                release();
            }
            if (!ok) {
                if (lane == 0) fx.abort = 1;
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
            if (fx.abort) {
                drain();
                return;
            }
            // Rows split between warps: the warp that began row r left its part
            // as a tail; the following warps that continued it (possibly with
            // warps of empty ranges between them) left heads.  Thread w sums
            // warp w's tail and those heads in warp order.
            if (tid < kNW && fx.tail_row[tid] >= 0) {
                const int row = fx.tail_row[tid];
                float v = fx.tail_val[tid];
                for (int w2 = tid + 1; w2 < kNW; ++w2)
                    if (fx.head_row[w2] == row) v += fx.head_val[w2];
                ys[row] = v;
            }
            __syncthreads();

            // ---- epilogue ----
            const int R = cs.R, vr0 = cs.vr0;
            if (cs.kind == PH_QKV) {
                const int half = hs >> 1;
                const float2 *rr = p.rope + (size_t)pos * half;
                for (int i = tid; i < (R >> 1); i += kNT) {
                    const int j = 2 * i, v = vr0 + j;
                    const float y0 = ys[j] * inv, y1 = ys[j + 1] * inv;
                    if (v < p.dim) {
                        const float2 c2 = rr[(v % hs) >> 1];
                        p.q[v] = y0 * c2.x - y1 * c2.y;
                        p.q[v + 1] = y0 * c2.y + y1 * c2.x;
                    } else {
                        const bool is_k = v < p.dim + p.kv_dim;
                        const int cc = is_k ? v - p.dim : v - p.dim - p.kv_dim;
                        const int g = cc / hs, d = cc % hs;
                        const size_t idx = (((size_t)cs.layer * p.n_kv_heads + g) * p.seq_len + pos) * hs + d;
                        if (is_k) {
                            const float2 c2 = rr[d >> 1];
                            p.kcache[idx] = y0 * c2.x - y1 * c2.y;
                            p.kcache[idx + 1] = y0 * c2.y + y1 * c2.x;
                        } else {
                            p.vcache[idx] = y0;
                            p.vcache[idx + 1] = y1;
                        }
                    }
                }
            } else if (cs.kind == PH_WO || cs.kind == PH_W2) {
                for (int j = tid; j < R; j += kNT) p.x[vr0 + j] = __ldcg(p.x + vr0 + j) + ys[j];
            } else if (cs.kind == PH_W13) {
                for (int j = tid; j < R; j += kNT) p.hb[vr0 + j] = silu(ys[j] * inv) * (ys[R + j] * inv);
            } else {
                float *user = p.step->logits_out;
                for (int j = tid; j < R; j += kNT) {
                    const float y = ys[j] * inv;
                    p.logits[vr0 + j] = y;
                    if (user) user[vr0 + j] = y;
                }
            }
        } else if (cs.g >= 0) {
            // ---- attention item: KV head g, chunk c of its positions ----
            const int H = p.n_heads, KV = p.n_kv_heads, g = cs.g;
            const int h0 = (g * H + KV - 1) / KV, h1 = ((g + 1) * H + KV - 1) / KV;
            const int nq = h1 - h0;
            const int LP = p.lp, RPI = 32 / LP, rg = lane / LP, c4 = lane % LP;
            const bool lane_on = c4 < hs4;
            float4 q4[GQ], acc[GQ];
            float m[GQ], l[GQ];
#pragma unroll
            for (int j = 0; j < GQ; ++j) {
                q4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < nq && lane_on) q4[j] = __ldcg(reinterpret_cast<const float4 *>(p.q + (size_t)(h0 + j) * hs) + c4);
                m[j] = -CUDART_INF_F;
                l[j] = 0.f;
                acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            // Sum over the LP lanes of a row group (LP a power of two <= 32):
            // all five butterfly steps unrolled, the ones at or above LP off.
            auto group_sum = [&](float d) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    if (o < LP) d += __shfl_xor_sync(0xffffffffu, d, o);
                return d;
            };
            // Scores np rows of K in shared memory (row stride hs4 words)
            // against the group's queries and folds them into the running
            // softmax states.
            auto fold = [&](const float4 *Ks, const float4 *Vs, int np) {
#pragma unroll 1
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
                            const float d = group_sum(dot4(q4[j], kv, 0.f));
                            sc[u][j] = row_on ? d * p.scale : -CUDART_INF_F;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < GQ; ++j) {
                        if (j >= nq) continue;
                        float mx = sc[0][j];
#pragma unroll
                        for (int u = 1; u < kPPG; ++u) mx = fmaxf(mx, sc[u][j]);
                        const float mn = fmaxf(m[j], mx);
                        if (mn == -CUDART_INF_F) continue;
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
            };
#pragma unroll 1
            for (long long tc = cs.b; tc < cs.e;) {
                const int np = (int)min((long long)TP, cs.e - tc);
                const float4 *buf = take();
                if (!buf) {
                    ok = false;
                    break;
                }
                fold(buf, buf + (size_t)TP * hs4, np);
                tc += np;
                release();
            }
            // the row written during this step, read from L2 by row group 0
            if (ok && cs.wt0 <= pos && pos < cs.wt1) {
                float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
                if (rg == 0 && lane_on) {
                    kv = __ldcg(reinterpret_cast<const float4 *>(cs.kb + (size_t)pos * hs) + c4);
                    vv = __ldcg(reinterpret_cast<const float4 *>(cs.vb + (size_t)pos * hs) + c4);
                }
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    const float d = group_sum(dot4(q4[j], kv, 0.f));
                    if (rg != 0 || j >= nq) continue;
                    const float sc = d * p.scale, mn = fmaxf(m[j], sc);
                    const float corr = expf(m[j] - mn), pe = expf(sc - mn);
                    l[j] = l[j] * corr + pe;
                    acc[j] = make_float4(fmaf(pe, vv.x, acc[j].x * corr), fmaf(pe, vv.y, acc[j].y * corr),
                                         fmaf(pe, vv.z, acc[j].z * corr), fmaf(pe, vv.w, acc[j].w * corr));
                    m[j] = mn;
                }
            }
            if (!ok && lane == 0) fx.abort = 1;

            // merge the row groups of the warp (lanes LP apart share a column word)
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                if (o < LP) continue;
#pragma unroll
                for (int j = 0; j < GQ; ++j) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m[j], o);
                    const float l2v = __shfl_xor_sync(0xffffffffu, l[j], o);
                    float4 a2;
                    a2.x = __shfl_xor_sync(0xffffffffu, acc[j].x, o);
                    a2.y = __shfl_xor_sync(0xffffffffu, acc[j].y, o);
                    a2.z = __shfl_xor_sync(0xffffffffu, acc[j].z, o);
                    a2.w = __shfl_xor_sync(0xffffffffu, acc[j].w, o);
                    const float M = fmaxf(m[j], m2);
                    if (M == -CUDART_INF_F) continue;
                    const float ea = expf(m[j] - M), eb = expf(m2 - M);
                    l[j] = l[j] * ea + l2v * eb;
                    acc[j].x = acc[j].x * ea + a2.x * eb;
                    acc[j].y = acc[j].y * ea + a2.y * eb;
                    acc[j].z = acc[j].z * ea + a2.z * eb;
                    acc[j].w = acc[j].w * ea + a2.w * eb;
                    m[j] = M;
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
            __syncthreads();
            if (fx.abort) {
                drain();
                return;
            }
            // merge the warps in warp order
            const int na = cs.n_active, NC = p.n_chunks;
            auto merge_warps = [&](int j, int w4, float &mm, float &ll, float4 &aa) {
                mm = -CUDART_INF_F;
                ll = 0.f;
                aa = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int w = 0; w < kNW; ++w) {
                    const float m2 = mrg[(w * GQ + j) * 2], l2v = mrg[(w * GQ + j) * 2 + 1];
                    const float M = fmaxf(mm, m2);
                    if (M == -CUDART_INF_F) continue;
                    const float4 a2 = accs[(size_t)(w * GQ + j) * hs4 + w4];
                    const float ea = expf(mm - M), eb = expf(m2 - M);
                    ll = ll * ea + l2v * eb;
                    aa = make_float4(aa.x * ea + a2.x * eb, aa.y * ea + a2.y * eb, aa.z * ea + a2.z * eb,
                                     aa.w * ea + a2.w * eb);
                    mm = M;
                }
            };
            if (na == 1) {
                for (int idx = tid; idx < nq * hs4; idx += kNT) {
                    const int j = idx / hs4, w4 = idx % hs4;
                    float mm, ll;
                    float4 aa;
                    merge_warps(j, w4, mm, ll, aa);
                    const float inv = 1.0f / ll;
                    reinterpret_cast<float4 *>(p.xb + (size_t)(h0 + j) * hs)[w4] =
                        make_float4(aa.x * inv, aa.y * inv, aa.z * inv, aa.w * inv);
                }
            } else {
                for (int idx = tid; idx < nq * hs4; idx += kNT) {
                    const int j = idx / hs4, w4 = idx % hs4;
                    float mm, ll;
                    float4 aa;
                    merge_warps(j, w4, mm, ll, aa);
                    const size_t slot = (size_t)(h0 + j) * NC + cs.c;
                    reinterpret_cast<float4 *>(p.ws_acc + slot * hs)[w4] = aa;
                    if (w4 == 0) {
                        p.ws_ml[slot * 2 + 0] = mm;
                        p.ws_ml[slot * 2 + 1] = ll;
                    }
                }
                __threadfence();
                __syncthreads();
                if (tid == 0) {
                    const unsigned t = atomicAdd(&p.tickets[g], 1u);
                    fx.last = (t == (unsigned)(na - 1)) ? 1 : 0;
                }
                __syncthreads();
                if (fx.last) {
                    __threadfence();
                    if (tid < nq) {
                        const int j = tid;
                        float M = -CUDART_INF_F;
                        for (int cc = 0; cc < na; ++cc)
                            M = fmaxf(M, __ldcg(p.ws_ml + ((size_t)(h0 + j) * NC + cc) * 2));
                        float Ls = 0.f;
                        for (int cc = 0; cc < na; ++cc) {
                            const size_t sl = (size_t)(h0 + j) * NC + cc;
                            Ls += __ldcg(p.ws_ml + sl * 2 + 1) * expf(__ldcg(p.ws_ml + sl * 2) - M);
                        }
                        fin[j * 2] = M;
                        fin[j * 2 + 1] = Ls;
                    }
                    __syncthreads();
                    for (int idx = tid; idx < nq * hs4; idx += kNT) {
                        const int j = idx / hs4, w4 = idx % hs4;
                        const float M = fin[j * 2], inv = 1.0f / fin[j * 2 + 1];
                        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int cc = 0; cc < na; ++cc) {
                            const size_t sl = (size_t)(h0 + j) * NC + cc;
                            const float e = expf(__ldcg(p.ws_ml + sl * 2) - M);
                            const float4 a = __ldcg(reinterpret_cast<const float4 *>(p.ws_acc + sl * hs) + w4);
                            o.x += a.x * e;
                            o.y += a.y * e;
                            o.z += a.z * e;
                            o.w += a.w * e;
                        }
                        reinterpret_cast<float4 *>(p.xb + (size_t)(h0 + j) * hs)[w4] =
                            make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
                    }
                    if (tid == 0) p.tickets[g] = 0u;
                }
            }
        }
        if (ph + 1 < NPH && !grid_sync(nbar++)) {
            drain();
            return;
        }
    }
}

// ---------------------------------------------------------------- host side

namespace {
typedef void (*StepFn)(const StepKParams);

StepFn pick(int gq) {
    switch (gq) {
        case 1: return step_kernel<1>;
        case 2: return step_kernel<2>;
        case 4: return step_kernel<4>;
        case 8: return step_kernel<8>;
    }
    return nullptr;
}
}  // namespace

int step_kernel_threads() { return kNT; }

size_t step_kernel_smem(int gq, int head_size, int xs_floats, int ys_floats, int stages, int ch4) {
    const size_t gemv = (size_t)xs_floats * 4 + align_up((size_t)ys_floats * 4, 16);
    const size_t att = (size_t)kNW * gq * (head_size / 4) * 16 + ((size_t)kNW * gq * 2 + (size_t)gq * 2) * 4;
    return kFixedBytes + (size_t)kNW * stages * ch4 * 16 + (gemv > att ? gemv : att);
}

int step_kernel_ring(int gq, int head_size, int xs_floats, int ys_floats, int stages, int max_ch4) {
    if (stages < 1 || stages > kMaxStages) return 0;
    const size_t rest = step_kernel_smem(gq, head_size, xs_floats, ys_floats, stages, 0);
    if (rest >= 227 * 1024) return 0;
    long long ch4 = (long long)(227 * 1024 - rest) / ((long long)kNW * stages * 16);
    if (ch4 > max_ch4) ch4 = max_ch4;
    ch4 &= ~7LL;
    // two cache rows (one K, one V) must fit a buffer
    if (ch4 * 4 < 2LL * head_size) return 0;
    return (int)ch4;
}

cudaError_t step_kernel_init() {
    for (int gq : {1, 2, 4, 8}) {
        cudaError_t e = cudaFuncSetAttribute(pick(gq), cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

int step_kernel_ctas_per_sm(int gq, size_t smem) {
    int n = 0;
    StepFn fn = pick(gq);
    if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kNT, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_step_kernel(int gq, const StepKParams &p, int grid, size_t smem, cudaStream_t stream) {
    StepFn fn = pick(gq);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<StepKParams *>(&p)};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(fn), args);
}

}  // namespace l2
