// Fused matrix-vector kernels for a step of B independent sequences (B >= 2):
// Y[b][r] = sum_k W[r][k] v_b[k], with the same fused prologues and epilogues
// as the batch-1 kernels in gemv.cu (RMSNorm, RoPE + KV write, SwiGLU,
// residual, classifier), each sequence at its own position.
//
// Every weight is read from HBM once per step for all B sequences, so the
// arithmetic intensity is B/2 flop per weight byte: at B = 16 the step is
// still bandwidth-bound, at B = 64 it is bound by the fp32 CUDA cores.
//
// Design.  CTA c owns a balanced range of output rows (all pieces of it, e.g.
// its W1 rows and the same W3 rows).  The K dimension is walked in tiles of
// 64 columns: per tile, the CTA's row segments (256 B each) and the B input
// segments land in shared memory by 1-D bulk async copies (TMA) on one
// mbarrier per ring stage.  Each thread owns 4 rows x 8 sequences of the
// output (32 accumulators, two such tiles at most) for a subset of the tile's
// 16-byte column words; per word it loads 4 weight and 8 input words and does
// 128 FMAs.  Partial sums of the column groups are added in a fixed order at
// the end, so results do not depend on timing.  RMSNorm: the gain is applied
// to the input tile in shared memory, the 1/rms factor of each sequence to its
// outputs; the sums of squares come from the residual kernels' epilogues
// (per-CTA partials added in CTA order), so no CTA re-reads all of x.
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kBT = 256;        // threads
constexpr int kTK = 64;         // K columns per tile
constexpr int kTKP = kTK + 4;   // padded shared-memory row (floats): rows start 16 B apart in bank terms
constexpr int kRR = 4;          // rows per thread tile
constexpr int kBB = 8;          // sequences per thread tile
constexpr int kMT = 2;          // thread tiles per thread at most
constexpr int kMaxStages = 4;

struct BPiece {
    const float *src;  // first row of the piece
    int rows;
    int yoff;          // local row of the piece's first row
};

struct BatchFixed {
    uint64_t bars[kMaxStages];
    BPiece pieces[3];
    int npieces;
    int failed;
    float inv[kMaxBatch];
};

__host__ __device__ constexpr size_t fixed_b_bytes() { return (sizeof(BatchFixed) + 127) / 128 * 128; }

__device__ __forceinline__ float silu_b(float v) { return v / (1.0f + expf(-v)); }

__host__ __device__ inline int kgroups_for(int tiles) {
    int kg = 1;
    while (kg < 16 && tiles * kg * 2 <= kBT) kg <<= 1;
    return kg;
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kBT, 1) gemv_batched_kernel(const GemvParams p, int stages) {
    extern __shared__ __align__(128) unsigned char smem[];
    auto &fx = *reinterpret_cast<BatchFixed *>(smem);
    float *region = reinterpret_cast<float *>(smem + fixed_b_bytes());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.batch, n = p.n;

    const long long u0 = (long long)blockIdx.x * p.total_units / gridDim.x;
    const long long u1 = (long long)(blockIdx.x + 1) * p.total_units / gridDim.x;
    const int vr0 = (int)(u0 * p.unit_rows);
    const int R = (int)((u1 - u0) * p.unit_rows);
    const int RT = (MODE == GEMV_W13) ? 2 * R : R;
    const int stage_floats = (RT + B) * kTKP;
    const int NKT = (n + kTK - 1) / kTK;

    if (tid == 0) {
        int np = 0;
        if (R > 0) {
            if (MODE == GEMV_QKV) {
                const float *mats[3] = {p.mat0, p.mat1, p.mat2};
                const int rws[3] = {p.rows0, p.rows1, p.rows2};
                int b0 = 0;
                for (int m = 0; m < 3; ++m) {
                    const int lo = max(vr0, b0), hi = min(vr0 + R, b0 + rws[m]);
                    if (lo < hi) fx.pieces[np++] = {mats[m] + (size_t)(lo - b0) * n, hi - lo, lo - vr0};
                    b0 += rws[m];
                }
            } else if (MODE == GEMV_W13) {
                fx.pieces[0] = {p.mat0 + (size_t)vr0 * n, R, 0};
                fx.pieces[1] = {p.mat1 + (size_t)vr0 * n, R, R};
                np = 2;
            } else {
                fx.pieces[0] = {p.mat0 + (size_t)vr0 * n, R, 0};
                np = 1;
            }
        }
        fx.npieces = np;
        fx.failed = 0;
        for (int i = 0; i < stages; ++i) mbar_init(&fx.bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (RT == 0) return;

    // Global address of local weight row i.
    auto row_src = [&](int i) -> const float * {
        int pi = 0;
        while (pi + 1 < fx.npieces && i >= fx.pieces[pi + 1].yoff) ++pi;
        return fx.pieces[pi].src + (size_t)(i - fx.pieces[pi].yoff) * n;
    };
    // Global address of sequence b's input vector.
    auto in_src = [&](int b) -> const float * {
        if (MODE == GEMV_RESID) return p.in_vec + (size_t)b * n;
        if (MODE == GEMV_QKV && p.layer == 0) return p.emb + (size_t)p.step->token[b] * p.dim;
        return p.x + (size_t)b * n;
    };
    const bool in_ready_early = (MODE == GEMV_QKV && p.layer == 0);  // embedding rows: read-only

    // Issue K tile kt into stage s (warp 0).  With `weights_only`, only the
    // weight rows (which do not depend on the previous kernel).
    auto issue = [&](int kt, int s, bool weights_only, bool inputs_only) {
        const int k0 = kt * kTK, len = min(kTK, n - k0);
        const uint32_t bytes = (uint32_t)len * 4u;
        float *W = region + (size_t)s * stage_floats;
        float *X = W + (size_t)RT * kTKP;
        if (lane == 0) {
            // One arrival per stage use.  A weights-only request only raises the
            // expected bytes, so the stage cannot complete before the inputs'
            // request (which arrives) has been made.
            if (weights_only)
                asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&fx.bars[s])),
                             "r"((uint32_t)RT * bytes)
                             : "memory");
            else
                mbar_arrive_expect_tx(&fx.bars[s], (inputs_only ? 0u : (uint32_t)RT * bytes) + (uint32_t)B * bytes);
        }
        __syncwarp();
        if (!inputs_only)
            for (int i = lane; i < RT; i += 32) bulk_g2s_nohint(W + (size_t)i * kTKP, row_src(i) + k0, bytes, &fx.bars[s]);
        if (!weights_only)
            for (int b = lane; b < B; b += 32) bulk_g2s_nohint(X + (size_t)b * kTKP, in_src(b) + k0, bytes, &fx.bars[s]);
    };

    // Weights of the first stages before waiting on the previous kernel.
    const int pre = min(stages, NKT);
    if (warp == 0)
        for (int kt = 0; kt < pre; ++kt) issue(kt, kt, !in_ready_early, false);

    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0 && !in_ready_early)
        for (int kt = 0; kt < pre; ++kt) issue(kt, kt, false, true);

    // 1/rms of each sequence
    if (MODE != GEMV_RESID) {
        if (MODE == GEMV_QKV && p.layer == 0) {
            for (int b = warp; b < B; b += kBT / 32) {
                const float4 *e4 = reinterpret_cast<const float4 *>(in_src(b));
                float ss = 0.f;
                for (int i = lane; i < n / 4; i += 32) {
                    const float4 v = e4[i];
                    ss = fmaf(v.x, v.x, ss);
                    ss = fmaf(v.y, v.y, ss);
                    ss = fmaf(v.z, v.z, ss);
                    ss = fmaf(v.w, v.w, ss);
                }
                ss = warp_sum(ss);
                if (lane == 0) fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
                if (blockIdx.x == 0) {
                    float4 *x4 = reinterpret_cast<float4 *>(p.x + (size_t)b * n);
                    for (int i = lane; i < n / 4; i += 32) x4[i] = e4[i];
                }
            }
        } else {
            for (int b = tid; b < B; b += kBT) {
                float ss = 0.f;
                for (int i = 0; i < p.ss_parts; ++i) ss += __ldcg(p.ss_part + (size_t)i * B + b);
                fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
            }
        }
    }

    // thread tiles
    const int TRG = (RT + kRR - 1) / kRR, TBG = (B + kBB - 1) / kBB, T = TRG * TBG;
    const int KG = kgroups_for(T);
    const int kg = tid % KG, t0 = tid / KG, tstride = kBT / KG;
    float acc[kMT][kRR][kBB];
#pragma unroll
    for (int m = 0; m < kMT; ++m)
#pragma unroll
        for (int i = 0; i < kRR; ++i)
#pragma unroll
            for (int j = 0; j < kBB; ++j) acc[m][i][j] = 0.f;

    bool ok = true;
#pragma unroll 1
    for (int kt = 0; kt < NKT; ++kt) {
        const int s = kt % stages;
        if (!mbar_wait(&fx.bars[s], (uint32_t)(kt / stages) & 1u, p.err)) {
            ok = false;
            fx.failed = 1;
        }
        __syncthreads();
        if (fx.failed) {
            ok = false;
            break;
        }
        const int k0 = kt * kTK, len = min(kTK, n - k0), len4 = len >> 2;
        const float *W = region + (size_t)s * stage_floats;
        float *X = const_cast<float *>(W) + (size_t)RT * kTKP;
        if (MODE != GEMV_RESID) {
            for (int e = tid; e < B * len; e += kBT) {
                const int b = e / len, k = e - b * len;
                X[(size_t)b * kTKP + k] *= __ldg(p.norm_w + k0 + k);
            }
            __syncthreads();
        }
#pragma unroll
        for (int m = 0; m < kMT; ++m) {
            const int t = t0 + m * tstride;
            if (t < T) {
                const int rg = t % TRG, bg = t / TRG;
                const float4 *wr[kRR];
                const float4 *xr[kBB];
#pragma unroll
                for (int i = 0; i < kRR; ++i)
                    wr[i] = reinterpret_cast<const float4 *>(W + (size_t)min(rg * kRR + i, RT - 1) * kTKP);
#pragma unroll
                for (int j = 0; j < kBB; ++j)
                    xr[j] = reinterpret_cast<const float4 *>(X + (size_t)min(bg * kBB + j, B - 1) * kTKP);
#pragma unroll 1
                for (int k4 = kg; k4 < len4; k4 += KG) {
                    float4 w4[kRR], x4[kBB];
#pragma unroll
                    for (int i = 0; i < kRR; ++i) w4[i] = wr[i][k4];
#pragma unroll
                    for (int j = 0; j < kBB; ++j) x4[j] = xr[j][k4];
#pragma unroll
                    for (int i = 0; i < kRR; ++i)
#pragma unroll
                        for (int j = 0; j < kBB; ++j) acc[m][i][j] = dot4(w4[i], x4[j], acc[m][i][j]);
                }
            }
        }
        __syncthreads();
        if (warp == 0 && kt + stages < NKT) issue(kt + stages, s, false, false);
    }
    if (!ok) {
        // Let the copies already requested land (bounded waits) before leaving.
        if (tid == 0)
            for (int j = 0; j < NKT && j < stages; ++j) (void)mbar_wait(&fx.bars[j], 0u, p.err);
        return;
    }

    // add up the column groups in a fixed order
    float *red = region;  // [KG][RT][B]
#pragma unroll
    for (int m = 0; m < kMT; ++m) {
        const int t = t0 + m * tstride;
        if (t < T) {
            const int rg = t % TRG, bg = t / TRG;
#pragma unroll
            for (int i = 0; i < kRR; ++i)
#pragma unroll
                for (int j = 0; j < kBB; ++j) {
                    const int r = rg * kRR + i, b = bg * kBB + j;
                    if (r < RT && b < B) red[((size_t)kg * RT + r) * B + b] = acc[m][i][j];
                }
        }
    }
    __syncthreads();
    float *ys = region + (size_t)KG * RT * B;  // [RT][B]
    for (int e = tid; e < RT * B; e += kBT) {
        float v = 0.f;
        for (int g = 0; g < KG; ++g) v += red[(size_t)g * RT * B + e];
        if (MODE != GEMV_RESID) v *= fx.inv[e % B];
        ys[e] = v;
    }
    __syncthreads();

    // ---- epilogue ----
    if (MODE == GEMV_QKV) {
        const int hs = p.head_size, half = hs >> 1;
        for (int e = tid; e < (R >> 1) * B; e += kBT) {
            const int pi = e / B, b = e - pi * B;
            const int j = 2 * pi, v = vr0 + j;
            const float y0 = ys[(size_t)j * B + b], y1 = ys[(size_t)(j + 1) * B + b];
            const int pos = p.step->pos[b];
            const float2 *rr = p.rope + (size_t)pos * half;
            if (v < p.dim) {
                const float2 cs = rr[(v % hs) >> 1];
                float *q = p.q + (size_t)b * p.dim;
                q[v] = y0 * cs.x - y1 * cs.y;
                q[v + 1] = y0 * cs.y + y1 * cs.x;
            } else {
                const bool is_k = v < p.dim + p.kv_dim;
                const int c = is_k ? v - p.dim : v - p.dim - p.kv_dim;
                const int g = c / hs, d = c % hs;
                const size_t idx =
                    ((((size_t)b * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + pos) * hs + d;
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
    } else if (MODE == GEMV_W13) {
        const int hidden = p.total_units;
        for (int e = tid; e < R * B; e += kBT) {
            const int r = e / B, b = e - r * B;
            p.hb[(size_t)b * hidden + vr0 + r] = silu_b(ys[e]) * ys[(size_t)(R + r) * B + b];
        }
    } else if (MODE == GEMV_RESID) {
        const int dim = p.total_units;
        for (int e = tid; e < R * B; e += kBT) {
            const int r = e / B, b = e - r * B;
            float *xp = p.x + (size_t)b * dim + vr0 + r;
            const float nv = *xp + ys[e];
            *xp = nv;
            ys[e] = nv;
        }
        __syncthreads();
        for (int b = tid; b < B; b += kBT) {
            float ss = 0.f;
            for (int r = 0; r < R; ++r) ss = fmaf(ys[(size_t)r * B + b], ys[(size_t)r * B + b], ss);
            p.ss_part[(size_t)blockIdx.x * B + b] = ss;
        }
    } else {
        float *user = p.step->logits_out;
        const int V = p.total_units;
        for (int e = tid; e < R * B; e += kBT) {
            const int r = e / B, b = e - r * B;
            p.logits[(size_t)b * V + vr0 + r] = ys[e];
            if (user) user[(size_t)b * V + vr0 + r] = ys[e];
        }
    }
}

// ---------------------------------------------------------------- host side

size_t gemv_batched_smem(int rows_max, int batch, int *stages) {
    const size_t stage = (size_t)(rows_max + batch) * kTKP * 4;
    int st = kMaxStages;
    const size_t limit = 227 * 1024 - fixed_b_bytes();
    while (st > 2 && st * stage > limit) --st;
    *stages = st;
    // After the K loop the same memory holds the column-group partials
    // [KG][RT][B] and the sums [RT][B]; KG*RT <= max(1024, RT) for any RT.
    const size_t rb = (size_t)rows_max * batch;
    const size_t red = 4 * ((rb > 8192 ? rb : 8192) + rb);
    return fixed_b_bytes() + (st * stage > red ? st * stage : red);
}

int gemv_batched_rows_ok(int rows_max, int batch) {
    const int T = ((rows_max + kRR - 1) / kRR) * ((batch + kBB - 1) / kBB);
    return T <= kMT * kBT && batch <= kMaxBatch;
}

cudaError_t gemv_batched_init() {
    void *fns[] = {reinterpret_cast<void *>(gemv_batched_kernel<GEMV_QKV>),
                   reinterpret_cast<void *>(gemv_batched_kernel<GEMV_RESID>),
                   reinterpret_cast<void *>(gemv_batched_kernel<GEMV_W13>),
                   reinterpret_cast<void *>(gemv_batched_kernel<GEMV_CLS>)};
    for (void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv_batched(int mode, const GemvParams &p, int grid, size_t smem, int stages, cudaStream_t stream,
                                bool pdl) {
    void *fn = nullptr;
    switch (mode) {
        case GEMV_QKV: fn = reinterpret_cast<void *>(gemv_batched_kernel<GEMV_QKV>); break;
        case GEMV_RESID: fn = reinterpret_cast<void *>(gemv_batched_kernel<GEMV_RESID>); break;
        case GEMV_W13: fn = reinterpret_cast<void *>(gemv_batched_kernel<GEMV_W13>); break;
        case GEMV_CLS: fn = reinterpret_cast<void *>(gemv_batched_kernel<GEMV_CLS>); break;
        default: return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kBT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<GemvParams *>(&p), &stages};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace l2
