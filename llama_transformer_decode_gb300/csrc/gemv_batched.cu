// Fused matrix-vector kernels for a step of B independent sequences (B >= 2):
// Y[b][r] = sum_k W[r][k] v_b[k], with the same fused prologues and epilogues
// as the batch-1 kernels in gemv.cu (RMSNorm, RoPE + KV write, SwiGLU,
// residual, classifier), each sequence at its own position.
//
// Every weight is read from HBM once per step for all B sequences, so the
// arithmetic intensity is B/2 flop per weight byte: at B = 16 the step is
// still bandwidth-bound, at B = 64 it is bound by the fp32 CUDA cores.
//
// Design.  CTA c owns a balanced range of rows of one matrix (for W1/W3 the
// same rows of both).  K is walked in tiles of up to 256 columns: per tile,
// one 2-D tensor copy (TMA, cp.async.bulk.tensor) brings the CTA's rows x tile
// columns of each weight matrix into shared memory and one brings the B input
// rows x tile columns, all completing on one mbarrier per ring stage.  (Copies
// per row would be many small TMA operations, and the operation count, not the
// bytes, then limits the rate.)  Each warp owns an output tile of 8 rows x 8
// sequences (64 accumulators per lane); its lanes split the columns, so every
// shared-memory read is 32 consecutive 16-byte words of one row, and per word
// a lane loads 8 weight and 8 input words for 256 FMAs.  A CTA holds at most
// 8 tiles, so the host sizes the row ranges (and the grid) from the batch.
// Lane partials are reduced with shuffles in a fixed order.  RMSNorm: the gain
// scales the input tile in shared memory, 1/rms scales the outputs, and the
// sums of squares come from the residual kernels' epilogues (per-CTA partials
// added in CTA order), so no CTA re-reads the whole of x.
#include <cuda.h>
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kBT = 256;             // threads
constexpr int kTR = 8;               // rows per warp tile
constexpr int kTB = 8;               // sequences per warp tile
constexpr int kMaxTiles = kBT / 32;  // one warp tile per warp
constexpr int kMaxStages = 4;

struct BatchFixed {
    uint64_t bars[kMaxStages];
    int failed;
    float inv[kMaxBatch];
};

__host__ __device__ constexpr size_t fixed_b_bytes() { return (sizeof(BatchFixed) + 127) / 128 * 128; }

__device__ __forceinline__ float silu_b(float v) { return v / (1.0f + expf(-v)); }

// Raises the bytes a barrier phase waits for, without arriving on it.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// 2-D tiled tensor copy global -> shared; coordinates {column, row}.
__device__ __forceinline__ void tensor_g2s(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kBT, 1) gemv_batched_kernel(const __grid_constant__ BatchParams bp) {
    const GemvParams &p = bp.g;
    extern __shared__ __align__(128) unsigned char smem[];
    auto &fx = *reinterpret_cast<BatchFixed *>(smem);
    float *region = reinterpret_cast<float *>(smem + fixed_b_bytes());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.batch, n = p.n, tk = bp.tk, RB = bp.rows_box, stages = bp.stages;

    // ---- this CTA's matrix and rows ----
    int m = 0, cta = blockIdx.x;
    while (m < 2 && cta >= bp.part_ctas[m]) cta -= bp.part_ctas[m++];
    const int units = bp.part_units[m], nct = bp.part_ctas[m];
    const long long u0 = (long long)cta * units / nct, u1 = (long long)(cta + 1) * units / nct;
    const int r0 = (int)(u0 * p.unit_rows);        // first row within matrix m
    const int R = (int)((u1 - u0) * p.unit_rows);  // rows of this CTA (<= RB)
    const int npc = (MODE == GEMV_W13) ? 2 : 1;    // weight pieces (W1 and W3 share rows)
    const int SR = npc * RB;                       // weight rows in a stage (piece pc at row pc*RB)
    const int mrows = (MODE == GEMV_QKV) ? (m == 0 ? p.rows0 : p.rows1) : p.total_units * p.unit_rows;
    const int wrow0 = (MODE == GEMV_CLS ? 0 : p.layer * mrows) + r0;  // tensor-map row of the first row
    const int stage_floats = (SR + B) * tk;
    const int NKT = (n + tk - 1) / tk;
    const bool emb_rows = (MODE == GEMV_QKV && p.layer == 0);  // inputs gathered from the embedding table

    if (tid == 0) {
        fx.failed = 0;
        for (int i = 0; i < stages; ++i) mbar_init(&fx.bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (R <= 0) return;

    // Requests for K tile kt into stage s, by lane 0 of warp 0 (lanes of warp 0
    // for the embedding rows).  The weight half only raises the expected bytes;
    // the input half arrives, so a stage cannot complete before both halves
    // have been requested.  The weights do not depend on the previous kernel
    // and are requested before waiting on it.
    auto issue_weights = [&](int kt, int s) {
        if (lane == 0) {
            float *W = region + (size_t)s * stage_floats;
            mbar_expect_tx(&fx.bars[s], (uint32_t)(SR * tk * 4));
            for (int pc = 0; pc < npc; ++pc)
                tensor_g2s(W + (size_t)pc * RB * tk, &bp.wmap[MODE == GEMV_QKV ? m : pc], kt * tk, wrow0, &fx.bars[s]);
        }
    };
    auto issue_inputs = [&](int kt, int s) {
        float *X = region + (size_t)s * stage_floats + (size_t)SR * tk;
        const int k0 = kt * tk, len = min(tk, n - k0);
        if (emb_rows) {
            // one embedding row per sequence; columns past n stay unused
            if (lane == 0) mbar_arrive_expect_tx(&fx.bars[s], (uint32_t)(B * len * 4));
            __syncwarp();
            for (int b = lane; b < B; b += 32)
                bulk_g2s_nohint(X + (size_t)b * tk, p.emb + (size_t)p.step->token[b] * p.dim + k0, (uint32_t)len * 4u,
                                &fx.bars[s]);
        } else if (lane == 0) {
            mbar_arrive_expect_tx(&fx.bars[s], (uint32_t)(B * tk * 4));
            tensor_g2s(X, &bp.xmap, k0, 0, &fx.bars[s]);
        }
    };

    const int pre = min(stages, NKT);
    if (warp == 0)
        for (int kt = 0; kt < pre; ++kt) {
            issue_weights(kt, kt);
            if (emb_rows) issue_inputs(kt, kt);  // the embedding table is read-only
        }

    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0 && !emb_rows)
        for (int kt = 0; kt < pre; ++kt) issue_inputs(kt, kt);

    // 1/rms of each sequence
    if (MODE != GEMV_RESID) {
        if (emb_rows) {
            for (int b = warp; b < B; b += kBT / 32) {
                const float4 *e4 = reinterpret_cast<const float4 *>(p.emb + (size_t)p.step->token[b] * p.dim);
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
            // a warp per sequence; lanes add strided partials, then a fixed-order reduction
            for (int b = warp; b < B; b += kBT / 32) {
                float ss = 0.f;
                for (int i = lane; i < p.ss_parts; i += 32) ss += __ldcg(p.ss_part + (size_t)i * B + b);
                ss = warp_sum(ss);
                if (lane == 0) fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
            }
        }
    }

    // Warp w owns the output tile of stage rows 8*(w % TRG).. and sequences
    // 8*(w / TRG)..; its 32 lanes split the tile's columns.
    const int TRG = (SR + kTR - 1) / kTR, TBG = (B + kTB - 1) / kTB, T = TRG * TBG;
    const bool busy = warp < T;
    const int rg = warp % TRG, bg = warp / TRG;
    float acc[kTR][kTB];
#pragma unroll
    for (int i = 0; i < kTR; ++i)
#pragma unroll
        for (int j = 0; j < kTB; ++j) acc[i][j] = 0.f;

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
        const int k0 = kt * tk, len = min(tk, n - k0), len4 = len >> 2;
        const float *W = region + (size_t)s * stage_floats;
        float *X = const_cast<float *>(W) + (size_t)SR * tk;
        if (MODE != GEMV_RESID) {
            // the RMSNorm gain, applied to the input tile in place
            const float4 *g4 = reinterpret_cast<const float4 *>(p.norm_w + k0);
            for (int f = lane; f < len4; f += 32) {
                const float4 g = __ldg(g4 + f);
                for (int b = warp; b < B; b += kBT / 32) {
                    float4 *xv = reinterpret_cast<float4 *>(X + (size_t)b * tk) + f;
                    float4 v = *xv;
                    v.x *= g.x;
                    v.y *= g.y;
                    v.z *= g.z;
                    v.w *= g.w;
                    *xv = v;
                }
            }
            __syncthreads();
        }
        if (busy) {
            const float4 *wr[kTR];
            const float4 *xr[kTB];
#pragma unroll
            for (int i = 0; i < kTR; ++i)
                wr[i] = reinterpret_cast<const float4 *>(W + (size_t)min(rg * kTR + i, SR - 1) * tk);
#pragma unroll
            for (int j = 0; j < kTB; ++j)
                xr[j] = reinterpret_cast<const float4 *>(X + (size_t)min(bg * kTB + j, B - 1) * tk);
#pragma unroll 1
            for (int f = lane; f < len4; f += 32) {
                float4 w4[kTR], x4[kTB];
#pragma unroll
                for (int i = 0; i < kTR; ++i) w4[i] = wr[i][f];
#pragma unroll
                for (int j = 0; j < kTB; ++j) x4[j] = xr[j][f];
#pragma unroll
                for (int i = 0; i < kTR; ++i)
#pragma unroll
                    for (int j = 0; j < kTB; ++j) acc[i][j] = dot4(w4[i], x4[j], acc[i][j]);
            }
        }
        __syncthreads();
        if (warp == 0 && kt + stages < NKT) {
            issue_weights(kt + stages, s);
            issue_inputs(kt + stages, s);
        }
    }
    if (!ok) {
        // Let the copies already requested land (bounded waits) before leaving.
        if (tid == 0)
            for (int j = 0; j < NKT && j < stages; ++j) (void)mbar_wait(&fx.bars[j], 0u, p.err);
        return;
    }

    // reduce each output over the lanes; ys[stage row][sequence] in shared memory
    float *ys = region;
    if (busy) {
#pragma unroll
        for (int i = 0; i < kTR; ++i)
#pragma unroll
            for (int j = 0; j < kTB; ++j) {
                const float v = warp_sum(acc[i][j]);
                const int r = rg * kTR + i, b = bg * kTB + j;
                if (lane == 0 && r < SR && b < B) ys[(size_t)r * B + b] = (MODE != GEMV_RESID) ? v * fx.inv[b] : v;
            }
    }
    __syncthreads();

    // ---- epilogue (rows 0..R-1 of each piece) ----
    if (MODE == GEMV_QKV) {
        const int hs = p.head_size, half = hs >> 1;
        for (int e = tid; e < (R >> 1) * B; e += kBT) {
            const int pi = e / B, b = e - pi * B;
            const int j = 2 * pi;
            const float y0 = ys[(size_t)j * B + b], y1 = ys[(size_t)(j + 1) * B + b];
            const int pos = p.step->pos[b];
            const float2 *rr = p.rope + (size_t)pos * half;
            const int v = r0 + j;  // row within matrix m
            if (m == 0) {
                const float2 cs = rr[(v % hs) >> 1];
                float *q = p.q + (size_t)b * p.dim;
                q[v] = y0 * cs.x - y1 * cs.y;
                q[v + 1] = y0 * cs.y + y1 * cs.x;
            } else {
                const int g = v / hs, d = v % hs;
                const size_t idx =
                    ((((size_t)b * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + pos) * hs + d;
                if (m == 1) {
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
            p.hb[(size_t)b * hidden + r0 + r] = silu_b(ys[e]) * ys[(size_t)(RB + r) * B + b];
        }
    } else if (MODE == GEMV_RESID) {
        const int dim = p.total_units;
        for (int e = tid; e < R * B; e += kBT) {
            const int r = e / B, b = e - r * B;
            float *xp = p.x + (size_t)b * dim + r0 + r;
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
            p.logits[(size_t)b * V + r0 + r] = ys[e];
            if (user) user[(size_t)b * V + r0 + r] = ys[e];
        }
    }
}

// ---------------------------------------------------------------- host side

int gemv_batched_rows_cap(int batch) { return kTR * (kMaxTiles / ((batch + kTB - 1) / kTB)); }

size_t gemv_batched_smem(int stage_rows, int batch, int n, int *stages, int *tk) {
    // The widest K tile (fewer, bigger copies and fewer barriers) that still
    // leaves three ring stages; two stages of 64 columns at the least.
    const size_t limit = 227 * 1024 - fixed_b_bytes();
    int t = 256;
    while (t > 64 && (3 * (size_t)(stage_rows + batch) * t * 4 > limit || t >= 2 * n)) t >>= 1;
    const size_t stage = (size_t)(stage_rows + batch) * t * 4;
    int st = kMaxStages;
    while (st > 2 && st * stage > limit) --st;
    *stages = st;
    *tk = t;
    const size_t ys = (size_t)stage_rows * batch * 4;  // reuses the ring after the K loop
    return fixed_b_bytes() + (st * stage > ys ? st * stage : ys);
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

cudaError_t launch_gemv_batched(int mode, const BatchParams &bp, int grid, size_t smem, cudaStream_t stream, bool pdl) {
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
    void *args[] = {const_cast<BatchParams *>(&bp)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace l2
