// Fused matrix-vector kernels for a step of B independent sequences (B >= 2):
// Y[b][r] = sum_k W[r][k] v_b[k], with the same fused prologues and epilogues
// as the batch-1 kernels in gemv.cu (RMSNorm, RoPE + KV write, SwiGLU,
// residual, classifier), each sequence at its own position.
//
// Every weight is read from HBM once per step for all B sequences, so the
// arithmetic intensity is B/2 flop per weight byte: at B = 16 the step is
// still bandwidth-bound, at B = 64 it is bound by the fp32 CUDA cores.  Steps
// of 16 or more rows therefore run on the tensor-core kernels (gemv_tc.cu)
// unless the handle was created with L2_FLAG_NO_TC; this kernel serves 2..15.
//
// Design.  CTA c owns a balanced range of rows of one matrix (for W1/W3 the
// same rows of both), walked in blocks of a few rows; each block walks K in
// tiles of up to 256 columns, and the ring runs on across blocks.  Per tile,
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
// vector sits in shared memory and scales each weight word as it is read
// (w g x = w (g x)), 1/rms scales the outputs, and the sums of squares come
// from the residual kernels' epilogues (per-CTA partials added in CTA order),
// so no CTA re-reads the whole of x.
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
__global__ void __launch_bounds__(kBT, 1) l2dec_matvec_batched_kernel(const __grid_constant__ BatchParams bp) {
    const GemvParams &p = bp.g;
    extern __shared__ __align__(128) unsigned char smem[];
    auto &fx = *reinterpret_cast<BatchFixed *>(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.batch, n = p.n, tk = bp.tk, RB = bp.rows_box, stages = bp.stages;
    const int npc = (MODE == GEMV_W13) ? 2 : 1;  // weight pieces (W1 and W3 share rows)
    const int SR = npc * RB;                     // weight rows in a stage (piece pc at row pc*RB)
    // shared memory: fixed | gain [n] | ys [SR][B] | ring of stages [(SR + B) * tk]
    float *gain = reinterpret_cast<float *>(smem + fixed_b_bytes());
    float *ys = gain + ((MODE == GEMV_RESID) ? 0 : ((n + 31) & ~31));
    float *region = ys + (((size_t)SR * B + 31) & ~(size_t)31);

    // ---- this CTA's matrix and rows, walked in blocks of RB rows ----
    int m = 0, cta = blockIdx.x;
    while (m < 2 && cta >= bp.part_ctas[m]) cta -= bp.part_ctas[m++];
    const int units = bp.part_units[m], nct = bp.part_ctas[m];
    const long long u0 = (long long)cta * units / nct, u1 = (long long)(cta + 1) * units / nct;
    const int r0 = (int)(u0 * p.unit_rows);        // first row within matrix m
    const int R = (int)((u1 - u0) * p.unit_rows);  // rows of this CTA
    const int mrows = (MODE == GEMV_QKV) ? (m == 0 ? p.rows0 : p.rows1) : p.total_units * p.unit_rows;
    const int wrow0 = (MODE == GEMV_CLS ? 0 : p.layer * mrows) + r0;  // tensor-map row of the first row
    const int stage_floats = (SR + B) * tk;
    const int NKT = (n + tk - 1) / tk;
    const int NB = (R + RB - 1) / RB;  // row blocks
    const int NQ = NB * NKT;           // K tiles over all blocks
    const bool emb_rows = (MODE == GEMV_QKV && p.layer == 0);  // inputs gathered from the embedding table

    if (tid == 0) {
        fx.failed = 0;
        for (int i = 0; i < stages; ++i) mbar_init(&fx.bars[i], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (R <= 0) return;

    // Requests for tile q (block q / NKT, K tile q % NKT) into stage s, by
    // warp 0.  The weight half only raises the expected bytes; the input half
    // arrives, so a stage cannot complete before both halves are requested.
    // The weights do not depend on the previous kernel and are requested
    // before waiting on it.
    auto issue_weights = [&](int q, int s) {
        if (lane == 0) {
            float *W = region + (size_t)s * stage_floats;
            const int blk = q / NKT, kt = q - blk * NKT;
            mbar_expect_tx(&fx.bars[s], (uint32_t)(SR * tk * 4));
            for (int pc = 0; pc < npc; ++pc)
                tensor_g2s(W + (size_t)pc * RB * tk, &bp.wmap[MODE == GEMV_QKV ? m : pc], kt * tk, wrow0 + blk * RB,
                           &fx.bars[s]);
        }
    };
    auto issue_inputs = [&](int q, int s) {
        float *X = region + (size_t)s * stage_floats + (size_t)SR * tk;
        const int kt = q % NKT, k0 = kt * tk, len = min(tk, n - k0);
        if (emb_rows) {
            // one embedding row per sequence; columns past n stay unused
            if (lane == 0) mbar_arrive_expect_tx(&fx.bars[s], (uint32_t)(B * len * 4));
            __syncwarp();
            for (int b = lane; b < B; b += 32) {
                // a row outside the table (bounds-checked build) is read from row 0 instead
                const size_t row = in_bounds((size_t)p.step->token[b] * p.dim + k0, (size_t)len, p.ext->emb, p.err)
                                       ? (size_t)p.step->token[b] * p.dim : 0;
                bulk_g2s_nohint(X + (size_t)b * tk, p.emb + row + k0, (uint32_t)len * 4u, &fx.bars[s]);
            }
        } else if (lane == 0) {
            mbar_arrive_expect_tx(&fx.bars[s], (uint32_t)(B * tk * 4));
            tensor_g2s(X, &bp.xmap, k0, 0, &fx.bars[s]);
        }
    };

    const int pre = min(stages, NQ);
    if (warp == 0)
        for (int q = 0; q < pre; ++q) {
            issue_weights(q, q);
            if (emb_rows) issue_inputs(q, q);  // the embedding table is read-only
        }

    pdl_launch_dependents();
    pdl_wait();

    if (warp == 0 && !emb_rows)
        for (int q = 0; q < pre; ++q) issue_inputs(q, q);

    // RMSNorm: the gain vector into shared memory, 1/rms of each sequence
    if (MODE != GEMV_RESID) {
        for (int i = tid; i < n / 4; i += kBT)
            reinterpret_cast<float4 *>(gain)[i] = __ldg(reinterpret_cast<const float4 *>(p.norm_w) + i);
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
    } else {
        for (int b = tid; b < B; b += kBT) fx.inv[b] = 0.f;  // sum of squares of the CTA's new x rows
    }
    __syncthreads();

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

#pragma unroll 1
    for (int q = 0; q < NQ; ++q) {
        const int s = q % stages;
        const int blk = q / NKT, kt = q - blk * NKT;
        if (!mbar_wait(&fx.bars[s], (uint32_t)(q / stages) & 1u, p.err)) fx.failed = 1;
        const int k0 = kt * tk, len = min(tk, n - k0), len4 = len >> 2;
        const float *W = region + (size_t)s * stage_floats;
        const float *X = W + (size_t)SR * tk;
        if (busy && !fx.failed) {
            const float4 *wr[kTR];
            const float4 *xr[kTB];
#pragma unroll
            for (int i = 0; i < kTR; ++i)
                wr[i] = reinterpret_cast<const float4 *>(W + (size_t)min(rg * kTR + i, SR - 1) * tk);
#pragma unroll
            for (int j = 0; j < kTB; ++j)
                xr[j] = reinterpret_cast<const float4 *>(X + (size_t)min(bg * kTB + j, B - 1) * tk);
            const float4 *g4 = reinterpret_cast<const float4 *>(gain + k0);
#pragma unroll 1
            for (int f = lane; f < len4; f += 32) {
                float4 w4[kTR], x4[kTB];
#pragma unroll
                for (int i = 0; i < kTR; ++i) w4[i] = wr[i][f];
                if (MODE != GEMV_RESID) {
                    const float4 g = g4[f];
#pragma unroll
                    for (int i = 0; i < kTR; ++i) {
                        w4[i].x *= g.x;
                        w4[i].y *= g.y;
                        w4[i].z *= g.z;
                        w4[i].w *= g.w;
                    }
                }
#pragma unroll
                for (int j = 0; j < kTB; ++j) x4[j] = xr[j][f];
                // component-major order: 64 independent FMAs per component
#pragma unroll
                for (int i = 0; i < kTR; ++i)
#pragma unroll
                    for (int j = 0; j < kTB; ++j) acc[i][j] = fmaf(w4[i].x, x4[j].x, acc[i][j]);
#pragma unroll
                for (int i = 0; i < kTR; ++i)
#pragma unroll
                    for (int j = 0; j < kTB; ++j) acc[i][j] = fmaf(w4[i].y, x4[j].y, acc[i][j]);
#pragma unroll
                for (int i = 0; i < kTR; ++i)
#pragma unroll
                    for (int j = 0; j < kTB; ++j) acc[i][j] = fmaf(w4[i].z, x4[j].z, acc[i][j]);
#pragma unroll
                for (int i = 0; i < kTR; ++i)
#pragma unroll
                    for (int j = 0; j < kTB; ++j) acc[i][j] = fmaf(w4[i].w, x4[j].w, acc[i][j]);
            }
        }
        __syncthreads();
        if (fx.failed) {
            // Let the copies already requested land (bounded waits) before leaving.
            if (tid == 0)
                for (int j = q + 1; j < NQ && j < q + stages; ++j)
                    (void)mbar_wait(&fx.bars[j % stages], (uint32_t)(j / stages) & 1u, p.err);
            return;
        }
        if (warp == 0 && q + stages < NQ) {
            issue_weights(q + stages, s);
            issue_inputs(q + stages, s);
        }
        if (kt != NKT - 1) continue;

        // ---- end of a row block: reduce over the lanes, then the epilogue ----
        if (busy) {
#pragma unroll
            for (int i = 0; i < kTR; ++i)
#pragma unroll
                for (int j = 0; j < kTB; ++j) {
                    const float v = warp_sum(acc[i][j]);
                    const int r = rg * kTR + i, b = bg * kTB + j;
                    if (lane == 0 && r < SR && b < B) ys[(size_t)r * B + b] = (MODE != GEMV_RESID) ? v * fx.inv[b] : v;
                    acc[i][j] = 0.f;
                }
        }
        __syncthreads();
        const int rb0 = blk * RB;                  // block's first row within the CTA
        const int RR = min(RB, R - rb0);           // rows of this block
        const int rr0 = r0 + rb0;                  // block's first row within matrix m
        if (MODE == GEMV_QKV) {
            const int hs = p.head_size, half = hs >> 1;
            for (int e = tid; e < (RR >> 1) * B; e += kBT) {
                const int pi = e / B, b = e - pi * B;
                const int j = 2 * pi;
                const float y0 = ys[(size_t)j * B + b], y1 = ys[(size_t)(j + 1) * B + b];
                const int pos = p.step->pos[b];
                const float2 *rr = p.rope + (size_t)pos * half;
                const int v = rr0 + j;  // row within matrix m
                if (!in_bounds((size_t)pos * half + half - 1, 1, p.ext->rope, p.err)) continue;
                if (m == 0) {
                    if (!in_bounds((size_t)b * p.dim + v, 2, p.ext->q, p.err)) continue;
                    const float2 cs = rr[(v % hs) >> 1];
                    float *qv = p.q + (size_t)b * p.dim;
                    qv[v] = y0 * cs.x - y1 * cs.y;
                    qv[v + 1] = y0 * cs.y + y1 * cs.x;
                } else {
                    const int g = v / hs, d = v % hs;
                    const size_t idx =
                        ((((size_t)p.step->slot[b] * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + pos) * hs +
                        d;
                    if (!in_bounds(idx, 2, p.ext->cache, p.err)) continue;
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
            for (int e = tid; e < RR * B; e += kBT) {
                const int r = e / B, b = e - r * B;
                if (!in_bounds((size_t)b * hidden + rr0 + r, 1, p.ext->hb, p.err)) continue;
                p.hb[(size_t)b * hidden + rr0 + r] = silu_b(ys[e]) * ys[(size_t)(RB + r) * B + b];
            }
        } else if (MODE == GEMV_RESID) {
            const int dim = p.total_units;
            for (int e = tid; e < RR * B; e += kBT) {
                const int r = e / B, b = e - r * B;
                if (!in_bounds((size_t)b * dim + rr0 + r, 1, p.ext->x, p.err)) continue;
                float *xp = p.x + (size_t)b * dim + rr0 + r;
                const float nv = *xp + ys[e];
                *xp = nv;
                ys[e] = nv;
            }
            __syncthreads();
            for (int b = tid; b < B; b += kBT) {
                float ss = fx.inv[b];
                for (int r = 0; r < RR; ++r) ss = fmaf(ys[(size_t)r * B + b], ys[(size_t)r * B + b], ss);
                fx.inv[b] = ss;
            }
        } else {
            float *user = p.step->logits_out;
            const int V = p.total_units;
            for (int e = tid; e < RR * B; e += kBT) {
                const int r = e / B, b = e - r * B;
                if (!in_bounds((size_t)b * V + rr0 + r, 1, p.ext->logits, p.err)) continue;
                p.logits[(size_t)b * V + rr0 + r] = ys[e];
                if (user) user[(size_t)b * V + rr0 + r] = ys[e];
            }
        }
        __syncthreads();
    }
    if (MODE == GEMV_RESID)
        for (int b = tid; b < B; b += kBT)
            if (in_bounds((size_t)blockIdx.x * B + b, 1, p.ext->ss_part, p.err)) p.ss_part[(size_t)blockIdx.x * B + b] = fx.inv[b];
}

// ---------------------------------------------------------------- host side

int gemv_batched_rows_cap(int batch) { return kTR * (kMaxTiles / ((batch + kTB - 1) / kTB)); }

size_t gemv_batched_smem(int stage_rows, int batch, int n, bool norm, int *stages, int *tk) {
    // The widest K tile (fewer, bigger copies and fewer barriers) that still
    // leaves three ring stages; two stages of 64 columns at the least.
    const size_t head = fixed_b_bytes() + (norm ? (size_t)((n + 31) & ~31) * 4 : 0) +
                        (((size_t)stage_rows * batch + 31) & ~(size_t)31) * 4;
    const size_t limit = 227 * 1024 - head;
    int t = 256;
    while (t > 64 && (3 * (size_t)(stage_rows + batch) * t * 4 > limit || t >= 2 * n)) t >>= 1;
    const size_t stage = (size_t)(stage_rows + batch) * t * 4;
    int st = kMaxStages;
    while (st > 2 && st * stage > limit) --st;
    *stages = st;
    *tk = t;
    return head + st * stage;
}

cudaError_t gemv_batched_init() {
    void *fns[] = {reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_QKV>),
                   reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_RESID>),
                   reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_W13>),
                   reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_CLS>)};
    for (void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemv_batched(int mode, const BatchParams &bp, int grid, size_t smem, cudaStream_t stream, bool pdl) {
    void *fn = nullptr;
    switch (mode) {
        case GEMV_QKV: fn = reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_QKV>); break;
        case GEMV_RESID: fn = reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_RESID>); break;
        case GEMV_W13: fn = reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_W13>); break;
        case GEMV_CLS: fn = reinterpret_cast<void *>(l2dec_matvec_batched_kernel<GEMV_CLS>); break;
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
