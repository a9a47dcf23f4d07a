// Fused matrix-vector kernels for steps of B >= 16 rows (batched decoding or
// prompt chunks) on the tensor cores: Y[b][r] = sum_k W[r][k] v_b[k] with the
// fused epilogues of the other kernels (RoPE + KV write, SwiGLU, residual,
// classifier) and the RMSNorm scale.
//
// Precision.  The data are fp32; tcgen05.mma kind::tf32 reads the top 19
// bits of each operand.  Each product is taken as hi*hi + hi*lo + lo*hi with
// hi the truncated tf32 part and lo = x - hi (the "3xTF32" split of Ootomo
// and Yokota), accumulating in fp32 in tensor memory: the dropped lo*lo term
// and the truncation of lo leave a relative error near 2^-21 per product,
// fp32-level for these sums.  The raw fp32 tile serves as hi (the hardware
// truncates); converter warps write lo beside it.  W*x_hi and W*x_lo are one
// MMA of N = 2*bpad (the input rows followed by their lo rows), so the weight
// tile is read twice per K step (W, W_lo) rather than three times.
//
// Inputs.  The RMSNorm modes read x * gain, written by the previous residual
// kernel (or the embedding kernel) beside x, and scale the outputs by 1/rms
// from the residual kernels' per-tile sums of squares.
//
// Work.  An output tile is 128 weight rows (64 rows of W1 over the same 64
// rows of W3, so SwiGLU pairs stay in one tile) by bpad sequences (B rounded
// up to 16).  Items are (tile, K range); the host splits K so that the items
// fill the SMs; with several ranges the partial tiles go to a workspace and
// the last CTA of the tile (ticket) adds them in range order, so results do
// not depend on timing.  Warp roles, all walking the CTA's items in order:
//   warp 0      2-D tensor copies (TMA, 128-byte swizzle) of the weight and
//               input tiles of 32 K columns into a 4-stage ring;
//   warp 1      the MMAs (M 128, K 8) of each converted stage, committed to
//               the stage's "empty" barrier, and per item to an accumulator
//               barrier; two accumulators in tensor memory alternate;
//   warps 4-7   lo parts of each stage;
//   warps 8-11  epilogue: accumulator -> shared memory -> outputs, while the
//               next item's MMAs run in the other accumulator.
#include <algorithm>

#include <cuda.h>
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kTT = 384;        // threads: 12 warps
constexpr int kTS = 4;          // ring stages
constexpr int kTK = 32;         // K columns per tile (128 bytes)
constexpr int kTM = 128;        // output rows per tile
constexpr int kTN = 64;         // most sequences
constexpr int kConvWarp0 = 4;   // converter warps 4..7
constexpr int kEpiWarp0 = 8;    // epilogue warps 8..11
constexpr int kRoleThreads = 128;
constexpr uint32_t kABytes = kTM * kTK * 4;          // 16 KB
constexpr uint32_t kXBytes = 2 * kTN * kTK * 4;      // inputs and their lo rows, 16 KB
constexpr uint32_t kStageBytes = 2 * kABytes + kXBytes;
constexpr uint32_t kAccCols = 2 * kTN;                // one accumulator: columns [x_hi | x_lo]
constexpr uint32_t kTmemCols = 2 * kAccCols;          // two accumulators
constexpr int kYsStride = kTN + 1;                    // ys row stride bound (bpad + 1)
constexpr int kMaxSplits = 16;                        // K ranges per tile

struct TcFixed {
    uint64_t full[kTS];     // copies landed
    uint64_t conv[kTS];     // lo parts written
    uint64_t empty[kTS];    // MMAs done with the stage
    uint64_t acc_full[2];   // accumulator complete
    uint64_t acc_free[2];   // accumulator read out
    uint64_t fin;
    uint32_t tmem;
    int abort;
    int last;
    float inv[kMaxBatch];
    float red[kRoleThreads];
};

__host__ __device__ constexpr size_t tc_fixed_bytes() { return (sizeof(TcFixed) + 1023) / 1024 * 1024; }
__host__ __device__ constexpr size_t tc_ys_bytes() { return ((size_t)kTM * kYsStride * 4 + 1023) / 1024 * 1024; }

__device__ __forceinline__ float silu_t(float v) { return v / (1.0f + expf(-v)); }
__device__ __forceinline__ float tf32_lo(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }
__device__ __forceinline__ float4 tf32_lo4(float4 v) {
    return make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tensor2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, for an operand whose rows are 128-byte lines.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

// One lane of the (converged) warp; the others skip.  Descriptors built
// outside such a branch stay warp-uniform, which keeps the MMA issue cheap.
__device__ __forceinline__ uint32_t elect_one() {
    uint32_t pred = 0;
    asm volatile("{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\telect.sync rx|px, %1;\n\t@px mov.s32 %0, 1;\n\t}"
                 : "+r"(pred)
                 : "r"(0xffffffffu));
    return pred;
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t addr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(addr));
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The 128 epilogue threads only.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ bool aborted(const TcFixed &fx) { return *reinterpret_cast<const volatile int *>(&fx.abort) != 0; }
__device__ __forceinline__ void set_abort(TcFixed &fx) { *reinterpret_cast<volatile int *>(&fx.abort) = 1; }
// Warp-uniform stop decision: a lane's failed wait or the CTA's abort flag.
__device__ __forceinline__ bool warp_stop(TcFixed &fx, bool ok) {
    if (!ok) set_abort(fx);
    return __any_sync(0xffffffffu, !ok || aborted(fx));
}

}  // namespace

// Layer-0 inputs of a step on the tensor-core path: x[b] = emb[token[b]],
// x[b] * gain for the first RMSNorm, and the sum of squares of each row
// (ss_part row 0, read with ss_parts = 1).
__global__ void tc_embed_kernel(const GemvParams p, float *xg) {
    const int b = blockIdx.x, tid = threadIdx.x;
    __shared__ float red[32];
    pdl_launch_dependents();
    pdl_wait();  // the step's tokens may come from the previous kernel
    const float4 *e4 = reinterpret_cast<const float4 *>(p.emb + (size_t)p.step->token[b] * p.dim);
    const float4 *g4 = reinterpret_cast<const float4 *>(p.norm_w);
    float4 *x4 = reinterpret_cast<float4 *>(p.x + (size_t)b * p.dim);
    float4 *xg4 = reinterpret_cast<float4 *>(xg + (size_t)b * p.dim);
    float ss = 0.f;
    for (int i = tid; i < p.dim / 4; i += blockDim.x) {
        const float4 v = e4[i], g = __ldg(g4 + i);
        x4[i] = v;
        xg4[i] = make_float4(v.x * g.x, v.y * g.y, v.z * g.z, v.w * g.w);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
        p.ss_part[b] = t;
    }
}

template <int MODE>
__global__ void __launch_bounds__(kTT, 1) gemv_tc_kernel(const __grid_constant__ TcParams tp) {
    const GemvParams &p = tp.g;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    TcFixed &fx = *reinterpret_cast<TcFixed *>(smem);
    float *ys = reinterpret_cast<float *>(smem + tc_fixed_bytes());  // [128][bpad + 1]
    unsigned char *ring = smem + tc_fixed_bytes() + tc_ys_bytes();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.batch, BP = tp.bpad, n = p.n;
    const int YS = BP + 1;
    const int KT = (n + kTK - 1) / kTK;
    const int S = tp.splits;
    const int items = tp.ntiles * S;

    if (tid == 0) {
        for (int i = 0; i < kTS; ++i) {
            mbar_init(&fx.full[i], 1);
            mbar_init(&fx.conv[i], kRoleThreads);
            mbar_init(&fx.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&fx.acc_full[i], 1);
            mbar_init(&fx.acc_free[i], kRoleThreads);
        }
        mbar_init(&fx.fin, 1);
        fence_barrier_init();
        fx.abort = 0;
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&fx.tmem)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = fx.tmem;
    pdl_launch_dependents();

    // item -> matrix, first row within it, tensor-map row, K range, tile
    auto item_geom = [&](int it, int &m, int &r0, int &wrow, int &k0t, int &k1t, int &tile) {
        tile = it / S;
        const int sp = it - tile * S;
        m = 0;
        int t = tile;
        if (MODE == GEMV_QKV)
            while (m < 2 && t >= tp.tiles[m]) t -= tp.tiles[m++];
        r0 = t * ((MODE == GEMV_W13) ? kTM / 2 : kTM);
        wrow = (MODE == GEMV_CLS ? 0 : p.layer * tp.mrows[m]) + r0;
        k0t = (int)((long long)sp * KT / S);
        k1t = (int)((long long)(sp + 1) * KT / S);
    };
    auto stage_ptr = [&](int s) { return ring + (size_t)s * kStageBytes; };

    if (warp == 0) {
        // ---------------- producer: tensor copies into the ring (whole warp, one lane issues) ----------------
        const uint32_t stage_tx = kABytes + (uint32_t)BP * kTK * 4;
        long long nl = 0;
        bool stop = false;
        auto issue_weights = [&](int s, int m, int wrow, int kt) {
            unsigned char *st = stage_ptr(s);
            mbar_arrive_expect_tx(&fx.full[s], stage_tx);
            if (MODE == GEMV_W13) {
                tensor2d(st, &tp.wmap[0], kt * kTK, wrow, &fx.full[s]);
                tensor2d(st + kABytes / 2, &tp.wmap[1], kt * kTK, wrow, &fx.full[s]);
            } else {
                tensor2d(st, &tp.wmap[MODE == GEMV_QKV ? m : 0], kt * kTK, wrow, &fx.full[s]);
            }
        };
        // the weights do not depend on the previous kernel: the first stages' tiles go out before the wait
        int npre = 0;
        if ((int)blockIdx.x < items) {
            int m, r0, wrow, k0t, k1t, tile;
            item_geom(blockIdx.x, m, r0, wrow, k0t, k1t, tile);
            npre = min(k1t - k0t, kTS);
            if (elect_one())
                for (int i = 0; i < npre; ++i) issue_weights(i, m, wrow, k0t + i);
            __syncwarp();
        }
        pdl_wait();  // the inputs come from the previous kernel
        for (int it = blockIdx.x; it < items && !stop; it += gridDim.x) {
            int m, r0, wrow, k0t, k1t, tile;
            item_geom(it, m, r0, wrow, k0t, k1t, tile);
            for (int kt = k0t; kt < k1t; ++kt) {
                const int s = (int)(nl % kTS);
                const bool ok = nl < kTS || mbar_wait(&fx.empty[s], (uint32_t)(((nl / kTS) - 1) & 1), p.err);
                if ((stop = warp_stop(fx, ok))) break;
                if (elect_one()) {
                    if (nl >= npre) issue_weights(s, m, wrow, kt);
                    tensor2d(stage_ptr(s) + 2 * kABytes, &tp.xmap, kt * kTK, 0, &fx.full[s]);
                }
                __syncwarp();
                ++nl;
            }
        }
        if (stop)  // the copies still in flight land before the CTA's memory goes
            for (long long j = nl > kTS ? nl - kTS : 0; j < nl; ++j)
                (void)mbar_wait(&fx.full[j % kTS], (uint32_t)((j / kTS) & 1), p.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, one lane issues) ----------------
        const uint32_t idesc2 = idesc_tf32(kTM, 2 * BP), idesc1 = idesc_tf32(kTM, BP);
        const uint64_t dring = desc_sw128(smem_u32(ring));  // stage 0's weight tile
        long long nc = 0, ni = 0;
        bool stop = false;
        for (int it = blockIdx.x; it < items && !stop; it += gridDim.x, ++ni) {
            int m, r0, wrow, k0t, k1t, tile;
            item_geom(it, m, r0, wrow, k0t, k1t, tile);
            const int a = (int)(ni & 1);
            const bool ok = ni < 2 || mbar_wait(&fx.acc_free[a], (uint32_t)(((ni / 2) - 1) & 1), p.err);
            if ((stop = warp_stop(fx, ok))) break;
            tc_fence_after();
            const uint32_t dacc = tmem + (uint32_t)a * kAccCols;
            for (int kt = k0t; kt < k1t; ++kt, ++nc) {
                const int s = (int)(nc % kTS);
                const bool okc = mbar_wait(&fx.conv[s], (uint32_t)((nc / kTS) & 1), p.err);
                if ((stop = warp_stop(fx, okc))) break;
                tc_fence_after();
                // descriptor start addresses are in 16-byte units; a K step of 8 is 32 bytes
                const uint64_t dw = dring + (uint64_t)((uint32_t)s * (kStageBytes >> 4));
                const uint64_t dwl = dw + (kABytes >> 4), dx = dw + ((2 * kABytes) >> 4);
                const uint32_t first = kt == k0t ? 0u : 1u;
                if (elect_one()) {
#pragma unroll
                    for (int ks = 0; ks < kTK / 8; ++ks) {
                        // columns [0, BP): W x_hi; [BP, 2 BP): W x_lo; then W_lo x_hi into [0, BP)
                        mma_tf32(dacc, dw + 2 * ks, dx + 2 * ks, idesc2, ks == 0 ? first : 1u);
                        mma_tf32(dacc, dwl + 2 * ks, dx + 2 * ks, idesc1, 1u);
                    }
                    mma_commit(&fx.empty[s]);
                }
                __syncwarp();
            }
            if (stop) break;
            if (elect_one()) mma_commit(&fx.acc_full[a]);
            __syncwarp();
        }
        // nothing of this CTA's may still run on the tensor core when its memory goes
        if (elect_one()) mma_commit(&fx.fin);
        __syncwarp();
        (void)mbar_wait(&fx.fin, 0u, p.err);
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
        // ---------------- converters: lo parts of weights and inputs ----------------
        const int ct = tid - kConvWarp0 * 32;
        long long nc = 0;
        for (int it = blockIdx.x; it < items && !aborted(fx); it += gridDim.x) {
            int m, r0, wrow, k0t, k1t, tile;
            item_geom(it, m, r0, wrow, k0t, k1t, tile);
            for (int kt = k0t; kt < k1t; ++kt, ++nc) {
                const int s = (int)(nc % kTS);
                if (!mbar_wait(&fx.full[s], (uint32_t)((nc / kTS) & 1), p.err)) set_abort(fx);
                if (aborted(fx)) break;
                float4 *A4 = reinterpret_cast<float4 *>(stage_ptr(s));
                float4 *Alo4 = A4 + kTM * kTK / 4;
                float4 *X4 = Alo4 + kTM * kTK / 4;
                float4 *Xlo4 = X4 + BP * kTK / 4;  // right after the BP input rows
                float4 a[kTM * kTK / 4 / kRoleThreads];
#pragma unroll
                for (int i = 0; i < kTM * kTK / 4 / kRoleThreads; ++i) a[i] = A4[ct + i * kRoleThreads];
#pragma unroll
                for (int i = 0; i < kTM * kTK / 4 / kRoleThreads; ++i) Alo4[ct + i * kRoleThreads] = tf32_lo4(a[i]);
                for (int i = ct; i < BP * kTK / 4; i += kRoleThreads) Xlo4[i] = tf32_lo4(X4[i]);
                fence_proxy_async_smem();
                mbar_arrive(&fx.conv[s]);
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue ----------------
        const int et = tid - kEpiWarp0 * 32, q = warp & 3, row = 32 * q + lane;
        pdl_wait();  // sums of squares, x, the step's positions and slots
        if (MODE != GEMV_RESID) {
            for (int b = et >> 5; b < B; b += kRoleThreads / 32) {
                float ss = 0.f;
                for (int i = lane; i < p.ss_parts; i += 32) ss += __ldcg(p.ss_part + (size_t)i * B + b);
                ss = warp_sum(ss);
                if (lane == 0) fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
            }
        }
        epi_sync();
        long long ni = 0;
        for (int it = blockIdx.x; it < items && !aborted(fx); it += gridDim.x, ++ni) {
            int m, r0, wrow, k0t, k1t, tile;
            item_geom(it, m, r0, wrow, k0t, k1t, tile);
            const int a = (int)(ni & 1);
            if (!mbar_wait(&fx.acc_full[a], (uint32_t)((ni / 2) & 1), p.err)) set_abort(fx);
            if (aborted(fx)) break;
            tc_fence_after();
            // this thread's row of the accumulator: y = W x_hi + W x_lo + W_lo x_hi
            const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)a * kAccCols;
            float *wsrow = (S > 1) ? tp.ws + (size_t)it * kTM * BP : nullptr;  // [BP][128] per item
            for (int c0 = 0; c0 < B; c0 += 8) {
                float v[8], w[8];
                tmem_ld8(base + (uint32_t)c0, v);
                tmem_ld8(base + (uint32_t)(BP + c0), w);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float y = v[j] + w[j];
                    if (S > 1) wsrow[(size_t)(c0 + j) * kTM + row] = y;
                    else ys[row * YS + c0 + j] = y;
                }
            }
            tc_fence_before();
            mbar_arrive(&fx.acc_free[a]);
            if (S > 1) {
                // publish the partial tile; the last CTA of the tile adds all in range order
                __threadfence();
                epi_sync();
                if (et == 0) fx.last = atomicAdd(&tp.tickets[tile], 1u) == (unsigned)(S - 1) ? 1 : 0;
                epi_sync();
                if (!fx.last) continue;
                __threadfence();
                // 4 rows of one sequence per float4; all S partials in flight at once, added in range order
                const float4 *tb = reinterpret_cast<const float4 *>(tp.ws + (size_t)tile * S * kTM * BP);
                for (int v = et; v < B * (kTM / 4); v += kRoleThreads) {
                    float4 part[kMaxSplits];
#pragma unroll
                    for (int sp = 0; sp < kMaxSplits; ++sp)
                        if (sp < S) part[sp] = __ldcg(tb + (size_t)sp * (BP * kTM / 4) + v);
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int sp = 0; sp < kMaxSplits; ++sp)
                        if (sp < S) {
                            y.x += part[sp].x;
                            y.y += part[sp].y;
                            y.z += part[sp].z;
                            y.w += part[sp].w;
                        }
                    const int c = v / (kTM / 4), r = (v - c * (kTM / 4)) * 4;
                    ys[r * YS + c] = y.x;
                    ys[(r + 1) * YS + c] = y.y;
                    ys[(r + 2) * YS + c] = y.z;
                    ys[(r + 3) * YS + c] = y.w;
                }
                if (et == 0) tp.tickets[tile] = 0u;
            }
            epi_sync();

            // ---- rows r0.. of matrix m, sequences 0..B-1 (row index fastest) ----
            if (MODE == GEMV_QKV) {
                const int hs = p.head_size, half = hs >> 1, mr = tp.mrows[m];
                for (int e = et; e < (kTM / 2) * B; e += kRoleThreads) {
                    const int b = e / (kTM / 2), j = 2 * (e - b * (kTM / 2)), v = r0 + j;
                    if (v >= mr) continue;
                    const float y0 = ys[j * YS + b] * fx.inv[b], y1 = ys[(j + 1) * YS + b] * fx.inv[b];
                    const int pos = p.step->pos[b];
                    const float2 *rr = p.rope + (size_t)pos * half;
                    if (m == 0) {
                        const float2 cs = rr[(v % hs) >> 1];
                        float *qv = p.q + (size_t)b * p.dim;
                        qv[v] = y0 * cs.x - y1 * cs.y;
                        qv[v + 1] = y0 * cs.y + y1 * cs.x;
                    } else {
                        const int g = v / hs, d = v % hs;
                        const size_t idx =
                            ((((size_t)p.step->slot[b] * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + pos) *
                                hs +
                            d;
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
                const int hidden = tp.mrows[0];
                for (int e = et; e < (kTM / 2) * B; e += kRoleThreads) {
                    const int b = e / (kTM / 2), j = e - b * (kTM / 2);
                    if (r0 + j >= hidden) continue;
                    const float h1 = ys[j * YS + b] * fx.inv[b], h3 = ys[(j + kTM / 2) * YS + b] * fx.inv[b];
                    p.hb[(size_t)b * hidden + r0 + j] = silu_t(h1) * h3;
                }
            } else if (MODE == GEMV_RESID) {
                const int dim = tp.mrows[0];
                for (int e = et; e < kTM * B; e += kRoleThreads) {
                    const int b = e / kTM, j = e - b * kTM;
                    if (r0 + j >= dim) continue;
                    const size_t o = (size_t)b * dim + r0 + j;
                    const float nv = p.x[o] + ys[j * YS + b];
                    p.x[o] = nv;
                    tp.xg[o] = nv * __ldg(tp.next_gain + r0 + j);
                    ys[j * YS + b] = nv;
                }
                epi_sync();
                // this tile's sum of squares of the new x rows, per sequence, in a fixed order
                const int parts = kRoleThreads / B, rows = min(kTM, dim - r0);
                float ss = 0.f;
                if (et < parts * B) {
                    const int b = et % B;
                    for (int j = et / B; j < rows; j += parts) ss = fmaf(ys[j * YS + b], ys[j * YS + b], ss);
                }
                fx.red[et] = ss;
                epi_sync();
                if (et < B) {
                    float t = 0.f;
                    for (int i = 0; i < parts; ++i) t += fx.red[i * B + et];
                    p.ss_part[(size_t)tile * B + et] = t;
                }
            } else {
                float *user = p.step->logits_out;
                const int V = tp.mrows[0];
                for (int e = et; e < kTM * B; e += kRoleThreads) {
                    const int b = e / kTM, j = e - b * kTM;
                    if (r0 + j >= V) continue;
                    const float y = ys[j * YS + b] * fx.inv[b];
                    p.logits[(size_t)b * V + r0 + j] = y;
                    if (user) user[(size_t)b * V + r0 + j] = y;
                }
            }
            epi_sync();  // ys free for the next item
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

// ---------------------------------------------------------------- host side

int gemv_tc_max_batch() { return kTN; }

size_t gemv_tc_smem() { return 1024 + tc_fixed_bytes() + tc_ys_bytes() + (size_t)kTS * kStageBytes; }

// K ranges per tile: the count that minimises the estimated time in ring
// stages -- waves of items x K tiles per item, where an item of a split tile
// costs at least kSplitItemStages (its partial-tile publish), plus the final
// merge of the last tile's partials.
constexpr int kSplitItemStages = 6;
constexpr int kMergeStages = 6;
int gemv_tc_splits(int ntiles, int n, int ctas) {
    const int KT = (n + kTK - 1) / kTK;
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= kMaxSplits && s <= KT; ++s) {
        const long long waves = ((long long)ntiles * s + ctas - 1) / ctas;
        const long long per = (KT + s - 1) / s;
        const long long cost = s == 1 ? waves * per : waves * std::max<long long>(per, kSplitItemStages) + kMergeStages;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

cudaError_t gemv_tc_init() {
    void *fns[] = {reinterpret_cast<void *>(gemv_tc_kernel<GEMV_QKV>), reinterpret_cast<void *>(gemv_tc_kernel<GEMV_RESID>),
                   reinterpret_cast<void *>(gemv_tc_kernel<GEMV_W13>), reinterpret_cast<void *>(gemv_tc_kernel<GEMV_CLS>)};
    for (void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gemv_tc_smem());
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

static cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                                     cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t launch_tc_embed(const TcParams &tp, int batch, cudaStream_t stream, bool pdl) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(batch), dim3(256), 0, stream, pdl, attr);
    float *xg = tp.xg;
    void *args[] = {const_cast<GemvParams *>(&tp.g), &xg};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(tc_embed_kernel), args);
}

cudaError_t launch_gemv_tc(int mode, const TcParams &tp, int grid, cudaStream_t stream, bool pdl) {
    void *fn = nullptr;
    switch (mode) {
        case GEMV_QKV: fn = reinterpret_cast<void *>(gemv_tc_kernel<GEMV_QKV>); break;
        case GEMV_RESID: fn = reinterpret_cast<void *>(gemv_tc_kernel<GEMV_RESID>); break;
        case GEMV_W13: fn = reinterpret_cast<void *>(gemv_tc_kernel<GEMV_W13>); break;
        case GEMV_CLS: fn = reinterpret_cast<void *>(gemv_tc_kernel<GEMV_CLS>); break;
        default: return cudaErrorInvalidValue;
    }
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kTT), gemv_tc_smem(), stream, pdl, attr);
    void *args[] = {const_cast<TcParams *>(&tp)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace l2
