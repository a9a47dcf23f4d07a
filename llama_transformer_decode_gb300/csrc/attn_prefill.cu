// Causal attention for a prompt chunk: R rows of one cache slot at the
// consecutive positions p0 .. p0 + R - 1, all written by this step's QKV
// kernel.  Same values as the per-row decode attention (attention.cu) --
// for query head h of row r, softmax over t = 0 .. p0 + r of
// q . K[t, g(h)] / sqrt(head_size), times V[t, g(h)] ("run.c 逐行解讀",
// §4 forward() step 2e; "run.c", transformer(), multihead attention) --
// but a K/V tile is read once for 16 query vectors instead of once per row.
//
// Grid (query blocks, KV heads).  A CTA takes 16 query vectors of KV head g:
// rows r0 .. r0 + 16/GQ - 1, every query head of the group.  It walks the
// positions 0 .. (its last row's position) in tiles of 32: warp 0 copies the
// tile's K and V rows into a 2-stage ring (one 1-D bulk copy per row, K rows
// padded by 16 bytes so the 16-byte reads below are conflict-free).  Scores:
// thread (query q, lane group pj) takes positions pj, pj+8, pj+16, pj+24 of
// the tile over the whole head; the 8 threads of a query keep its online
// softmax (max, sum) with 3-level shuffles; the probabilities go through
// shared memory; PV: the same 8 threads hold head_size/8 output dimensions
// of query q each (16-byte chunk pj + 8i of the head: conflict-free reads).
// Positions after a row's own are masked.  Head sizes 64 and 128; 16
// divisible by the group size.
#include <cuda_runtime.h>
#include <math_constants.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {
constexpr int kPfThreads = 128;  // 4 warps
constexpr int kPfNQ = 16;        // query vectors per CTA
constexpr int kPfTK = 32;        // cache positions per tile

template <int HS>
struct PfLayout {
    static constexpr int KP = HS + 4;  // padded K / q row, floats
    static constexpr size_t bars = 0;
    static constexpr size_t qs = 128;
    static constexpr size_t ks = qs + (size_t)kPfNQ * KP * 4;
    static constexpr size_t vs = ks + (size_t)2 * kPfTK * KP * 4;
    static constexpr size_t ps = vs + (size_t)2 * kPfTK * HS * 4;
    static constexpr size_t bytes = ps + (size_t)kPfNQ * kPfTK * 4;
};
}  // namespace

template <int HS, int GQ>
__global__ void __launch_bounds__(kPfThreads) attn_prefill_kernel(const AttnParams p, int rows) {
    using L = PfLayout<HS>;
    constexpr int KP = L::KP, HS4 = HS / 4, QR = kPfNQ / GQ, DPT = HS / 8;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bars);
    float *qs = reinterpret_cast<float *>(smem + L::qs);
    float *ks = reinterpret_cast<float *>(smem + L::ks);
    float *vs = reinterpret_cast<float *>(smem + L::vs);
    float *ps = reinterpret_cast<float *>(smem + L::ps);
    __shared__ int fail;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = blockIdx.y, r0 = blockIdx.x * QR;
    const int nr = min(QR, rows - r0);
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
        fail = 0;
    }
    pdl_launch_dependents();
    pdl_wait();  // q and the chunk's K/V rows come from the QKV kernel

    const int slot = p.step->slot[r0];
    const int p0 = p.step->pos[r0];
    const int P = p.step->pos[r0 + nr - 1] + 1;  // positions the block reads
    const size_t head_base = (((size_t)slot * p.n_layers + p.layer) * p.n_kv_heads + g) * (size_t)p.seq_len * HS;
    const float *kb = p.kcache + head_base;
    const float *vb = p.vcache + head_base;
    const int h0 = g * GQ;

    // query vector qi: row r0 + qi / GQ, head h0 + qi % GQ (zeros past the chunk)
    for (int i = tid; i < kPfNQ * HS4; i += kPfThreads) {
        const int qi = i / HS4, c4 = i - qi * HS4, r = qi / GQ, j = qi - r * GQ;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nr && in_bounds((size_t)(r0 + r) * p.dim + (size_t)(h0 + j) * HS + 4 * c4, 4, p.ext->q, p.err))
            v = reinterpret_cast<const float4 *>(p.q + (size_t)(r0 + r) * p.dim + (size_t)(h0 + j) * HS)[c4];
        reinterpret_cast<float4 *>(qs + qi * KP)[c4] = v;
    }
    __syncthreads();  // barriers initialised, query vectors in place

    const int ntiles = (P + kPfTK - 1) / kPfTK;
    // warp 0: tile `tile` into ring stage `st`, one copy per K row and per V row
    auto issue = [&](int tile, int st) {
        const int t0 = tile * kPfTK, n = min(kPfTK, P - t0);
        // rows outside the cache (bounds-checked build) are skipped; the barrier expects nothing
        const bool ok = in_bounds(head_base + (size_t)t0 * HS, (size_t)n * HS, p.ext->cache, p.err);
        if (lane == 0) mbar_arrive_expect_tx(&bars[st], ok ? 2u * (uint32_t)n * HS * 4u : 0u);
        __syncwarp();
        if (ok && lane < n) {
            bulk_g2s_nohint(ks + ((size_t)st * kPfTK + lane) * KP, kb + (size_t)(t0 + lane) * HS, HS * 4, &bars[st]);
            bulk_g2s_nohint(vs + ((size_t)st * kPfTK + lane) * HS, vb + (size_t)(t0 + lane) * HS, HS * 4, &bars[st]);
        }
    };
    if (warp == 0) {
        issue(0, 0);
        if (ntiles > 1) issue(1, 1);
    }

    // thread tid serves query q = tid / 8 in both passes: lanes 8(q % 4) .. + 7 of warp q / 4
    const int q = tid >> 3, pj = tid & 7;
    const int qrow = q / GQ;
    const bool q_on = qrow < nr;
    const int qpos = p0 + qrow;  // the row's own position: later ones are masked
    float m = -CUDART_INF_F, l = 0.f;
    float o[DPT];
#pragma unroll
    for (int d = 0; d < DPT; ++d) o[d] = 0.f;

#pragma unroll 1
    for (int tile = 0; tile < ntiles; ++tile) {
        const int st = tile & 1;
        if (!mbar_wait(&bars[st], (uint32_t)((tile >> 1) & 1), p.err)) fail = 1;
        __syncthreads();
        if (fail) break;
        const int t0 = tile * kPfTK, n = min(kPfTK, P - t0);
        const float *kt = ks + (size_t)st * kPfTK * KP;
        const float *vt = vs + (size_t)st * kPfTK * HS;
        // scores of query q at positions t0 + pj + 8u
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 *q4 = reinterpret_cast<const float4 *>(qs + q * KP);
#pragma unroll 8
        for (int c4 = 0; c4 < HS4; ++c4) {
            const float4 qv = q4[c4];
#pragma unroll
            for (int u = 0; u < 4; ++u) s[u] = dot4(qv, reinterpret_cast<const float4 *>(kt + (pj + 8 * u) * KP)[c4], s[u]);
        }
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int tl = pj + 8 * u;
            const bool on = q_on && tl < n && t0 + tl <= qpos;
            s[u] = on ? s[u] * p.scale : -CUDART_INF_F;
            mx = fmaxf(mx, s[u]);
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float mn = fmaxf(m, mx);
        const float corr = mn == -CUDART_INF_F ? 1.f : expf(m - mn);
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float pe = s[u] == -CUDART_INF_F ? 0.f : expf(s[u] - mn);
            ps[q * kPfTK + pj + 8 * u] = pe;
            sum += pe;
        }
#pragma unroll
        for (int off = 4; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        l = l * corr + sum;
        m = mn;
        __syncwarp();
        // PV: 16-byte chunks pj + 8 d4 of query q's head over the tile's positions
#pragma unroll
        for (int d = 0; d < DPT; ++d) o[d] *= corr;
        const float *pq = ps + q * kPfTK;
#pragma unroll 4
        for (int tt = 0; tt < n; ++tt) {
            const float pe = pq[tt];
            const float4 *v4 = reinterpret_cast<const float4 *>(vt + (size_t)tt * HS) + pj;
#pragma unroll
            for (int d4 = 0; d4 < DPT / 4; ++d4) {
                const float4 v = v4[8 * d4];
                o[4 * d4] = fmaf(pe, v.x, o[4 * d4]);
                o[4 * d4 + 1] = fmaf(pe, v.y, o[4 * d4 + 1]);
                o[4 * d4 + 2] = fmaf(pe, v.z, o[4 * d4 + 2]);
                o[4 * d4 + 3] = fmaf(pe, v.w, o[4 * d4 + 3]);
            }
        }
        __syncthreads();  // the stage and the probabilities are free
        if (warp == 0 && tile + 2 < ntiles) {
            if (lane == 0) fence_proxy_async_smem();
            __syncwarp();
            issue(tile + 2, st);
        }
    }
    if (fail) {
        // let the copies in flight land before the CTA's memory goes
        if (tid == 0)
            for (int tile = 0; tile < ntiles && tile < 2; ++tile) (void)mbar_wait(&bars[tile & 1], 0u, p.err);
        return;
    }
    if (q_on) {
        const int j = q - qrow * GQ;
        const float inv = 1.0f / l;
        float4 *out = reinterpret_cast<float4 *>(p.out + (size_t)(r0 + qrow) * p.dim + (size_t)(h0 + j) * HS) + pj;
#pragma unroll
        for (int d4 = 0; d4 < DPT / 4; ++d4)
            if (in_bounds((size_t)(r0 + qrow) * p.dim + (size_t)(h0 + j) * HS + 4 * (pj + 8 * d4), 4, p.ext->xb, p.err))
                out[8 * d4] = make_float4(o[4 * d4] * inv, o[4 * d4 + 1] * inv, o[4 * d4 + 2] * inv, o[4 * d4 + 3] * inv);
    }
}

namespace {
typedef void (*PfFn)(const AttnParams, int);

template <int HS>
PfFn pick_pf1(int gq) {
    switch (gq) {
        case 1: return attn_prefill_kernel<HS, 1>;
        case 2: return attn_prefill_kernel<HS, 2>;
        case 4: return attn_prefill_kernel<HS, 4>;
        case 8: return attn_prefill_kernel<HS, 8>;
        case 16: return attn_prefill_kernel<HS, 16>;
    }
    return nullptr;
}

PfFn pick_pf(int hs, int gq) { return hs == 64 ? pick_pf1<64>(gq) : hs == 128 ? pick_pf1<128>(gq) : nullptr; }

size_t pf_smem(int hs) { return hs == 64 ? PfLayout<64>::bytes : PfLayout<128>::bytes; }
}  // namespace

bool attn_prefill_supported(int head_size, int n_heads, int n_kv_heads) {
    if (n_heads % n_kv_heads) return false;
    const int gq = n_heads / n_kv_heads;
    return pick_pf(head_size, gq) != nullptr;
}

cudaError_t attn_prefill_init() {
    for (int hs : {64, 128})
        for (int gq : {1, 2, 4, 8, 16}) {
            cudaError_t e = cudaFuncSetAttribute(pick_pf(hs, gq), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pf_smem(hs));
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}

cudaError_t launch_attn_prefill(const AttnParams &p, int rows, cudaStream_t stream, bool pdl) {
    const int gq = p.n_heads / p.n_kv_heads;
    PfFn fn = pick_pf(p.head_size, gq);
    if (!fn || rows < 1) return cudaErrorInvalidValue;
    const int qr = kPfNQ / gq;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((rows + qr - 1) / qr, p.n_kv_heads);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = pf_smem(p.head_size);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<AttnParams *>(&p), &rows};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(fn), args);
}

}  // namespace l2
