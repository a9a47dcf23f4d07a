// Fused matrix-vector kernels for steps of B >= 16 rows (batched decoding or
// prompt chunks) on the tensor cores: Y[b][r] = sum_k W[r][k] v_b[k] -- the
// pages' matmul ("run.c", matmul(): W (d,n) @ x (n,) -> (d,)) for B input
// vectors at once -- with the fused epilogues of the other kernels (RoPE +
// KV write, SwiGLU, residual, classifier; the walkthrough §4 forward() steps
// 2a-2h and 3) and the RMSNorm scale.
//
// Precision.  The data are fp32; tcgen05.mma kind::tf32 reads the top 19
// bits of each operand.  Each product is taken as hi*hi + hi*lo + lo*hi (the
// "3xTF32" split of Ootomo and Yokota), accumulating in fp32 in tensor
// memory.  For the weights, hi is the copied tile as the MMA truncates it and
// lo = w - hi (truncated in turn: under 2^-20 relative); for the inputs, hi is
// the tf32 value nearest to x (written back over the input tile) and lo the
// tf32 value nearest to x - hi.  Converter warps write the inputs' lo rows
// beside the inputs in shared memory and the weights' lo parts into tensor
// memory (one row per TMEM lane), where the MMA reads its A operand directly.
// Per K step: one MMA of N = 2*bpad, W * [x_hi; x_lo], and one of N = bpad,
// W_lo * x_hi.  The tensor core's fp32 accumulation loses more than an fp32
// FMA chain as a chain of MMAs into one accumulator grows (measured on GB300:
// attention probabilities 20 layers on were 10x further from the oracle than
// on the CUDA cores with whole K ranges in one accumulator), so the MMAs of at
// most kDrain ring stages share an accumulator and the epilogue warps add the
// groups up in fp32, in K order.
//
// Inputs.  The RMSNorm modes read x * gain, written by the previous residual
// kernel (or the embedding kernel) beside x, and scale the outputs by 1/rms
// from the residual kernels' per-tile sums of squares.
//
// Work.  An output tile is 128 weight rows (64 rows of W1 over the same 64
// rows of W3, so SwiGLU pairs stay in one tile) by bpad sequences (B rounded
// up to 16).  The (tile, K stage) pairs, tile-major, are split evenly over
// the CTAs ("stream-K"): a CTA's range is whole tiles plus at most a partial
// tile at each end.  Whole tiles are finished at once; partial ones go to a
// workspace, and after its last tile -- with no copies of its own in flight,
// when the one release fence it needs no longer waits behind returning data --
// the CTA takes a ticket per partial tile; the last CTA of a tile adds the
// parts in K order, so results do not depend on timing.  Warp roles, all
// walking the CTA's range (its tile segments) in order:
//   warp 0      2-D tensor copies (TMA, 128-byte swizzle) of the weight and
//               input tiles of 64 K columns into a ring of 3 to 5 stages
//               (as many as shared memory holds for the batch width);
//   warp 1      the MMAs (M 128, K 8) of each converted stage, committed to
//               the stage's "empty" barrier, and per segment to an
//               accumulator barrier; two accumulators in TMEM alternate;
//   warps 4-7   lo parts of each stage (weights into the stage's TMEM
//               columns, inputs into shared memory);
//   warps 8-11  epilogue of whole tiles: accumulator -> shared memory ->
//               outputs (partial tiles -> the workspace), while the next
//               segment's MMAs run in the other accumulator;
//   all 12      after the CTA's last tile: tickets, and the K-order merge and
//               epilogue of each partial tile this CTA completes (warps 2-3
//               idle until then).
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kTT = 384;        // threads: 12 warps
constexpr int kMaxStages = 8;   // ring stages (fewer for wide batches)
constexpr int kBK = 32;         // K columns of one tensor-copy box (128 bytes)
constexpr int kSK = 2 * kBK;    // K columns per ring stage: two adjacent boxes
constexpr int kTM = 128;        // output rows per tile
constexpr int kTN = 64;         // most sequences
constexpr int kConvWarp0 = 4;   // converter warps 4..7
constexpr int kEpiWarp0 = 8;    // epilogue warps 8..11
constexpr int kRoleThreads = 128;
constexpr uint32_t kABytes = kTM * kBK * 4;          // 16 KB: one box of weights (128 rows x 32)
constexpr uint32_t kTmemCols = 512;                   // accumulators [0, 2 bpad naccs), W_lo ring above
constexpr int kMaxAccs = 4;                           // accumulators in tensor memory (2..4, as TMEM allows)
// Ring stages the MMAs add into one accumulator before the epilogue takes it and
// adds it to the tile's running sum in fp32: the tensor core's accumulation
// error grows faster than linearly with the length of a chain of MMAs into one
// accumulator, so the chains are kept short.
#ifndef L2_TC_DRAIN
#define L2_TC_DRAIN 4
#endif
constexpr int kDrain = L2_TC_DRAIN;
// RMSNorm modes: from this many sequences on, the partial sums of squares arrive by one
// bulk copy; below it each epilogue warp loads its few sequences' sums directly.
// Partial tiles: the last CTA of a tile fetches the parts by bulk copies (1) or loads (0).
#ifndef L2_TC_MERGE_COPY
#define L2_TC_MERGE_COPY 1
#endif
#ifndef L2_TC_SS_COPY_MIN_ROWS
#define L2_TC_SS_COPY_MIN_ROWS 32
#endif
constexpr size_t kSmemLimit = 227 * 1024;

// A stage covers 64 K columns.  fp32 weights (WT 0): two 32-column halves h,
// weights W_h (16 KB each), then per half the bpad input rows X_h followed by
// their bpad lo rows.  bf16 weights (WT 1): one 16 KB tile of weights (128 rows
// of 64), the two fp32 input boxes X_0, X_1, then the inputs split into three
// bf16 parts (hi, mid, lo), 3 bpad rows of 64 -- the MMA's B operand.  Whole
// stages move with one barrier phase: fewer, larger phases stream from HBM
// markedly faster than twice as many 16 KB ones.
__host__ __device__ constexpr uint32_t xbox_bytes(int bpad) { return (uint32_t)bpad * kBK * 4; }
__host__ __device__ constexpr uint32_t wstage_bytes(int wt) { return wt ? (uint32_t)kTM * kSK * 2 : 2 * kABytes; }
__host__ __device__ constexpr uint32_t xparts_bytes(int bpad) { return 3u * (uint32_t)bpad * kSK * 2; }
__host__ __device__ constexpr uint32_t stage_bytes(int bpad, int wt) {
    return wt ? wstage_bytes(1) + 2 * xbox_bytes(bpad) + xparts_bytes(bpad) : 2 * kABytes + 4 * xbox_bytes(bpad);
}
// accumulator columns: W [x_hi; x_lo] (WT 0) or W [x_hi; x_mid; x_lo] (WT 1)
__host__ __device__ constexpr int acc_cols(int bpad, int wt) { return (wt ? 3 : 2) * bpad; }
// ys: the finished tile [128][bpad + 1] (odd stride: conflict-free columns)
__host__ __device__ constexpr size_t ys_bytes(int bpad) { return (size_t)kTM * (bpad + 1) * 4; }

struct TcFixed {
    uint64_t full[kMaxStages];   // copies landed
    uint64_t conv[kMaxStages];   // lo parts written
    uint64_t empty[kMaxStages];  // MMAs done with the stage
    uint64_t acc_full[kMaxAccs];   // accumulator complete
    uint64_t acc_free[kMaxAccs];   // accumulator read out
    uint64_t fin;
    uint64_t ssbar;  // the partial sums of squares copied into ys (RMSNorm modes)
    uint64_t mrg;    // the parts of a partial tile copied into the ring (its last CTA)
    uint32_t tmem;
    int abort;
    int last_w[2];
    int part_tile[2];     // the CTA's partial tiles (first, last segment), -1 if none
    float inv[kMaxBatch];
    int pos[kMaxBatch];   // the step's positions and cache slots (QKV)
    unsigned char slot[kMaxBatch];
};
// The ring stages start 1024-aligned after this block: keeping it within 1 KB keeps
// a whole ring stage (64 KB at 64 rows) that a second KB of header would cost.
static_assert(sizeof(TcFixed) <= 1024, "the tensor-core GEMV's fixed shared-memory block must fit 1 KB");

__host__ __device__ constexpr size_t tc_fixed_bytes() { return (sizeof(TcFixed) + 1023) / 1024 * 1024; }

// Ring stages for a batch width: what shared memory holds and, with fp32
// weights, the TMEM columns left beside two accumulators (the W_lo ring).
__host__ __device__ constexpr int tc_stages(int bpad, int wt) {
    const int by_smem = (int)((kSmemLimit - 1024 - tc_fixed_bytes() - ys_bytes(bpad)) / stage_bytes(bpad, wt));
    const int by_tmem = wt ? kMaxStages : (int)((kTmemCols - 4u * (uint32_t)bpad) / kSK);
    const int n = by_smem < by_tmem ? by_smem : by_tmem;
    return n < kMaxStages ? n : kMaxStages;
}
// Accumulators: as many as fit beside the W_lo ring (fp32 weights), 2 to 4.
__host__ __device__ constexpr int tc_naccs(int bpad, int stages, int wt) {
    const int n = (int)((kTmemCols - (wt ? 0u : (uint32_t)(kSK * stages))) / (uint32_t)acc_cols(bpad, wt));
    return n < 2 ? 2 : n > kMaxAccs ? kMaxAccs : n;
}

__device__ __forceinline__ float silu_t(float v) { return v / (1.0f + expf(-v)); }
// x = hi + lo with hi the tf32 value nearest to x and lo the tf32 value nearest to
// x - hi (both exact in fp32, so the MMA reads them without further rounding):
// |x - hi - lo| <= 2^-22 |x|.
__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ void tf32_split4(float4 v, float4 &hi, float4 &lo) {
    hi = make_float4(tf32_rna(v.x), tf32_rna(v.y), tf32_rna(v.z), tf32_rna(v.w));
    lo = make_float4(tf32_rna(v.x - hi.x), tf32_rna(v.y - hi.y), tf32_rna(v.z - hi.z), tf32_rna(v.w - hi.w));
}
// The weights' lo part against the tile as copied, whose hi part the MMA takes
// by truncating each operand to tf32: lo = w - trunc(w), itself truncated by the
// MMA, |w - trunc(w) - trunc(lo)| < 2^-20 |w| (rounding the weight tile to
// nearest in place would halve that, but writing 32 KB per stage back into
// shared memory measurably slowed the converter warps).
__device__ __forceinline__ float tf32_lo_trunc(float x) { return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

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

// Instruction descriptor: D fp32, A and B tf32 (kind::tf32) or bf16 (kind::f16),
// both K-major, M x N.
__device__ __forceinline__ uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t da, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(da), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

// x = hi + mid + lo in bf16, each part the bf16 value nearest to what the parts
// before it leave: fp32's 24-bit significand in three 8-bit pieces, so the sum
// is exact for every fp32 that is not far below 2^-100.  Returns the three
// parts' bits.
__device__ __forceinline__ void bf16_split3(float x, uint32_t &h, uint32_t &m, uint32_t &l) {
    const __nv_bfloat16 bh = __float2bfloat16_rn(x);
    const float r1 = x - __bfloat162float(bh);
    const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(bm);
    const __nv_bfloat16 bl = __float2bfloat16_rn(r2);
    h = __bfloat16_as_ushort(bh);
    m = __bfloat16_as_ushort(bm);
    l = __bfloat16_as_ushort(bl);
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

// A operand from tensor memory (one row per lane, K along the columns).
__device__ __forceinline__ void mma_tf32_ta(uint32_t tmem, uint32_t ta, uint64_t db, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
        "r"(ta), "l"(db), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t addr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%"
        "19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

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
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(addr));
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// The 128 epilogue threads only.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Same barrier; every epilogue thread gets the OR of all their flags.
__device__ __forceinline__ bool epi_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Thread-block clusters: this CTA's rank, the address of a shared-memory word
// in another CTA of the cluster, a load through it, and a barrier of every
// thread of the cluster (release / acquire: shared-memory writes before it are
// visible to the other CTAs' reads after it).

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
__global__ void l2dec_tc_embed_kernel(const GemvParams p, float *xg, float *xg_hi, float *xg_lo) {
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
        const float4 xv = make_float4(v.x * g.x, v.y * g.y, v.z * g.z, v.w * g.w);
        xg4[i] = xv;
        if (xg_hi) {
            float4 hi, lo;
            tf32_split4(xv, hi, lo);
            reinterpret_cast<float4 *>(xg_hi + (size_t)b * p.dim)[i] = hi;
            reinterpret_cast<float4 *>(xg_lo + (size_t)b * p.dim)[i] = lo;
        }
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

// WT: 0 fp32 weights (3xTF32 products), 1 bf16 weights (kind::f16, exact products
// of the bf16 weights and the three bf16 parts of each input).
template <int MODE, int WT>
__global__ void __launch_bounds__(kTT, 1) l2dec_matvec_tc_kernel(const __grid_constant__ TcParams tp) {
    const GemvParams &p = tp.g;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    TcFixed &fx = *reinterpret_cast<TcFixed *>(smem);
    const int B = p.batch, BP = tp.bpad, n = p.n;
    const int NS = tp.stages;
    const uint32_t SB = stage_bytes(BP, WT);
    unsigned char *ring = smem + tc_fixed_bytes();  // 1024-aligned stages, then ys
    float *ys = reinterpret_cast<float *>(ring + (size_t)NS * SB);  // [128][bpad + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int YS = BP + 1;
    const int KT = (n + kSK - 1) / kSK;  // ring stages of 64 columns per tile
    // Stream-K: the (tile, stage) pairs in tile-major order, split evenly over the CTAs.
    // Cluster split (CS > 1): CTA rank r of cluster t takes stages [KT r / CS, KT (r + 1) / CS)
    // of tile t (the host keeps CS <= KT).
    const long long T = (long long)tp.ntiles * KT;
    const int G = gridDim.x, CS = tp.csplit;
    const long long s_begin = CS > 1 ? (long long)(blockIdx.x / CS) * KT + (long long)KT * (blockIdx.x % CS) / CS
                                     : (long long)blockIdx.x * T / G;
    const long long s_end = CS > 1 ? (long long)(blockIdx.x / CS) * KT + (long long)KT * (blockIdx.x % CS + 1) / CS
                                   : (long long)(blockIdx.x + 1) * T / G;
    // RMSNorm modes: the residual kernels' partial sums of squares ss_part[parts][B] come
    // in one bulk copy into ys, which the epilogue needs only from its first drain on.
    // Loaded one sequence per round trip per warp, they queued behind the ring's copies
    // for tens of microseconds at 64 sequences while the accumulators waited to be drained.
    const uint32_t ss_bytes = (uint32_t)(((size_t)p.ss_parts * B * 4 + 15) & ~(size_t)15);
    const bool ss_copy = B >= L2_TC_SS_COPY_MIN_ROWS && MODE != GEMV_RESID && ss_bytes <= (uint32_t)ys_bytes(BP) && (size_t)p.ss_parts * B + 3 <= (size_t)kMaxParts * B;
    // the CTA holding stage x of the sequence
    auto cta_of = [&](long long x) { return (int)(((x + 1) * G + T - 1) / T - 1); };
    // the next segment (one tile's part of the CTA's range) at sequence position sq
    auto segment = [&](long long sq, int &tile, int &k0, int &k1) {
        tile = (int)(sq / KT);
        k0 = (int)(sq - (long long)tile * KT);
        k1 = (int)min((long long)KT, k0 + (s_end - sq));
    };
    // tile -> matrix, its first row within it, its tensor-map row
    auto tile_geom = [&](int tile, int &m, int &r0, int &wrow) {
        m = 0;
        int t = tile;
        if (MODE == GEMV_QKV)
            while (m < 2 && t >= tp.tiles[m]) t -= tp.tiles[m++];
        r0 = t * ((MODE == GEMV_W13) ? kTM / 2 : kTM);
        wrow = (MODE == GEMV_CLS ? 0 : p.layer * tp.mrows[m]) + r0;
    };

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&fx.full[i], 1);
            mbar_init(&fx.conv[i], kRoleThreads);
            mbar_init(&fx.empty[i], 1);
        }
        for (int i = 0; i < kMaxAccs; ++i) {
            mbar_init(&fx.acc_full[i], 1);
            mbar_init(&fx.acc_free[i], kRoleThreads);
        }
        mbar_init(&fx.fin, 1);
        mbar_init(&fx.ssbar, 1);
        mbar_init(&fx.mrg, 1);
        fence_barrier_init();
        fx.abort = 0;
        fx.part_tile[0] = fx.part_tile[1] = -1;
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

    auto stage_ptr = [&](int s) { return ring + (size_t)s * SB; };
    // stage s, fp32 weights: W_0 | W_1 | X_0 | X_0 lo | X_1 | X_1 lo;
    //          bf16 weights: W | X_0 | X_1 | X parts (hi, mid, lo rows)
    auto wbox = [&](int s, int h) { return stage_ptr(s) + h * kABytes; };
    auto xbox = [&](int s, int h) {
        return WT ? stage_ptr(s) + wstage_bytes(1) + h * xbox_bytes(BP) : stage_ptr(s) + 2 * kABytes + 2 * h * xbox_bytes(BP);
    };
    auto xparts = [&](int s) { return stage_ptr(s) + wstage_bytes(1) + 2 * xbox_bytes(BP); };
    // TMEM: accumulator a at columns [AC a, AC (a + 1)); with fp32 weights stage s's W_lo
    // at AC NA + 64 s
    const int AC = acc_cols(BP, WT), NA = tc_naccs(BP, NS, WT);
    auto wlo_col = [&](int s) { return (uint32_t)(AC * NA + kSK * s); };

    // A finished tile in src ([128][bpad + 1]) -> the outputs of its rows jlo..jhi-1
    // (for W1/W3: the SwiGLU pairs jlo..jhi-1 of rows j and j + 64; for QKV jlo and
    // jhi are even, keeping RoPE pairs together), sequences 0..B-1.  The residual
    // mode writes its rows' sums of squares to ss_part row `part`.
    auto finish = [&](int tile, int ti, int nt, auto sync, float *src, int jlo, int jhi, int part) {
        int m, r0, wrow;
        tile_geom(tile, m, r0, wrow);
        const int nj = jhi - jlo;
        if (MODE == GEMV_QKV) {
            // pairs (j, j+1) of rows: RoPE on q and k, then the KV cache; the table reads of
            // 8 pairs go out before their stores
            const int hs = p.head_size, half = hs >> 1, mr = tp.mrows[m], npr = nj >> 1;
            for (int e0 = ti; e0 < npr * B; e0 += 8 * nt) {
                float2 cs[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = e0 + i * nt, b = e / npr, v = r0 + jlo + 2 * (e - b * npr);
                    cs[i] = make_float2(1.f, 0.f);
                    if (m < 2 && e < npr * B && v < mr &&
                        in_bounds((size_t)fx.pos[b] * half + ((v % hs) >> 1), 1, p.ext->rope, p.err))
                        cs[i] = p.rope[(size_t)fx.pos[b] * half + ((v % hs) >> 1)];
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int e = e0 + i * nt, b = e / npr, j = jlo + 2 * (e - b * npr), v = r0 + j;
                    if (e >= npr * B || v >= mr) continue;
                    const float y0 = src[j * YS + b] * fx.inv[b], y1 = src[(j + 1) * YS + b] * fx.inv[b];
                    if (m == 0) {
                        if (!in_bounds((size_t)b * p.dim + v, 2, p.ext->q, p.err)) continue;
                        float *qv = p.q + (size_t)b * p.dim;
                        qv[v] = y0 * cs[i].x - y1 * cs[i].y;
                        qv[v + 1] = y0 * cs[i].y + y1 * cs[i].x;
                    } else {
                        const int g = v / hs, d = v % hs;
                        const size_t idx =
                            ((((size_t)fx.slot[b] * p.n_layers + p.layer) * p.n_kv_heads + g) * p.seq_len + fx.pos[b]) * hs +
                            d;
                        if (!in_bounds(idx, 2, p.ext->cache, p.err)) continue;
                        if (m == 1) {
                            p.kcache[idx] = y0 * cs[i].x - y1 * cs[i].y;
                            p.kcache[idx + 1] = y0 * cs[i].y + y1 * cs[i].x;
                        } else {
                            p.vcache[idx] = y0;
                            p.vcache[idx + 1] = y1;
                        }
                    }
                }
            }
        } else if (MODE == GEMV_W13) {
            const int hidden = tp.mrows[0];
            for (int e = ti; e < nj * B; e += nt) {
                const int b = e / nj, j = jlo + (e - b * nj);
                if (r0 + j >= hidden || !in_bounds((size_t)b * hidden + r0 + j, 1, p.ext->hb, p.err)) continue;
                const float h1 = src[j * YS + b] * fx.inv[b], h3 = src[(j + kTM / 2) * YS + b] * fx.inv[b];
                const float hv = silu_t(h1) * h3;
                p.hb[(size_t)b * hidden + r0 + j] = hv;
                if (tp.hb_hi) {
                    const float hi = tf32_rna(hv);
                    tp.hb_hi[(size_t)b * hidden + r0 + j] = hi;
                    tp.hb_lo[(size_t)b * hidden + r0 + j] = tf32_rna(hv - hi);
                }
            }
        } else if (MODE == GEMV_RESID) {
            const int dim = tp.mrows[0];
            const int jend = min(jhi, dim - r0);
            // item = a row and a group of 8 sequences; x of the 8 loaded before any store
            const int ng = (B + 7) / 8;
            for (int e = ti; e < nj * ng; e += nt) {
                const int j = jlo + e % nj, b0 = 8 * (e / nj);
                if (j >= jend || !in_bounds((size_t)(B - 1) * dim + r0 + j, 1, p.ext->x, p.err) ||
                    !in_bounds((size_t)(B - 1) * dim + r0 + j, 1, p.ext->xg, p.err))
                    continue;
                const float g = __ldg(tp.next_gain + r0 + j);
                float xv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (b0 + i < B) xv[i] = p.x[(size_t)(b0 + i) * dim + r0 + j];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (b0 + i < B) {
                        const size_t o = (size_t)(b0 + i) * dim + r0 + j;
                        const float nv = xv[i] + src[j * YS + b0 + i];
                        p.x[o] = nv;
                        tp.xg[o] = nv * g;
                        if (tp.xg_hi) {
                            const float hi = tf32_rna(nv * g);
                            tp.xg_hi[o] = hi;
                            tp.xg_lo[o] = tf32_rna(nv * g - hi);
                        }
                        src[j * YS + b0 + i] = nv;
                    }
            }
            sync();
            // these rows' sum of squares of the new x, per sequence, in a fixed order
            // (128 partials whatever the thread count: the padding column has 128 rows)
            const int parts = kTM / B;
            if (ti < kTM) {
                float ss = 0.f;
                if (ti < parts * B) {
                    const int b = ti % B;
                    for (int jr = jlo + ti / B; jr < jend; jr += parts) ss = fmaf(src[jr * YS + b], src[jr * YS + b], ss);
                }
                src[ti * YS + BP] = ss;
            }
            sync();
            if (ti < B && in_bounds((size_t)part * B + ti, 1, p.ext->ss_part, p.err)) {
                float t = 0.f;
                for (int i = 0; i < parts; ++i) t += src[(i * B + ti) * YS + BP];
                p.ss_part[(size_t)part * B + ti] = t;
            }
        } else {
            float *user = p.step->logits_out;
            const int V = tp.mrows[0];
            for (int e = ti; e < nj * B; e += nt) {
                const int b = e / nj, j = jlo + (e - b * nj);
                if (r0 + j >= V || !in_bounds((size_t)b * V + r0 + j, 1, p.ext->logits, p.err)) continue;
                const float y = src[j * YS + b] * fx.inv[b];
                p.logits[(size_t)b * V + r0 + j] = y;
                if (user) user[(size_t)b * V + r0 + j] = y;
            }
        }
    };
    constexpr int kUnit = MODE == GEMV_W13 ? kTM / 2 : kTM;  // rows (W1/W3: row pairs) of a tile

    if (warp == 0) {
        // ---------------- producer: tensor copies into the ring (whole warp, one lane issues) ----------------
        // the copies of a stage: its weights and the two fp32 input boxes (the lo rows or
        // the bf16 parts are written here)
        const bool xs = !WT && tp.xsplit;  // the inputs' lo rows come by tensor copy too
        const uint32_t stage_tx = wstage_bytes(WT) + (xs ? 4 : 2) * xbox_bytes(BP);
        long long nl = 0;
        bool stop = false;
        auto issue_weights = [&](int s, int m, int wrow, int kt) {
            mbar_arrive_expect_tx(&fx.full[s], stage_tx);
            if (WT) {
                // one box of 64 bf16 columns (128-byte rows): 128 rows, or 64 of W1 over 64 of W3
                const int x = kt * kSK;
                if (MODE == GEMV_W13) {
                    tensor2d(wbox(s, 0), &tp.wmap[0], x, wrow, &fx.full[s]);
                    tensor2d(wbox(s, 0) + wstage_bytes(1) / 2, &tp.wmap[1], x, wrow, &fx.full[s]);
                } else {
                    tensor2d(wbox(s, 0), &tp.wmap[MODE == GEMV_QKV ? m : 0], x, wrow, &fx.full[s]);
                }
                return;
            }
            for (int h = 0; h < 2; ++h) {
                const int x = kt * kSK + h * kBK;
                if (MODE == GEMV_W13) {
                    tensor2d(wbox(s, h), &tp.wmap[0], x, wrow, &fx.full[s]);
                    tensor2d(wbox(s, h) + kABytes / 2, &tp.wmap[1], x, wrow, &fx.full[s]);
                } else {
                    tensor2d(wbox(s, h), &tp.wmap[MODE == GEMV_QKV ? m : 0], x, wrow, &fx.full[s]);
                }
            }
        };
        // the weights do not depend on the previous kernel: the first stages' tiles go out before the wait
        int npre = 0;
        if (s_begin < s_end) {
            int tile, k0, k1, m, r0, wrow;
            segment(s_begin, tile, k0, k1);
            tile_geom(tile, m, r0, wrow);
            npre = min(k1 - k0, NS);
            if (elect_one())
                for (int i = 0; i < npre; ++i) issue_weights(i, m, wrow, k0 + i);
            __syncwarp();
        }
        pdl_wait();  // the inputs come from the previous kernel
        const bool ss_ok = ss_copy && in_bounds(0, ss_bytes / 4, p.ext->ss_part, p.err);
        if (ss_copy && elect_one()) {
            mbar_arrive_expect_tx(&fx.ssbar, ss_ok ? ss_bytes : 0u);
            if (ss_ok) bulk_g2s_nohint(ys, p.ss_part, ss_bytes, &fx.ssbar);
        }
        __syncwarp();
        for (long long sq = s_begin; sq < s_end && !stop;) {
            int tile, k0, k1, m, r0, wrow;
            segment(sq, tile, k0, k1);
            tile_geom(tile, m, r0, wrow);
            sq += k1 - k0;
            for (int kt = k0; kt < k1; ++kt) {
                const int s = (int)(nl % NS);
                const bool ok = nl < NS || mbar_wait(&fx.empty[s], (uint32_t)(((nl / NS) - 1) & 1), p.err);
                if ((stop = warp_stop(fx, ok))) break;
                if (elect_one()) {
                    if (nl >= npre) issue_weights(s, m, wrow, kt);
                    tensor2d(xbox(s, 0), &tp.xmap, kt * kSK, 0, &fx.full[s]);
                    tensor2d(xbox(s, 1), &tp.xmap, kt * kSK + kBK, 0, &fx.full[s]);
                    if (xs) {
                        tensor2d(xbox(s, 0) + xbox_bytes(BP), &tp.xmap_lo, kt * kSK, 0, &fx.full[s]);
                        tensor2d(xbox(s, 1) + xbox_bytes(BP), &tp.xmap_lo, kt * kSK + kBK, 0, &fx.full[s]);
                    }
                }
                __syncwarp();
                ++nl;
            }
        }
        if (stop)  // the copies still in flight land before the CTA's memory goes
            for (long long j = nl > NS ? nl - NS : 0; j < nl; ++j)
                (void)mbar_wait(&fx.full[j % NS], (uint32_t)((j / NS) & 1), p.err);
        if (ss_copy) (void)mbar_wait(&fx.ssbar, 0u, p.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer (whole warp, one lane issues) ----------------
        const uint32_t idesc2 = idesc_tf32(kTM, 2 * BP), idesc1 = idesc_tf32(kTM, BP), idesc3 = idesc_bf16(kTM, 3 * BP);
        const uint64_t dring = desc_sw128(smem_u32(ring));  // stage 0's weight tile
        long long nc = 0, ng = 0;  // stages, accumulator groups
        bool stop = false;
        for (long long sq = s_begin; sq < s_end && !stop;) {
            int tile, k0, k1;
            segment(sq, tile, k0, k1);
            sq += k1 - k0;
            for (int kt = k0; kt < k1; ++kt, ++nc) {
                const int s = (int)(nc % NS);
                // every kDrain stages of a segment start a fresh accumulator (NA of them
                // rotate): the epilogue adds the groups up in fp32, so no MMA accumulation
                // chain is longer than kDrain stages
                const bool g_first = (kt - k0) % kDrain == 0, g_last = (kt - k0) % kDrain == kDrain - 1 || kt == k1 - 1;
                const int a = (int)(ng % NA);
                if (g_first) {
                    const bool okf = ng < NA || mbar_wait(&fx.acc_free[a], (uint32_t)(((ng / NA) - 1) & 1), p.err);
                    if ((stop = warp_stop(fx, okf))) break;
                }
                const bool okc = mbar_wait(&fx.conv[s], (uint32_t)((nc / NS) & 1), p.err);
                if ((stop = warp_stop(fx, okc))) break;
                tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)(AC * a);
                // descriptor start addresses are in 16-byte units; a K step of 8 tf32 or of 16
                // bf16 is 32 bytes
                const uint64_t dw = dring + (uint64_t)((uint32_t)s * (SB >> 4));
                if (WT) {
                    // columns [0, BP): W x_hi; [BP, 2 BP): W x_mid; [2 BP, 3 BP): W x_lo
                    const uint64_t dxp = dw + ((wstage_bytes(1) + 2 * xbox_bytes(BP)) >> 4);
                    if (elect_one()) {
#pragma unroll
                        for (int ks = 0; ks < kSK / 16; ++ks)
                            mma_bf16(dacc, dw + 2 * ks, dxp + 2 * ks, idesc3, (g_first && ks == 0) ? 0u : 1u);
                        mma_commit(&fx.empty[s]);
                        if (g_last) mma_commit(&fx.acc_full[a]);
                    }
                    __syncwarp();
                    if (g_last) ++ng;
                    continue;
                }
                const uint64_t dx = dw + ((2 * kABytes) >> 4), dxh = (2 * xbox_bytes(BP)) >> 4;
                const uint32_t twl = tmem + wlo_col(s);
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int ks = 0; ks < kBK / 8; ++ks) {
                            // columns [0, BP): W x_hi; [BP, 2 BP): W x_lo; then W_lo x_hi into [0, BP)
                            const uint64_t a = dw + h * (kABytes >> 4) + 2 * ks, b = dx + h * dxh + 2 * ks;
                            mma_tf32(dacc, a, b, idesc2, (g_first && h == 0 && ks == 0) ? 0u : 1u);
                            mma_tf32_ta(dacc, twl + (uint32_t)(kBK * h + 8 * ks), b, idesc1, 1u);
                        }
                    mma_commit(&fx.empty[s]);
                    if (g_last) mma_commit(&fx.acc_full[a]);
                }
                __syncwarp();
                if (g_last) ++ng;
            }
        }
        // nothing of this CTA's may still run on the tensor core when its memory goes
        if (elect_one()) mma_commit(&fx.fin);
        __syncwarp();
        (void)mbar_wait(&fx.fin, 0u, p.err);
    } else if (warp >= kConvWarp0 && warp < kConvWarp0 + 4) {
        // ---------------- converters: lo parts of weights (-> TMEM) and inputs ----------------
        const int ct = tid - kConvWarp0 * 32;
        const int q = warp & 3, row = 32 * q + lane;  // this thread's weight row = its TMEM lane
        long long nc = 0;
        bool stop = false;
        for (long long sq = s_begin; sq < s_end && !stop;) {
            int tile, k0, k1;
            segment(sq, tile, k0, k1);
            sq += k1 - k0;
            for (int kt = k0; kt < k1; ++kt, ++nc) {
                const int s = (int)(nc % NS);
                if ((stop = warp_stop(fx, mbar_wait(&fx.full[s], (uint32_t)((nc / NS) & 1), p.err)))) break;
                if (WT) {
                    // bf16 weights: the inputs' three bf16 parts, rows [part][bpad] of 64 columns in
                    // the 128-byte swizzled layout of the fp32 boxes (16-byte chunk g of row r at
                    // g ^ (r % 8); bpad is a multiple of 16, so row part * bpad + r swizzles as r)
                    uint4 *XP = reinterpret_cast<uint4 *>(xparts(s));
                    for (int i = ct; i < BP * 8; i += kRoleThreads) {
                        const int r = i >> 3, g = i & 7;                   // row, group of 8 columns
                        const int j0 = (g & 3) * 2;                         // its first fp32 chunk in box g / 4
                        const float4 *Xr = reinterpret_cast<const float4 *>(xbox(s, g >> 2)) + r * (kBK / 4);
                        const float4 u0 = Xr[j0 ^ (r & 7)], u1 = Xr[(j0 + 1) ^ (r & 7)];
                        const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                        uint32_t ph[4], pm[4], pl[4];
#pragma unroll
                        for (int k2 = 0; k2 < 4; ++k2) {
                            uint32_t h0, m0, l0, h1, m1, l1;
                            bf16_split3(v[2 * k2], h0, m0, l0);
                            bf16_split3(v[2 * k2 + 1], h1, m1, l1);
                            ph[k2] = h0 | (h1 << 16);  // the lower column at the lower address
                            pm[k2] = m0 | (m1 << 16);
                            pl[k2] = l0 | (l1 << 16);
                        }
                        const int pc = g ^ (r & 7);
                        XP[(size_t)r * 8 + pc] = make_uint4(ph[0], ph[1], ph[2], ph[3]);
                        XP[(size_t)(BP + r) * 8 + pc] = make_uint4(pm[0], pm[1], pm[2], pm[3]);
                        XP[(size_t)(2 * BP + r) * 8 + pc] = make_uint4(pl[0], pl[1], pl[2], pl[3]);
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(&fx.conv[s]);
                    continue;
                }
                tc_fence_after();  // after the MMAs that last read this stage's TMEM columns
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // the row's 8 16-byte chunks of half h, logical chunk j stored at j ^ (row % 8)
                    const float4 *A4 = reinterpret_cast<const float4 *>(wbox(s, h)) + row * (kBK / 4);
                    uint32_t v[kBK];
#pragma unroll
                    for (int j = 0; j < kBK / 4; ++j) {
                        const float4 w4 = A4[j ^ (row & 7)];
                        const float4 a =
                            make_float4(tf32_lo_trunc(w4.x), tf32_lo_trunc(w4.y), tf32_lo_trunc(w4.z), tf32_lo_trunc(w4.w));
                        v[4 * j] = __float_as_uint(a.x);
                        v[4 * j + 1] = __float_as_uint(a.y);
                        v[4 * j + 2] = __float_as_uint(a.z);
                        v[4 * j + 3] = __float_as_uint(a.w);
                    }
                    tmem_st32(tmem + ((uint32_t)(32 * q) << 16) + wlo_col(s) + (uint32_t)(kBK * h), v);
                }
                // (inputs split by the kernel that wrote them arrive split)
                for (int h = 0; h < (tp.xsplit ? 0 : 2); ++h) {
                    float4 *X4 = reinterpret_cast<float4 *>(xbox(s, h));
                    float4 *Xlo4 = X4 + BP * kBK / 4;  // right after the BP input rows
                    for (int i = ct; i < BP * kBK / 4; i += kRoleThreads) {
                        float4 hi, lo;
                        tf32_split4(X4[i], hi, lo);
                        X4[i] = hi;
                        Xlo4[i] = lo;
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(&fx.conv[s]);
            }
        }
    } else if (warp >= kEpiWarp0) {
        // ---------------- epilogue ----------------
        const int et = tid - kEpiWarp0 * 32, q = warp & 3, row = 32 * q + lane;
        pdl_wait();  // sums of squares, x, the step's positions and slots
        if (MODE == GEMV_QKV)
            for (int b = et; b < B; b += kRoleThreads) {
                fx.pos[b] = p.step->pos[b];
                fx.slot[b] = (unsigned char)p.step->slot[b];  // slots < kMaxBatch
            }
        if (ss_copy) {
            // the copy in ys: thread b adds sequence b's parts in order (conflict-free columns)
            if (!mbar_wait(&fx.ssbar, 0u, p.err)) set_abort(fx);
            for (int b = et; b < B; b += kRoleThreads) {
                float ss = 0.f;
                for (int i = 0; i < p.ss_parts; ++i) ss += ys[(size_t)i * B + b];
                fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
            }
        } else if (MODE != GEMV_RESID) {
            for (int b = et >> 5; b < B; b += kRoleThreads / 32) {
                float ss = 0.f;
                for (int i = lane; i < p.ss_parts; i += 32) ss += __ldcg(p.ss_part + (size_t)i * B + b);
                ss = warp_sum(ss);
                if (lane == 0) fx.inv[b] = 1.0f / sqrtf(ss / (float)n + 1e-5f);
            }
        }
        epi_sync();
        // partial segments (at most the first and the last): published now, merged after the last one
        int part0 = -1, part1 = -1;
        long long ng = 0;  // accumulator groups, in the MMA warp's order
        bool stop = false;
        for (long long sq = s_begin; sq < s_end && !stop;) {
            int tile, k0, k1;
            segment(sq, tile, k0, k1);
            const int which = sq == s_begin ? 0 : 1;
            sq += k1 - k0;
            const bool whole = k0 == 0 && k1 == KT;
            // this thread's row of each group's accumulator, y = W x_hi + W x_lo + W_lo x_hi,
            // added up over the segment's groups in ys (fp32, in K order)
            for (int kg = k0; kg < k1; kg += kDrain, ++ng) {
                const int a = (int)(ng % NA);
                const bool ok = mbar_wait(&fx.acc_full[a], (uint32_t)((ng / NA) & 1), p.err);
                if (!ok) set_abort(fx);
                if ((stop = epi_sync_or(!ok || aborted(fx)))) break;  // the same decision in all four warps
                tc_fence_after();
                const uint32_t base = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(AC * a);
                float *yr = ys + row * YS;
                for (int c0 = 0; c0 < B; c0 += 16) {
                    float v[16], w[16], u[16];
                    tmem_ld16(base + (uint32_t)c0, v);
                    tmem_ld16(base + (uint32_t)(BP + c0), w);
                    if (WT) tmem_ld16(base + (uint32_t)(2 * BP + c0), u);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j >= B) break;
                        const float y = WT ? (v[j] + w[j]) + u[j] : v[j] + w[j];
                        yr[c0 + j] = kg == k0 ? y : yr[c0 + j] + y;
                    }
                }
                tc_fence_before();
                mbar_arrive(&fx.acc_free[a]);
            }
            if (stop) break;
            if (!whole) {
                if (CS > 1) continue;  // the CTA's only segment: added up across the cluster below
                // a stream-K partial tile goes to this CTA's workspace slot [BP][128]
                float *wsrow = tp.ws + ((size_t)blockIdx.x * 2 + which) * kTM * BP;
                if (in_bounds(((size_t)blockIdx.x * 2 + which) * kTM * BP, (size_t)kTM * BP, p.ext->tc_ws, p.err))
                    for (int c = 0; c < B; ++c) wsrow[(size_t)c * kTM + row] = ys[row * YS + c];
                if (which == 0) part0 = tile;
                else part1 = tile;
                continue;
            }
            epi_sync();
            finish(tile, et, kRoleThreads, [] { epi_sync(); }, ys, 0, kUnit, tile);
            epi_sync();  // ys free for the next tile
        }
        if (!stop && et == 0) {
            fx.part_tile[0] = part0;
            fx.part_tile[1] = part1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");

    auto bar_all = []() { __syncthreads(); };
    if (CS > 1) {
        // Cluster split: every CTA of the cluster holds its K range's part of tile t in
        // ys.  After a cluster barrier, rank r adds the parts of its rows jlo..jhi-1 in
        // rank order (K order), reading the other CTAs' ys through distributed shared
        // memory, into the ring (free now); a second barrier keeps every ys alive until
        // all of those reads are done; then rank r finishes its rows.  Every CTA reaches
        // both barriers (the waits before them are bounded), aborted or not.
        const int tile = blockIdx.x / CS;
        const uint32_t rk = cluster_rank();
        const int jlo = (int)(((long long)kUnit * rk / CS) & ~1LL);
        const int jhi = rk + 1 == (uint32_t)CS ? kUnit : (int)(((long long)kUnit * (rk + 1) / CS) & ~1LL);
        const bool ab = aborted(fx);
        float *red = reinterpret_cast<float *>(ring);  // [kTM][bpad + 1], as ys
        cluster_sync_all();
        if (!ab) {
            const int half = MODE == GEMV_W13 ? 2 : 1;  // W1/W3: rows j and j + 64
            const int nj = jhi - jlo;
            for (int e = tid; e < nj * half * B; e += kTT) {
                const int b = e % B, jj = e / B;
                const int j = jlo + jj % nj + (jj / nj) * (kTM / 2);
                const int o = j * YS + b;
                float acc = 0.f;
                for (int q = 0; q < CS; ++q) acc += ld_dsmem(dsmem_addr(ys + o, (uint32_t)q));
                red[o] = acc;
            }
        }
        cluster_sync_all();
        if (ab) return;
        pdl_wait();  // the previous kernel's outputs (x, the step's positions) are read below
        finish(tile, tid, kTT, bar_all, red, jlo, jhi, tile * CS + (int)rk);
        return;
    }

    // Partial tiles, by the whole CTA: nothing of this CTA's is in flight any more, so
    // the one release fence it needs does not wait behind returning data.  Publish the
    // partial tiles and take the tickets; the last CTA of a tile adds its parts in K
    // order and finishes it.  (Every thread reads the same shared values after the
    // barrier, so the branches below are uniform.)
    if (aborted(fx) || (fx.part_tile[0] < 0 && fx.part_tile[1] < 0)) return;
    pdl_wait();  // every warp now reads the previous kernel's outputs (x, the RoPE table's step)
    if (tid == 0) {
        __threadfence();
        for (int w = 0; w < 2; ++w) {
            int last = 0;
            const int t = fx.part_tile[w];
            if (t >= 0 && in_bounds((size_t)t, 1, p.ext->tc_tickets, p.err)) {
                const int c0 = cta_of((long long)t * KT), c1 = cta_of((long long)(t + 1) * KT - 1);
                last = atomicAdd(&tp.tickets[t], 1u) == (unsigned)(c1 - c0) ? 1 : 0;
            }
            fx.last_w[w] = last;
        }
        __threadfence();
    }
    __syncthreads();
    int mphase = 0;  // phases of fx.mrg used so far
    for (int w = 0; w < 2; ++w) {
        if (!fx.last_w[w]) continue;
        const int t = fx.part_tile[w];
        const int c0 = cta_of((long long)t * KT), c1 = cta_of((long long)(t + 1) * KT - 1);
        const int nparts = c1 - c0 + 1;
        const uint32_t pbytes = (uint32_t)B * kTM * 4;  // a part: [B][128] floats
        if (L2_TC_MERGE_COPY && (size_t)nparts * pbytes <= (size_t)NS * SB) {
            // Every part with one bulk copy into the ring (free now): one round trip
            // instead of a few rounds of loads per part; added in K order below.
            if (tid == 0) {
                bool okp = true;
                for (int cc = c0; cc <= c1; ++cc) {
                    const int wh = (long long)cc * T / G >= (long long)t * KT ? 0 : 1;
                    okp = okp && in_bounds(((size_t)cc * 2 + wh) * kTM * BP, (size_t)B * kTM, p.ext->tc_ws, p.err);
                }
                fence_proxy_async_all();  // the parts are other CTAs' ordinary stores; the ring was read by this CTA
                mbar_arrive_expect_tx(&fx.mrg, okp ? (uint32_t)nparts * pbytes : 0u);
                if (okp)
                    for (int cc = c0; cc <= c1; ++cc) {
                        const int wh = (long long)cc * T / G >= (long long)t * KT ? 0 : 1;
                        bulk_g2s_nohint(ring + (size_t)(cc - c0) * pbytes, tp.ws + ((size_t)cc * 2 + wh) * kTM * BP, pbytes,
                                        &fx.mrg);
                    }
            }
            const bool okw = mbar_wait(&fx.mrg, (uint32_t)(mphase & 1), p.err);
            ++mphase;
            if (okw) {
                const float4 *P4 = reinterpret_cast<const float4 *>(ring);
                const int nv = B * (kTM / 4);
                for (int v = tid; v < nv; v += kTT) {
                    float4 a = P4[v];
                    for (int k = 1; k < nparts; ++k) {
                        const float4 b = P4[(size_t)k * nv + v];
                        a.x += b.x;
                        a.y += b.y;
                        a.z += b.z;
                        a.w += b.w;
                    }
                    const int c = v / (kTM / 4), r = (v - c * (kTM / 4)) * 4;
                    ys[r * YS + c] = a.x;
                    ys[(r + 1) * YS + c] = a.y;
                    ys[(r + 2) * YS + c] = a.z;
                    ys[(r + 3) * YS + c] = a.w;
                }
            }
        } else {
            // 4 rows of one sequence per float4, this thread's v = tid + 384 i (2 at a time);
            // up to 8 parts' loads in flight per round trip; parts added in K order
            constexpr int kV = 2, kPG = 8;
            const int nv = B * (kTM / 4);
            for (int i0 = 0; tid + kTT * i0 < nv; i0 += kV) {
                float4 acc[kV];
#pragma unroll
                for (int i = 0; i < kV; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int cb = c0; cb <= c1; cb += kPG) {
                    float4 part[kPG][kV];
#pragma unroll
                    for (int u = 0; u < kPG; ++u) {
                        const int cc = min(cb + u, c1);
                        const int wh = (long long)cc * T / G >= (long long)t * KT ? 0 : 1;
                        const bool cc_ok = in_bounds(((size_t)cc * 2 + wh) * kTM * BP, (size_t)kTM * BP, p.ext->tc_ws, p.err);
                        const float4 *src = reinterpret_cast<const float4 *>(tp.ws + (cc_ok ? ((size_t)cc * 2 + wh) * kTM * BP : 0));
#pragma unroll
                        for (int i = 0; i < kV; ++i) {
                            const int v = tid + kTT * (i0 + i);
                            if (v < nv && cb + u <= c1) part[u][i] = __ldcg(src + v);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kPG; ++u)
#pragma unroll
                        for (int i = 0; i < kV; ++i) {
                            const int v = tid + kTT * (i0 + i);
                            if (v < nv && cb + u <= c1) {
                                acc[i].x += part[u][i].x;
                                acc[i].y += part[u][i].y;
                                acc[i].z += part[u][i].z;
                                acc[i].w += part[u][i].w;
                            }
                        }
                }
#pragma unroll
                for (int i = 0; i < kV; ++i) {
                    const int v = tid + kTT * (i0 + i);
                    if (v >= nv) continue;
                    const int c = v / (kTM / 4), r = (v - c * (kTM / 4)) * 4;
                    ys[r * YS + c] = acc[i].x;
                    ys[(r + 1) * YS + c] = acc[i].y;
                    ys[(r + 2) * YS + c] = acc[i].z;
                    ys[(r + 3) * YS + c] = acc[i].w;
                }
            }
        }
        if (tid == 0) tp.tickets[t] = 0u;
        __syncthreads();
        finish(t, tid, kTT, bar_all, ys, 0, kUnit, t);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- host side

int gemv_tc_max_batch() { return kTN; }

int gemv_tc_stages(int bpad, int wt) { return tc_stages(bpad, wt); }

size_t gemv_tc_smem(int bpad, int wt) {
    return 1024 + tc_fixed_bytes() + (size_t)tc_stages(bpad, wt) * stage_bytes(bpad, wt) + ys_bytes(bpad);
}

// CTAs for a plan: one per SM, but each with at least kMinCtaStages ring
// stages of work (fewer, longer ranges: fewer partial tiles to add up).
#ifndef L2_TC_MIN_CTA_STAGES
#define L2_TC_MIN_CTA_STAGES 4
#endif
constexpr int kMinCtaStages = L2_TC_MIN_CTA_STAGES;
int gemv_tc_grid(int ntiles, int n, int ctas) {
    const long long T = (long long)ntiles * ((n + kSK - 1) / kSK);
    return (int)std::max<long long>(1, std::min<long long>(ctas, T / kMinCtaStages));
}

template <int WT>
static void *tc_fn_wt(int mode) {
    switch (mode) {
        case GEMV_QKV: return reinterpret_cast<void *>(l2dec_matvec_tc_kernel<GEMV_QKV, WT>);
        case GEMV_RESID: return reinterpret_cast<void *>(l2dec_matvec_tc_kernel<GEMV_RESID, WT>);
        case GEMV_W13: return reinterpret_cast<void *>(l2dec_matvec_tc_kernel<GEMV_W13, WT>);
        case GEMV_CLS: return reinterpret_cast<void *>(l2dec_matvec_tc_kernel<GEMV_CLS, WT>);
    }
    return nullptr;
}
static void *tc_fn(int mode, int wt) { return wt ? tc_fn_wt<1>(mode) : tc_fn_wt<0>(mode); }

// Cluster split for plans with few tiles (fewer than half the SMs): the largest
// cluster of 2..8 CTAs (at most one per K stage) of which all `ntiles` clusters
// are resident at once on this device (one CTA per SM, so a cluster takes that
// many SMs of one GPC).  0: no cluster size fits, use stream-K.
#ifndef L2_TC_CLUSTER
#define L2_TC_CLUSTER 1
#endif
int gemv_tc_cluster_split(int mode, int wt, int ntiles, int n, int bpad, int num_sms) {
    const int KT = (n + kSK - 1) / kSK;
    if (!L2_TC_CLUSTER || 2 * ntiles > num_sms) return 0;
    void *fn = tc_fn(mode, wt);
    for (int c = std::min(8, KT); c >= 2; --c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(ntiles * c);
        cfg.blockDim = dim3(kTT);
        cfg.dynamicSmemBytes = gemv_tc_smem(bpad, wt);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (clusters >= ntiles) return c;
    }
    return 0;
}

// Workspace floats for a grid: two partial tiles per CTA.
size_t gemv_tc_ws_floats(int grid, int bpad) { return (size_t)grid * 2 * kTM * bpad; }

cudaError_t gemv_tc_init() {
    for (int wt = 0; wt < 2; ++wt)
        for (int mode : {GEMV_QKV, GEMV_RESID, GEMV_W13, GEMV_CLS}) {
            cudaError_t e = cudaFuncSetAttribute(tc_fn(mode, wt), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemLimit);
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
    float *xg = tp.xg, *xg_hi = tp.xg_hi, *xg_lo = tp.xg_lo;
    void *args[] = {const_cast<GemvParams *>(&tp.g), &xg, &xg_hi, &xg_lo};
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<void *>(l2dec_tc_embed_kernel), args);
}

cudaError_t launch_gemv_tc(int mode, const TcParams &tp, int grid, cudaStream_t stream, bool pdl) {
    void *fn = tc_fn(mode, tp.wt);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pdl_config(dim3(grid), dim3(kTT), gemv_tc_smem(tp.bpad, tp.wt), stream, pdl, attr);
    if (tp.csplit > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)tp.csplit;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    void *args[] = {const_cast<TcParams *>(&tp)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace l2
