// Token sampling on the device: the sampler of llama2.c's generation loop.
//
// What it computes ("run.c", argmax(), sample() and the main loop; "run.c
// 逐行解讀" §6 Sampler: random_u32() and sample()), per sequence b of B:
//   temperature == 0: the index of the first maximum of the logits; the
//     generator is not advanced;
//   otherwise: one xorshift* draw from rng_state[b], whose top 24 bits k are
//     the coin; the tempered softmax weights e_i = E(l_i / T - max_j l_j / T)
//     held as the integers q_i = floor(e_i * 2^48); r = floor(k * S / 2^24)
//     for the total S; the sampled index is the first whose running total
//     exceeds r;
//   with 0 < topp < 1 the draw is restricted to the nucleus: the shortest
//     prefix of the weights sorted descending (ties by lower index) whose
//     total P satisfies P * 2^24 >= floor(topp * 2^24) * S, and r is drawn
//     against P, walking the nucleus in that order.
// E is a specified fp32 exponential: k = rint(x log2 e), the Cody-Waite
// reduction r = x - k ln 2 with ln 2 split into fp32(ln 2) and fp32 of the
// remainder, a degree-7 Taylor polynomial in Horner form with fused
// multiply-adds, times 2^k; 0 below -87.  Every fp32 step is an explicitly
// rounded operation, so the weights are the same integers whatever compiler
// or order produced them, and all sums and comparisons are exact integer
// arithmetic: the sampled index does not depend on the order of any sum.
//
// How: one CTA of 1024 threads per sequence.  The tempered exponentials are
// cached in shared memory (vocabularies up to kMaxVocab, one pad word per 32
// against bank conflicts); sums are 64-bit integer CTA reductions.  The
// plain draw finds the crossing with a blocked prefix sum over index order.
// Top-p: no nucleus token weighs less than a proven lower bound; the tokens
// above it are usually few, and then they are sorted (bitonic, in shared
// memory: weight descending, index ascending) and walked with exact prefix
// sums.  When they do not fit the list, the whole CTA instead finds the
// weight v* at which the sorted running total reaches the threshold by a
// bitwise search over weight values (sum of the weights >= a candidate, 49
// rounds), takes as many tokens of weight v* (lowest indices first) as
// needed, and finds the drawn token the same way inside the nucleus.
#include <cuda_runtime.h>

#include "l2_device.cuh"
#include "l2_kernels.h"

namespace l2 {

namespace {

constexpr int kST = 1024;                // threads per sequence
constexpr int kMaxVocab = 48 * 1024;     // exponentials cached in shared memory
typedef unsigned long long u64;
typedef unsigned __int128 u128;

__device__ __forceinline__ float sampler_exp(float x) {
    const float log2e = 1.44269502162933349609375f;   // fp32(log2 e)
    const float ln2_hi = 0.693147182464599609375f;    // fp32(ln 2)
    const float ln2_lo = -1.9046542121259336e-09f;    // fp32(ln 2 - ln2_hi)
    const float c2 = 0.5f, c3 = 0.16666667163372039795f, c4 = 0.041666667908430099487f,
                c5 = 0.0083333337679505348206f, c6 = 0.0013888889225199818611f,
                c7 = 0.00019841270113829523325f;        // fp32(1/n!)
    if (!(x > -87.0f)) return 0.0f;
    const float k = rintf(__fmul_rn(x, log2e));
    float r = __fmaf_rn(-k, ln2_hi, x);
    r = __fmaf_rn(-k, ln2_lo, r);
    float p = c7;
    p = __fmaf_rn(p, r, c6);
    p = __fmaf_rn(p, r, c5);
    p = __fmaf_rn(p, r, c4);
    p = __fmaf_rn(p, r, c3);
    p = __fmaf_rn(p, r, c2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __int_as_float(((int)k + 127) << 23));
}

// floor(e * 2^48) for e = 0 or a normal fp32 value in (0, 1], from the bit
// fields (e = m 2^(E - 150) with the 24-bit significand m), in integer
// instructions only.
__device__ __forceinline__ u64 weight_of(float e) {
    const unsigned bits = __float_as_uint(e);
    const int E = (int)(bits >> 23);
    const u64 m = (u64)((bits & 0x7FFFFFu) | 0x800000u);
    const int sh = E - 102;  // e * 2^48 = m * 2^(E - 102)
    if (E == 0) return 0ull;
    return sh >= 0 ? m << sh : (sh > -24 ? m >> (-sh) : 0ull);
}

// Shared-memory slot of token i: one pad word per 32, so that a warp reading
// either 32 consecutive tokens or each thread's own block of 32 touches 32
// different banks.
__device__ __forceinline__ int slot(int i) { return i + (i >> 5); }

struct SampleScratch {
    u64 part[kST / 32];
    float fpart[kST / 32];
    int ipart[kST / 32];
    u64 bcast[4];
    float fbcast;
    int ibcast;
    unsigned k24;
};

__device__ __forceinline__ u64 warp_sum_u64(u64 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over the CTA (exact); every thread receives it.
__device__ u64 cta_sum(u64 v, SampleScratch &sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum_u64(v);
    __syncthreads();
    if (lane == 0) sc.part[warp] = v;
    __syncthreads();
    if (warp == 0) {
        u64 t = lane < kST / 32 ? sc.part[lane] : 0ull;
        t = warp_sum_u64(t);
        if (lane == 0) sc.bcast[0] = t;
    }
    __syncthreads();
    return sc.bcast[0];
}

__device__ float cta_max(float v, SampleScratch &sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    __syncthreads();
    if (lane == 0) sc.fpart[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < kST / 32 ? sc.fpart[lane] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
        if (lane == 0) sc.fbcast = t;
    }
    __syncthreads();
    return sc.fbcast;
}

// Exclusive prefix sum over the threads in thread order (exact).
__device__ u64 cta_exclusive_scan(u64 v, SampleScratch &sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    u64 incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const u64 n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __syncthreads();
    if (lane == 31) sc.part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        u64 t = lane < kST / 32 ? sc.part[lane] : 0ull;
        u64 ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const u64 n = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += n;
        }
        if (lane < kST / 32) sc.part[lane] = ti - t;  // exclusive warp offsets
    }
    __syncthreads();
    return sc.part[warp] + incl - v;
}

}  // namespace

__global__ void __launch_bounds__(kST, 1) sample_kernel(const SampleParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    SampleScratch &sc = *reinterpret_cast<SampleScratch *>(smem);
    float *ecache = reinterpret_cast<float *>(smem + sizeof(SampleScratch));
    const int b = blockIdx.x, tid = threadIdx.x;
    const int V = p.vocab;
    const float *l = p.logits + (size_t)b * V;

    if (p.temperature == 0.0f) {
        // first maximum: larger value, or equal value at a lower index
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += kST) {
            const float v = l[i];
            if (v > bv || (v == bv && i < bi)) {
                bv = v;
                bi = i;
            }
        }
        const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if (lane == 0) {
            sc.fpart[warp] = bv;
            sc.ipart[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            float v = sc.fpart[0];
            int i = sc.ipart[0];
            for (int w = 1; w < kST / 32; ++w)
                if (sc.fpart[w] > v || (sc.fpart[w] == v && sc.ipart[w] < i)) {
                    v = sc.fpart[w];
                    i = sc.ipart[w];
                }
            // all logits NaN: the pages' loop keeps index 0
            p.out[b] = i == 0x7fffffff ? 0 : i;
        }
        return;
    }

    // ---- tempered softmax weights ----
    const float T = p.temperature;
    float m = -INFINITY;
    for (int i = tid; i < V; i += kST) m = fmaxf(m, __fdiv_rn(l[i], T));
    m = cta_max(m, sc);
    for (int i = tid; i < V; i += kST) ecache[slot(i)] = sampler_exp(__fsub_rn(__fdiv_rn(l[i], T), m));
    if (tid == 0) {
        u64 s = p.rng[b];
        s ^= s >> 12;
        s ^= s << 25;
        s ^= s >> 27;
        const unsigned u = (unsigned)((s * 0x2545F4914F6CDD1DULL) >> 32);
        p.rng[b] = s;
        sc.k24 = u >> 8;
    }
    __syncthreads();
    const u64 k24 = sc.k24;

    // this thread's contiguous block of indices (for order-dependent walks)
    const int chunk = (V + kST - 1) / kST;
    const int i0 = min(V, tid * chunk), i1 = min(V, i0 + chunk);

    u64 s_loc = 0;
    for (int i = i0; i < i1; ++i) s_loc += weight_of(ecache[slot(i)]);
    const u64 S = cta_sum(s_loc, sc);

    const bool nucleus = p.topp > 0.0f && p.topp < 1.0f;
    if (!nucleus) {
        const u64 r = (u64)(((u128)k24 * S) >> 24);
        const u64 base = cta_exclusive_scan(s_loc, sc);
        if (r >= base && r < base + s_loc) {
            u64 c = base;
            for (int i = i0; i < i1; ++i) {
                c += weight_of(ecache[slot(i)]);
                if (r < c) {
                    p.out[b] = i;
                    break;
                }
            }
        }
        return;
    }

    // ---- top-p ----
    const u64 tp = (u64)__float2uint_rz(__fmul_rn(p.topp, 16777216.0f));  // floor(topp * 2^24)
    const u128 need = (u128)tp * S;
    // No token of the nucleus weighs less than cutoff: with P' the total
    // before the nucleus's last token (P' 2^24 < need), the tokens after P'
    // (at most V, each no heavier than that last token v*) carry S - P' >
    // S (2^24 - tp) / 2^24, so v* > S (2^24 - tp) / (2^24 V) >= cutoff.
    // Sums over the tokens with q >= cutoff therefore decide every search
    // below exactly as sums over all tokens would.
    const u64 cutoff = (u64)(((u128)S * (16777216ull - tp)) >> 24) / (u64)V;
    u64 ncand = 0;
    for (int i = i0; i < i1; ++i) ncand += weight_of(ecache[slot(i)]) >= cutoff ? 1 : 0;
    const u64 cbase = cta_exclusive_scan(ncand, sc);
    if (tid == kST - 1) sc.bcast[1] = cbase + ncand;
    __syncthreads();
    const u64 C = sc.bcast[1];

    int Cp = 1;
    while ((u64)Cp < C) Cp <<= 1;
    if (Cp <= p.cand_cap) {
        // Candidates in index order, padded to a power of two with -1, then
        // a bitonic sort into the nucleus order: weight descending, index
        // ascending (the padding last).
        int *cand = reinterpret_cast<int *>(ecache + slot(V) + 1);
        u64 k = cbase;
        for (int i = i0; i < i1; ++i)
            if (weight_of(ecache[slot(i)]) >= cutoff) cand[k++] = i;
        for (int i = (int)C + tid; i < Cp; i += kST) cand[i] = -1;
        __syncthreads();
        auto before = [&](int a, int b) -> bool {
            if (b < 0) return a >= 0;
            if (a < 0) return false;
            const u64 qa = weight_of(ecache[slot(a)]), qb = weight_of(ecache[slot(b)]);
            return qa > qb || (qa == qb && a < b);
        };
        for (int kk = 2; kk <= Cp; kk <<= 1)
            for (int j = kk >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < Cp; i += kST) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const int a = cand[i], b = cand[ixj];
                        if ((i & kk) == 0 ? before(b, a) : before(a, b)) {
                            cand[i] = b;
                            cand[ixj] = a;
                        }
                    }
                }
                __syncthreads();
            }
        // Running totals in that order (exact): the nucleus ends at the first
        // position whose total P has P 2^24 >= need; the drawn token is the
        // first whose total exceeds r = floor(k P / 2^24).
        const int nc = (int)C, per = (nc + kST - 1) / kST;
        const int j0 = min(nc, tid * per), j1 = min(nc, j0 + per);
        u64 loc = 0;
        for (int j = j0; j < j1; ++j) loc += weight_of(ecache[slot(cand[j])]);
        const u64 base = cta_exclusive_scan(loc, sc);
        if (j1 > j0 && ((u128)(base + loc) << 24) >= need && (j0 == 0 || ((u128)base << 24) < need)) {
            u64 run = base;
            for (int j = j0; j < j1; ++j) {
                run += weight_of(ecache[slot(cand[j])]);
                if (((u128)run << 24) >= need) {
                    sc.bcast[2] = run;
                    break;
                }
            }
        }
        __syncthreads();
        const u64 P = sc.bcast[2];
        const u64 r = (u64)(((u128)k24 * P) >> 24);
        if (j1 > j0 && r >= base && r < base + loc) {
            u64 run = base;
            for (int j = j0; j < j1; ++j) {
                run += weight_of(ecache[slot(cand[j])]);
                if (r < run) {
                    p.out[b] = cand[j];
                    break;
                }
            }
        }
        return;
    }

    // many candidates: the same searches over every token, by the whole CTA
    auto G = [&](u64 t) {
        u64 v = 0;
        for (int i = tid; i < V; i += kST) {
            const u64 q = weight_of(ecache[slot(i)]);
            if (q >= t) v += q;
        }
        return cta_sum(v, sc);
    };
    // v*: the largest t with G(t) * 2^24 >= need (a weight value: G only
    // changes at weight values)
    u64 vstar = 0;
    for (int bit = 48; bit >= 0; --bit) {
        const u64 cand = vstar | (1ull << bit);
        if (((u128)G(cand) << 24) >= need) vstar = cand;
    }
    const u64 A = G(vstar + 1);  // weight above v*, all in the nucleus
    // tokens of weight v* taken (lowest indices first): the fewest c >= 1 with
    // (A + c v*) 2^24 >= need
    const u128 D = need - ((u128)A << 24);
    const u64 Dh = (u64)(D >> 24), Dl = (u64)D & 0xFFFFFFull;
    u64 c = Dh / vstar + ((Dh % vstar != 0 || Dl != 0) ? 1 : 0);
    if (c < 1) c = 1;
    const u64 P = A + c * vstar;
    const u64 r = (u64)(((u128)k24 * P) >> 24);
    // w: the largest weight value whose tokens in the nucleus, together with
    // the heavier ones, total more than r
    auto N = [&](u64 t) { return t > vstar ? G(t) : P; };
    u64 w = 0;
    for (int bit = 48; bit >= 0; --bit) {
        const u64 cand = w | (1ull << bit);
        if (N(cand) > r) w = cand;
    }
    const u64 F = N(w + 1);
    const u64 j = (r - F) / w;  // rank (by index) of the drawn token among those of weight w
    u64 cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += weight_of(ecache[slot(i)]) == w ? 1 : 0;
    const u64 before = cta_exclusive_scan(cnt, sc);
    if (j >= before && j < before + cnt) {
        u64 seen = before;
        for (int i = i0; i < i1; ++i) {
            if (weight_of(ecache[slot(i)]) != w) continue;
            if (seen == j) {
                p.out[b] = i;
                break;
            }
            ++seen;
        }
    }
}

// ---------------------------------------------------------------- host side

int sample_max_vocab() { return kMaxVocab; }

// Shared memory: the scratch, the cached exponentials (slots 0..slot(vocab))
// and a candidate list of up to 8192 indices, as room allows.
size_t sample_smem_bytes(int vocab) {
    const size_t base = sizeof(SampleScratch) + ((size_t)vocab + (size_t)vocab / 32 + 2) * sizeof(float);
    const size_t limit = 227 * 1024;
    size_t want = base + 8192 * sizeof(int);
    return want < limit ? want : limit;
}

int sample_cand_cap(int vocab) {
    const size_t base = sizeof(SampleScratch) + ((size_t)vocab + (size_t)vocab / 32 + 2) * sizeof(float);
    return (int)((sample_smem_bytes(vocab) - base) / sizeof(int));
}

cudaError_t sample_init() {
    return cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t launch_sample(const SampleParams &p, int batch, cudaStream_t stream) {
    SampleParams q = p;
    q.cand_cap = sample_cand_cap(p.vocab);
    sample_kernel<<<batch, kST, sample_smem_bytes(p.vocab), stream>>>(q);
    return cudaGetLastError();
}

}  // namespace l2
