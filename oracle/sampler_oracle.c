/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain CPU statement of the token sampler of the llama2.c generation
 * loop, against which the GPU sampler is checked bit for bit.  It shares no
 * code with the CUDA path; both follow the definitions below.
 *
 * Sources:
 *   [RUNC]  "run.c" (play_with_baby_llama2 mirror of llama2.c): argmax()
 *           (the first maximum wins: only a strictly larger value moves it),
 *           sample() (a uniform r and the first index whose running sum of
 *           probabilities exceeds r; the last index as a fallback) and the
 *           main loop (temperature 0 -> argmax of the logits, otherwise
 *           logits / temperature, softmax, sample).
 *   [WALK]  "run.c 逐行解讀" §6 Sampler: random_u32() (xorshift*: a 64-bit
 *           state shifted right 12, left 25, right 27 with xor, the state
 *           times 0x2545F4914F6CDD1D, top 32 bits) and sample() (temperature
 *           0 -> argmax; otherwise divide, softmax, one coin per call, and
 *           with 0 < topp < 1 sampling from the smallest set of most
 *           probable tokens whose probability reaches topp).
 *
 * Readings where the pages are silent:
 *   - the coin: the top 24 bits of one random_u32() draw, k / 2^24;
 *   - the softmax is evaluated as e_i = E(l_i / T - max_j l_j / T), with E
 *     the fp32 exponential specified below, and each e_i is then held as
 *     the integer q_i = floor(e_i * 2^48).  Every sum and comparison of the
 *     sampler is exact integer arithmetic on the q_i, so the result does not
 *     depend on the order of any sum; sampling index i with probability
 *     q_i / sum q (tokens whose weight is below 2^-48 of the largest are
 *     never drawn);
 *   - r = floor(k * S / 2^24) for a total S; the sampled index is the first
 *     (in the order of the candidates) whose running total exceeds r;
 *   - top-p: candidates ordered by q descending, ties by index ascending;
 *     the nucleus is the shortest prefix whose total P satisfies
 *     P * 2^24 >= floor(topp * 2^24) * S; r is then drawn against P;
 *   - E(x) for x <= 0: 0 below -87 (no subnormal results); otherwise
 *     k = rint(x * log2 e) (fp32 product, ties to even), the Cody-Waite
 *     reduction r = x - k ln2 with ln 2 split into a nearest-fp32 high part
 *     and an fp32 low part (two fused multiply-adds), a degree-7 Taylor
 *     polynomial of e^r in Horner form with fused multiply-adds, times 2^k.
 *     Constants: log2 e and ln 2 rounded to fp32, the remainder
 *     ln 2 - fp32(ln 2) rounded to fp32, and 1/n! rounded to fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* [WALK] §6 random_u32(): xorshift*. */
uint32_t oracle_random_u32(uint64_t *state) {
    *state ^= *state >> 12;
    *state ^= *state << 25;
    *state ^= *state >> 27;
    return (uint32_t)((*state * 0x2545F4914F6CDD1DULL) >> 32);
}

static float pow2i(int k) { /* 2^k for -126 <= k <= 127 */
    uint32_t bits = (uint32_t)(k + 127) << 23;
    float f;
    memcpy(&f, &bits, 4);
    return f;
}

/* The sampler's exponential (see the header), for x <= 0. */
float oracle_sampler_exp(float x) {
    const float log2e = 1.44269502162933349609375f;        /* fp32(log2 e) */
    const float ln2_hi = 0.693147182464599609375f;         /* fp32(ln 2) */
    const float ln2_lo = -1.9046542121259336e-09f;         /* fp32(ln 2 - ln2_hi) */
    const float c2 = 0.5f, c3 = 0.16666667163372039795f, c4 = 0.041666667908430099487f,
                c5 = 0.0083333337679505348206f, c6 = 0.0013888889225199818611f,
                c7 = 0.00019841270113829523325f;              /* fp32(1/n!) */
    if (!(x > -87.0f)) return 0.0f;
    const float t = x * log2e;
    const float k = rintf(t);
    float r = fmaf(-k, ln2_hi, x);
    r = fmaf(-k, ln2_lo, r);
    float p = c7;
    p = fmaf(p, r, c6);
    p = fmaf(p, r, c5);
    p = fmaf(p, r, c4);
    p = fmaf(p, r, c3);
    p = fmaf(p, r, c2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return p * pow2i((int)k);
}

/* [RUNC] argmax(): the first index of the maximum. */
int oracle_argmax(const float *v, int n) {
    int best = 0;
    for (int i = 1; i < n; i++)
        if (v[i] > v[best]) best = i;
    return best;
}

/* Integer weights q_i of the tempered softmax (see the header). */
static void weights_of(const float *logits, int n, float temperature, uint64_t *q) {
    float m = logits[0] / temperature;
    for (int i = 1; i < n; i++) {
        const float v = logits[i] / temperature;
        if (v > m) m = v;
    }
    for (int i = 0; i < n; i++) {
        const float e = oracle_sampler_exp(logits[i] / temperature - m);
        q[i] = (uint64_t)(e * 281474976710656.0f); /* 2^48, exact scaling; truncation */
    }
}

static uint64_t draw_below(uint32_t k24, uint64_t total) {
    return (uint64_t)(((unsigned __int128)k24 * total) >> 24);
}

typedef struct {
    uint64_t q;
    int idx;
} Cand;

static int by_weight_desc(const void *a, const void *b) {
    const Cand *x = (const Cand *)a, *y = (const Cand *)b;
    if (x->q != y->q) return x->q > y->q ? -1 : 1;
    return x->idx < y->idx ? -1 : (x->idx > y->idx);
}

/*
 * [WALK] §6 sample(): one token from logits[n].  temperature == 0: argmax of
 * the logits, no draw.  Otherwise one draw from *state; topp in (0, 1)
 * restricts the draw to the nucleus.  *total_out, if not NULL, receives the
 * total the coin was scaled by (S, or P with top-p) and *r_out the scaled coin.
 */
int oracle_sample(const float *logits, int n, float temperature, float topp, uint64_t *state, uint64_t *total_out,
                  uint64_t *r_out) {
    if (n <= 0) return -1;
    if (temperature == 0.0f) return oracle_argmax(logits, n);
    uint64_t *q = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)n);
    if (!q) return -1;
    weights_of(logits, n, temperature, q);
    const uint32_t k24 = oracle_random_u32(state) >> 8;
    uint64_t S = 0;
    for (int i = 0; i < n; i++) S += q[i];
    int out = n - 1;
    if (topp <= 0.0f || topp >= 1.0f) {
        const uint64_t r = draw_below(k24, S);
        uint64_t c = 0;
        for (int i = 0; i < n; i++) {
            c += q[i];
            if (r < c) {
                out = i;
                break;
            }
        }
        if (total_out) *total_out = S;
        if (r_out) *r_out = r;
    } else {
        Cand *cand = (Cand *)malloc(sizeof(Cand) * (size_t)n);
        if (!cand) {
            free(q);
            return -1;
        }
        for (int i = 0; i < n; i++) {
            cand[i].q = q[i];
            cand[i].idx = i;
        }
        qsort(cand, (size_t)n, sizeof(Cand), by_weight_desc);
        const uint64_t tp = (uint64_t)(topp * 16777216.0f); /* floor(topp * 2^24) */
        const unsigned __int128 need = (unsigned __int128)tp * S;
        uint64_t P = 0;
        int last = n - 1;
        for (int j = 0; j < n; j++) {
            P += cand[j].q;
            if (((unsigned __int128)P << 24) >= need) {
                last = j;
                break;
            }
        }
        const uint64_t r = draw_below(k24, P);
        uint64_t c = 0;
        out = cand[last].idx;
        for (int j = 0; j <= last; j++) {
            c += cand[j].q;
            if (r < c) {
                out = cand[j].idx;
                break;
            }
        }
        if (total_out) *total_out = P;
        if (r_out) *r_out = r;
        free(cand);
    }
    free(q);
    return out;
}
