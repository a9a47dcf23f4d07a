/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, slow, obviously correct CPU statement of the llama2.c single-token
 * decode step forward(token, pos) -> logits.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or constant generator with the CUDA path.
 *
 * Sources (page title, then the function or section followed):
 *   [RUNC]  "run.c" (play_with_baby_llama2 mirror of llama2.c):
 *           rmsnorm(), softmax(), matmul(), transformer().
 *   [WALK]  "run.c 逐行解讀" (line-by-line walkthrough of the later run.c):
 *           §3 malloc_run_state (kv_dim), §4 RMSNorm / Softmax / Matmul,
 *           §4 forward() steps 1, 2a-2h and 3 (GQA, on-the-fly RoPE, KV
 *           written into the cache row, wcls).
 *
 * Readings where the pages leave a step open:
 *   - every stored vector (x, xb, q, k, v, the KV cache, hb, logits) is fp32
 *     as on the pages; dot products, the sum of squares, the softmax sum and
 *     the weighted V sum are accumulated in double and rounded to fp32 once;
 *   - RoPE angles, cos and sin are taken in double (the real-number value of
 *     theta = pos * 10000^(-(i mod hs)/hs)), the rotation in double, the
 *     rotated pair rounded to fp32;
 *   - query head h reads KV head g(h) = floor(h * n_kv_heads / n_heads),
 *     which equals the pages' h / kv_mul whenever n_heads % n_kv_heads == 0
 *     and is the contiguous, nearly equal grouping otherwise;
 *   - rmsnorm eps = 1e-5 inside the square root, scores divided by
 *     sqrt(head_size), pairs (2i, 2i+1) rotated, base 10000;
 *   - weights are row-major [out][in]; the KV cache is [layer][pos][kv_dim].
 */
#include <math.h>
#include <omp.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int dim, hidden_dim, n_layers, n_heads, n_kv_heads, vocab_size, seq_len;
} OracleConfig;

typedef struct {
    const float *token_embedding_table; /* (vocab_size, dim) */
    const float *rms_att_weight;        /* (layer, dim) */
    const float *rms_ffn_weight;        /* (layer, dim) */
    const float *wq;                    /* (layer, dim, dim) */
    const float *wk;                    /* (layer, kv_dim, dim) */
    const float *wv;                    /* (layer, kv_dim, dim) */
    const float *wo;                    /* (layer, dim, dim) */
    const float *w1;                    /* (layer, hidden_dim, dim) */
    const float *w2;                    /* (layer, dim, hidden_dim) */
    const float *w3;                    /* (layer, hidden_dim, dim) */
    const float *rms_final_weight;      /* (dim,) */
    const float *wcls;                  /* (vocab_size, dim) */
} OracleWeights;

/* Threads the parallel loops below run on (no arithmetic). */
int oracle_num_threads(void) { return omp_get_max_threads(); }

/* [RUNC] rmsnorm(): o_j = w_j * (x_j / sqrt(mean(x^2) + 1e-5)). */
void oracle_rmsnorm(float *o, const float *x, const float *weight, int size) {
    double ss = 0.0;
    for (int j = 0; j < size; j++) ss += (double)x[j] * (double)x[j];
    ss = ss / size + 1e-5;
    double inv = 1.0 / sqrt(ss);
    for (int j = 0; j < size; j++) o[j] = (float)((double)weight[j] * (inv * (double)x[j]));
}

/* [RUNC] softmax(): subtract the maximum, exponentiate, divide by the sum. */
void oracle_softmax_d(double *x, int size) {
    double max_val = x[0];
    for (int i = 1; i < size; i++)
        if (x[i] > max_val) max_val = x[i];
    double sum = 0.0;
    for (int i = 0; i < size; i++) {
        x[i] = exp(x[i] - max_val);
        sum += x[i];
    }
    for (int i = 0; i < size; i++) x[i] /= sum;
}

void oracle_softmax(float *x, int size) {
    double *t = (double *)malloc(sizeof(double) * (size_t)size);
    for (int i = 0; i < size; i++) t[i] = x[i];
    oracle_softmax_d(t, size);
    for (int i = 0; i < size; i++) x[i] = (float)t[i];
    free(t);
}

/* [RUNC] matmul(): W (d, n) @ x (n,) -> xout (d,), rows split across threads. */
void oracle_matmul(float *xout, const float *x, const float *w, int n, int d) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < d; i++) {
        const float *row = w + (size_t)i * (size_t)n;
        double val = 0.0;
        for (int j = 0; j < n; j++) val += (double)row[j] * (double)x[j];
        xout[i] = (float)val;
    }
}

/* [WALK] §4 forward() step 2d: rotate the pairs (vec[i], vec[i+1]), i even,
 * i < len, by theta = pos * 10000^(-(i mod head_size)/head_size). */
void oracle_rope(float *vec, int len, int head_size, int pos) {
    for (int i = 0; i < len; i += 2) {
        int head_dim = i % head_size;
        double freq = 1.0 / pow(10000.0, (double)head_dim / (double)head_size);
        double val = (double)pos * freq;
        double fcr = cos(val), fci = sin(val);
        double v0 = vec[i], v1 = vec[i + 1];
        vec[i] = (float)(v0 * fcr - v1 * fci);
        vec[i + 1] = (float)(v0 * fci + v1 * fcr);
    }
}

/* Query head -> KV head: floor(h * n_kv_heads / n_heads). */
int oracle_kv_head(int h, int n_heads, int n_kv_heads) {
    return (int)(((long long)h * (long long)n_kv_heads) / (long long)n_heads);
}

/* [WALK] §4 forward() step 2e, one query head: scores against cache rows
 * t = 0..pos, softmax, weighted sum of V.  q and out hold head_size floats;
 * k_rows / v_rows point at the head's slice of cache row 0, rows `stride`
 * floats apart.  att (nullable) receives the pos+1 probabilities. */
void oracle_attention_head(float *out, const float *q, const float *k_rows, const float *v_rows,
                           int stride, int head_size, int pos, double *att) {
    double *s = att ? att : (double *)malloc(sizeof(double) * (size_t)(pos + 1));
    for (int t = 0; t <= pos; t++) {
        const float *k = k_rows + (size_t)t * (size_t)stride;
        double score = 0.0;
        for (int i = 0; i < head_size; i++) score += (double)q[i] * (double)k[i];
        s[t] = score / sqrt((double)head_size);
    }
    oracle_softmax_d(s, pos + 1);
    for (int i = 0; i < head_size; i++) {
        double val = 0.0;
        for (int t = 0; t <= pos; t++) val += s[t] * (double)v_rows[(size_t)t * (size_t)stride + i];
        out[i] = (float)val;
    }
    if (!att) free(s);
}

/*
 * [WALK] §4 forward(), steps 1-3 (with [RUNC] transformer() filling in what
 * the walkthrough elides).  key_cache / value_cache are (layer, seq_len,
 * kv_dim) and are read for rows 0..pos-1 and written at row pos.
 * att_out (nullable) receives the softmax outputs as (layer, n_heads,
 * seq_len), entries t <= pos.  Returns 0, or -1 on a bad argument.
 */
int oracle_forward(const OracleConfig *p, const OracleWeights *w, float *key_cache,
                   float *value_cache, int token, int pos, float *logits, float *att_out) {
    const int dim = p->dim, hidden_dim = p->hidden_dim;
    if (dim <= 0 || p->n_heads <= 0 || p->n_kv_heads <= 0 || dim % p->n_heads) return -1;
    if (token < 0 || token >= p->vocab_size || pos < 0 || pos >= p->seq_len) return -1;
    const int head_size = dim / p->n_heads;
    const int kv_dim = (dim * p->n_kv_heads) / p->n_heads;
    const size_t seq = (size_t)p->seq_len;

    float *x = (float *)malloc(sizeof(float) * dim);
    float *xb = (float *)malloc(sizeof(float) * dim);
    float *xb2 = (float *)malloc(sizeof(float) * dim);
    float *q = (float *)malloc(sizeof(float) * dim);
    float *hb = (float *)malloc(sizeof(float) * hidden_dim);
    float *hb2 = (float *)malloc(sizeof(float) * hidden_dim);
    double *att = (double *)malloc(sizeof(double) * (size_t)p->n_heads * seq);

    /* step 1: token embedding row */
    memcpy(x, w->token_embedding_table + (size_t)token * dim, sizeof(float) * dim);

    for (int l = 0; l < p->n_layers; l++) {
        /* 2a: attention rmsnorm */
        oracle_rmsnorm(xb, x, w->rms_att_weight + (size_t)l * dim, dim);

        /* 2b: k and v are written straight into the cache row at pos */
        size_t loff = (size_t)l * seq * (size_t)kv_dim;
        float *k = key_cache + loff + (size_t)pos * kv_dim;
        float *v = value_cache + loff + (size_t)pos * kv_dim;

        /* 2c: QKV matmuls */
        oracle_matmul(q, xb, w->wq + (size_t)l * dim * dim, dim, dim);
        oracle_matmul(k, xb, w->wk + (size_t)l * dim * kv_dim, dim, kv_dim);
        oracle_matmul(v, xb, w->wv + (size_t)l * dim * kv_dim, dim, kv_dim);

        /* 2d: RoPE on q over dim and on k over kv_dim */
        oracle_rope(q, dim, head_size, pos);
        oracle_rope(k, kv_dim, head_size, pos);

        /* 2e: attention, one query head at a time */
#pragma omp parallel for schedule(static)
        for (int h = 0; h < p->n_heads; h++) {
            int g = oracle_kv_head(h, p->n_heads, p->n_kv_heads);
            oracle_attention_head(xb + (size_t)h * head_size, q + (size_t)h * head_size,
                                  key_cache + loff + (size_t)g * head_size,
                                  value_cache + loff + (size_t)g * head_size, kv_dim, head_size,
                                  pos, att + (size_t)h * seq);
        }
        if (att_out) {
            for (int h = 0; h < p->n_heads; h++)
                for (int t = 0; t <= pos; t++)
                    att_out[((size_t)l * p->n_heads + h) * seq + t] = (float)att[(size_t)h * seq + t];
        }

        /* 2f: output projection and residual */
        oracle_matmul(xb2, xb, w->wo + (size_t)l * dim * dim, dim, dim);
        for (int i = 0; i < dim; i++) x[i] = (float)((double)x[i] + (double)xb2[i]);

        /* 2g: ffn rmsnorm */
        oracle_rmsnorm(xb, x, w->rms_ffn_weight + (size_t)l * dim, dim);

        /* 2h: SwiGLU: w2(silu(w1 xb) * (w3 xb)), silu(v) = v / (1 + e^-v) */
        oracle_matmul(hb, xb, w->w1 + (size_t)l * dim * hidden_dim, dim, hidden_dim);
        oracle_matmul(hb2, xb, w->w3 + (size_t)l * dim * hidden_dim, dim, hidden_dim);
        for (int i = 0; i < hidden_dim; i++) {
            double val = hb[i];
            val *= 1.0 / (1.0 + exp(-val));
            val *= (double)hb2[i];
            hb[i] = (float)val;
        }
        oracle_matmul(xb, hb, w->w2 + (size_t)l * dim * hidden_dim, hidden_dim, dim);
        for (int i = 0; i < dim; i++) x[i] = (float)((double)x[i] + (double)xb[i]);
    }

    /* step 3: final rmsnorm and classifier */
    oracle_rmsnorm(x, x, w->rms_final_weight, dim);
    oracle_matmul(logits, x, w->wcls, dim, p->vocab_size);

    free(x); free(xb); free(xb2); free(q); free(hb); free(hb2); free(att);
    return 0;
}

/* Runs forward() over tokens[0..n) at positions pos0..pos0+n-1 (teacher
 * forcing), writing logits for every step into logits[n][vocab]. */
int oracle_decode(const OracleConfig *p, const OracleWeights *w, float *key_cache,
                  float *value_cache, const int *tokens, int pos0, int n, float *logits) {
    for (int s = 0; s < n; s++) {
        int rc = oracle_forward(p, w, key_cache, value_cache, tokens[s], pos0 + s,
                                logits + (size_t)s * p->vocab_size, NULL);
        if (rc) return rc;
    }
    return 0;
}
