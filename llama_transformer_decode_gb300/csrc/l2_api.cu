// Host side of the C ABI declared in include/l2.h: argument checks, device
// memory, the per-step orchestration and its CUDA graphs.
//
// One step of batch B is 5 * n_layers + 1 kernel launches (per layer: fused
// rmsnorm+QKV+RoPE+KV write, attention, Wo+residual, rmsnorm+W1/W3+SwiGLU,
// W2+residual; then the final rmsnorm+classifier), linked by programmatic
// dependent launch.  They are captured once per batch size into a CUDA graph
// and replayed.  The step's inputs (tokens, positions, output pointer) are
// not baked into the graph: each call writes them into a pinned ring slot and
// copies them to a device struct that every kernel reads, so one graph serves
// every position.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/l2.h"
#include "l2_device.cuh"
#include "l2_kernels.h"
#include "l2_params.h"

using namespace l2;

namespace {

constexpr int kRing = 64;      // pinned step-input slots in flight
#ifndef L2_ATTN_MIN_CHUNK
#define L2_ATTN_MIN_CHUNK 128
#endif
#ifndef L2_ATTN_MAX_PER_SM
#define L2_ATTN_MAX_PER_SM 4
#endif
// Ring of the persistent step kernel: buffers per warp, and the largest
// buffer in 16-byte words (the host fills the free shared memory up to it).
#ifndef L2_STEP_STAGES
#define L2_STEP_STAGES 3
#endif
#ifndef L2_STEP_MAX_CHUNK_WORDS
#define L2_STEP_MAX_CHUNK_WORDS 512
#endif
// Batched steps and prompt chunks of at least this many rows use the
// tensor-core GEMV (gemv_tc.cu) unless L2_FLAG_NO_TC.
#ifndef L2_TC_MIN_BATCH
#define L2_TC_MIN_BATCH 16
#endif
// Fewest cache positions per attention CTA.  Measured on GB300 (7B shape):
// 128 beats 32 and 64 at positions up to ~2000 (fewer chunks to merge, a
// single CTA per head below 128 positions) and ties above.
constexpr int kMinChunk = L2_ATTN_MIN_CHUNK;

thread_local std::string g_create_error;
int g_fail_alloc_at = 0;  // fault injection: fail the n-th device allocation
int g_fail_graph_at = 0;  // fault injection: fail the n-th graph instantiation

struct BatchPlan {
    BatchParams bp;  // tensor maps, partition, tiles (layer fields filled per launch)
    int grid;
    size_t smem;
};

struct BatchSet {
    bool built = false;
    BatchPlan plan[5];  // QKV, Wo, W1/W3, W2, classifier
    bool tc = false;    // the tensor-core plans below are used
    TcParams tcp[5];
    int tc_grid[5] = {};
    size_t tc_ws_floats = 0;  // split-K workspace the plans need
    int tc_tiles = 0;         // most tiles of a plan (tickets)
};

struct GemvPlan {
    int mode;
    int shape;  // GEMV launch shape (-1: none fits in shared memory)
    int grid;
    size_t smem;
    int units, unit_rows, factor;  // work split: units of unit_rows rows; factor rows per row for W1/W3
    GemvParams base;               // layer-independent fields
};

}  // namespace

struct l2_ctx {
    L2Config cfg{};
    L2Weights w{};
    // L2_FLAG_BF16_WEIGHTS: the matrices as bf16 (the handle's own copies), streamed by the batch-1 kernels
    int wt = 0;
    unsigned short *w16 = nullptr;
    const unsigned short *b16q = nullptr, *b16k = nullptr, *b16v = nullptr, *b16o = nullptr, *b16w1 = nullptr,
                         *b16w2 = nullptr, *b16w3 = nullptr, *b16cls = nullptr;
    int max_batch = 1;  // sequences, each with its own KV-cache slot
    int max_rows = 1;   // rows of a batched step: max_batch, or 64 for prompt chunks
    unsigned flags = 0;
    int device = 0, num_sms = 0;
    int head_size = 0, kv_dim = 0;
    cudaStream_t stream = nullptr, cap_stream = nullptr;
    bool own_stream = false;

    std::vector<void *> dev_allocs;
    float *x = nullptr, *xb = nullptr, *q = nullptr, *hb = nullptr, *logits = nullptr;
    float *kcache = nullptr, *vcache = nullptr, *ws_ml = nullptr, *ws_acc = nullptr, *dbg = nullptr;
    unsigned *tickets = nullptr;
    float2 *rope = nullptr;
    StepDev *step_dev = nullptr;
    int *err = nullptr;
    float *ss_part = nullptr;  // batched steps: partial sums of x^2 [kMaxParts][max_rows]
    float *tc_ws = nullptr;       // tensor-core GEMV split-K partial tiles
    float *xg = nullptr;          // tensor-core path: x * gain of the next RMSNorm [max_rows][dim]
    // tensor-core path with fp32 weights: the inputs' tf32 split (hi, lo) written once by
    // the kernels that produce them (x * gain, and the SwiGLU output for W2)
    float *xg_hi = nullptr, *xg_lo = nullptr, *hb_hi = nullptr, *hb_lo = nullptr;
    unsigned *tc_tickets = nullptr;
    size_t tc_tickets_n = 0;      // entries of tc_tickets
    size_t tc_ws_n = 0;           // floats of tc_ws

    StepDev *step_host = nullptr;  // pinned ring
    cudaEvent_t ring_ev[kRing] = {};
    bool ring_used[kRing] = {};
    int ring_next = 0;

    cudaGraphExec_t graph[kMaxBatch + 1] = {};
    cudaGraphExec_t graph_pf[kMaxBatch + 1] = {};  // prompt chunks (prefill attention)
    bool attn_pf = false;                           // the prefill attention kernel serves this shape

    AttnLaunch attn{};
    int attn_chunks = 1;
    int attn_per_sm = 1;  // attention CTAs resident per SM
    int attn_cluster = 0;  // steps of one row: chunks per KV head merged in a cluster (0: tickets)
    GemvPlan plan_qkv{}, plan_wo{}, plan_w13{}, plan_w2{}, plan_cls{};
    int last_rows = 0;         // rows of the last step submitted (l2_launch_op_batch)
    bool last_prefill = false;  // ... and whether it was a prompt chunk
    bool cta = false;      // batch-1 steps run as the one-block step kernel (small models)
    size_t cta_smem = 0;
    CtaStepParams ctap{};
    bool persist = false;  // batch-1 steps run as the persistent step kernel
    int persist_gq = 1;
    size_t persist_smem = 0;
    StepKParams sp{};
    std::vector<BatchSet> bsets;  // batched GEMV plans, indexed by batch size
    bool evict_first = false;

    float *static_scratch = nullptr;  // device address of the l2_forward_static array on this device
    Extents ext{}, ext_static{};      // buffer sizes for the bounds-checked build, and their device copies
    Extents *ext_dev = nullptr, *ext_static_dev = nullptr;
    std::vector<int> written;  // cache rows written per slot
    std::string error;
};

namespace {

int fail(l2_ctx *c, int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (c)
        c->error = buf;
    else
        g_create_error = buf;
    return code;
}

int cuda_fail(l2_ctx *c, cudaError_t e, const char *what) {
    return fail(c, L2_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

#define L2_CUDA(ctx, call)                                      \
    do {                                                        \
        cudaError_t e_ = (call);                                \
        if (e_ != cudaSuccess) return cuda_fail(ctx, e_, #call); \
    } while (0)

int dev_alloc(l2_ctx *c, void **p, size_t bytes, const char *what) {
    *p = nullptr;
    if (g_fail_alloc_at > 0 && --g_fail_alloc_at == 0)
        return fail(c, L2_ENOMEM, "allocation of %s (%zu bytes) failed (injected)", what, bytes);
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return fail(c, L2_ENOMEM, "cudaMalloc of %s (%zu bytes) failed: %s", what, bytes, cudaGetErrorString(e));
    }
    c->dev_allocs.push_back(*p);
    return L2_OK;
}

template <typename T>
int alloc_n(l2_ctx *c, T **p, size_t n, const char *what) {
    return dev_alloc(c, reinterpret_cast<void **>(p), n * sizeof(T), what);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void free_all(l2_ctx *c) {
    if (c->stream) cudaStreamSynchronize(c->stream);
    for (auto &g : c->graph)
        if (g) {
            cudaGraphExecDestroy(g);
            g = nullptr;
        }
    for (auto &g : c->graph_pf)
        if (g) {
            cudaGraphExecDestroy(g);
            g = nullptr;
        }
    for (auto &e : c->ring_ev)
        if (e) {
            cudaEventDestroy(e);
            e = nullptr;
        }
    for (void *p : c->dev_allocs) cudaFree(p);
    c->dev_allocs.clear();
    if (c->step_host) cudaFreeHost(c->step_host);
    c->step_host = nullptr;
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    c->cap_stream = nullptr;
    if (c->own_stream && c->stream) cudaStreamDestroy(c->stream);
    c->stream = nullptr;
}

int check_config(const L2Config &p) {
    if (p.dim <= 0 || p.hidden_dim <= 0 || p.n_layers <= 0 || p.n_heads <= 0 || p.n_kv_heads <= 0 ||
        p.vocab_size <= 0 || p.seq_len <= 0)
        return fail(nullptr, L2_EINVAL, "every Config field must be positive");
    if (p.dim % p.n_heads) return fail(nullptr, L2_EINVAL, "dim (%d) must be a multiple of n_heads (%d)", p.dim, p.n_heads);
    if (p.n_kv_heads > p.n_heads)
        return fail(nullptr, L2_EINVAL, "n_kv_heads (%d) exceeds n_heads (%d)", p.n_kv_heads, p.n_heads);
    const int hs = p.dim / p.n_heads;
    if (hs % 2) return fail(nullptr, L2_EINVAL, "head_size (%d) must be even for RoPE pairs", hs);
    if ((long long)p.dim * p.n_kv_heads % p.n_heads)
        return fail(nullptr, L2_EINVAL, "dim * n_kv_heads must be a multiple of n_heads");
    if (p.dim % 4 || p.hidden_dim % 4 || hs % 4)
        return fail(nullptr, L2_EINVAL, "this implementation needs dim, hidden_dim and head_size to be multiples of 4");
    if (hs > 128) return fail(nullptr, L2_EINVAL, "this implementation supports head_size <= 128 (got %d)", hs);
    if ((p.n_heads + p.n_kv_heads - 1) / p.n_kv_heads > 8)
        return fail(nullptr, L2_EINVAL, "this implementation supports at most 8 query heads per KV head");
    return L2_OK;
}

int check_weights(const L2Weights &w) {
    const float *ptrs[] = {w.token_embedding_table, w.rms_att_weight, w.rms_ffn_weight, w.wq, w.wk, w.wv,
                           w.wo,                    w.w1,           w.w2,           w.w3, w.rms_final_weight, w.wcls};
    for (const float *p : ptrs) {
        if (!p) return fail(nullptr, L2_EINVAL, "a weight pointer is NULL");
        if (!aligned16(p)) return fail(nullptr, L2_EINVAL, "weight pointers must be 16-byte aligned");
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            return fail(nullptr, L2_EINVAL, "weight pointers must be device memory");
        }
    }
    return L2_OK;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

void make_plans(l2_ctx *c) {
    const L2Config &p = c->cfg;
    const int G = c->num_sms;
    auto plan = [&](GemvPlan &pl, int mode, int n, int unit_rows, int units, int ymax_factor) {
        pl.mode = mode;
        pl.units = units;
        pl.unit_rows = unit_rows;
        pl.factor = ymax_factor;
        pl.grid = units < G ? units : G;
        const int per = ceil_div(units, pl.grid);
        pl.shape = gemv_pick_shape(n, per * unit_rows * ymax_factor, &pl.smem);
        GemvParams &b = pl.base;
        memset(&b, 0, sizeof(b));
        b.n = n;
        b.unit_rows = unit_rows;
        b.total_units = units;
        b.emb = c->w.token_embedding_table;
        b.x = c->x;
        b.q = c->q;
        b.kcache = c->kcache;
        b.vcache = c->vcache;
        b.rope = c->rope;
        b.hb = c->hb;
        b.logits = c->logits;
        b.step = c->step_dev;
        b.err = c->err;
        b.dim = p.dim;
        b.kv_dim = c->kv_dim;
        b.head_size = c->head_size;
        b.seq_len = p.seq_len;
        b.n_kv_heads = p.n_kv_heads;
        b.n_layers = p.n_layers;
        b.vocab = p.vocab_size;
        b.evict_first = c->evict_first ? 1 : 0;
        b.ext = c->ext_dev;
    };
    plan(c->plan_qkv, GEMV_QKV, p.dim, 2, (p.dim + 2 * c->kv_dim) / 2, 1);
    plan(c->plan_wo, GEMV_RESID, p.dim, 1, p.dim, 1);
    plan(c->plan_w13, GEMV_W13, p.dim, 1, p.hidden_dim, 2);
    plan(c->plan_w2, GEMV_RESID, p.hidden_dim, 1, p.dim, 1);
    plan(c->plan_cls, GEMV_CLS, p.dim, 1, p.vocab_size, 1);
    c->plan_qkv.base.rows0 = p.dim;
    c->plan_qkv.base.rows1 = c->kv_dim;
    c->plan_qkv.base.rows2 = c->kv_dim;
    c->plan_wo.base.in_vec = c->xb;
    c->plan_w2.base.in_vec = c->hb;
    c->plan_cls.base.mat0 = c->wt ? reinterpret_cast<const float *>(c->b16cls) : c->w.wcls;
    c->plan_cls.base.norm_w = c->w.rms_final_weight;
}

GemvParams layer_params(const l2_ctx *c, const GemvPlan &pl, int layer) {
    const L2Config &p = c->cfg;
    GemvParams g = pl.base;
    g.layer = layer;
    const size_t l = (size_t)layer;
    const size_t dd = (size_t)p.dim * p.dim, kd = (size_t)c->kv_dim * p.dim, hd = (size_t)p.hidden_dim * p.dim;
    if (c->wt) {
        // bf16 copies: element offsets in bf16 units
        auto f = [](const unsigned short *q) { return reinterpret_cast<const float *>(q); };
        if (&pl == &c->plan_qkv) {
            g.mat0 = f(c->b16q + l * dd);
            g.mat1 = f(c->b16k + l * kd);
            g.mat2 = f(c->b16v + l * kd);
            g.norm_w = c->w.rms_att_weight + l * p.dim;
        } else if (&pl == &c->plan_wo) {
            g.mat0 = f(c->b16o + l * dd);
        } else if (&pl == &c->plan_w13) {
            g.mat0 = f(c->b16w1 + l * hd);
            g.mat1 = f(c->b16w3 + l * hd);
            g.norm_w = c->w.rms_ffn_weight + l * p.dim;
        } else if (&pl == &c->plan_w2) {
            g.mat0 = f(c->b16w2 + l * hd);
        }
        return g;
    }
    if (&pl == &c->plan_qkv) {
        g.mat0 = c->w.wq + l * dd;
        g.mat1 = c->w.wk + l * kd;
        g.mat2 = c->w.wv + l * kd;
        g.norm_w = c->w.rms_att_weight + l * p.dim;
    } else if (&pl == &c->plan_wo) {
        g.mat0 = c->w.wo + l * dd;
    } else if (&pl == &c->plan_w13) {
        g.mat0 = c->w.w1 + l * hd;
        g.mat1 = c->w.w3 + l * hd;
        g.norm_w = c->w.rms_ffn_weight + l * p.dim;
    } else if (&pl == &c->plan_w2) {
        g.mat0 = c->w.w2 + l * hd;
    }
    return g;
}

// Attention CTAs per (slot, KV head): as many as fill every SM with the
// CTAs that fit on it, in one wave, and no more than one per kMinChunk
// positions of the cache.
int attn_chunks_for(const l2_ctx *c, int batch) {
    int per_sm = c->attn_per_sm;
    if (per_sm > L2_ATTN_MAX_PER_SM) per_sm = L2_ATTN_MAX_PER_SM;
    int nc = (int)(((long long)per_sm * c->num_sms) / ((long long)c->cfg.n_kv_heads * batch));
    const int cap = ceil_div(c->cfg.seq_len, kMinChunk);
    if (nc > cap) nc = cap;
    return nc < 1 ? 1 : nc;
}

AttnParams attn_params(const l2_ctx *c, int layer, int batch) {
    const L2Config &p = c->cfg;
    AttnParams a{};
    a.q = c->q;
    a.kcache = c->kcache;
    a.vcache = c->vcache;
    a.out = c->xb;
    a.ws_ml = c->ws_ml;
    a.ws_acc = c->ws_acc;
    a.tickets = c->tickets;
    a.dbg = c->dbg;
    a.step = c->step_dev;
    a.err = c->err;
    a.layer = layer;
    a.n_layers = p.n_layers;
    a.n_heads = p.n_heads;
    a.n_kv_heads = p.n_kv_heads;
    a.head_size = c->head_size;
    a.seq_len = p.seq_len;
    a.dim = p.dim;
    int nc = attn_chunks_for(c, batch);
    a.capacity = 0;
    if (batch > 1) {
        // Rows sit at different positions: each row's CTAs per KV head are planned on
        // the host (attn_chunk_plan) so that the step's CTAs fit `capacity` at once;
        // a row never gets more than capacity / n_kv_heads of them, and the grid
        // stops one above that.
        a.capacity = c->attn_per_sm * c->num_sms;
        nc = std::min(ceil_div(p.seq_len, kMinChunk), ceil_div(a.capacity, p.n_kv_heads) + 1);
    }
    if (nc > c->attn_chunks) nc = c->attn_chunks;
    a.n_chunks = nc;
    a.cluster = batch == 1 && c->attn_cluster == nc ? nc : 0;
    a.min_chunk = kMinChunk;
    a.scale = (float)(1.0 / std::sqrt((double)c->head_size));
    a.ext = c->ext_dev;
    return a;
}

// Attention CTAs per KV head for each row of a step of several rows, written
// into the step block with the order the grid takes the rows in.  Row b
// (P_b = pos[b] + 1 positions) gets n_b = ceil(P_b / X) CTAs, at least one and
// at most the grid's chunk dimension or one per kMinChunk positions.  X is
// chosen from a simple model of the launch: it lasts about
// max(X, all positions / capacity) -- the longest CTA, or the resident CTAs
// working through everything -- plus a fixed cost per CTA (kAttnCtaCost
// positions' worth: its ring fill and share of the merge) times the CTAs per
// resident slot.  Rows are taken longest CTA first, so the long CTAs start in
// the first wave and shorter ones fill in behind them.  (Sizing every row
// from the step's mean instead overflowed the capacity into an unbalanced
// second wave of CTAs with staggered positions.)
#ifndef L2_ATTN_CTA_COST
#define L2_ATTN_CTA_COST 96
#endif
constexpr int kAttnCtaCost = L2_ATTN_CTA_COST;

void attn_chunk_plan(const l2_ctx *c, int B, const int *pos, unsigned short *out, unsigned char *order) {
    const AttnParams a = attn_params(c, 0, B);
    const long long slots = std::max(1, a.capacity / c->cfg.n_kv_heads);  // resident CTAs per KV head
    int cap[kMaxBatch];
    long long work = 0;
    int pmax = 1;
    for (int b = 0; b < B; ++b) {
        cap[b] = std::max(1, std::min(a.n_chunks, ceil_div(pos[b] + 1, kMinChunk)));
        work += pos[b] + 1;
        pmax = std::max(pmax, pos[b] + 1);
    }
    auto count = [&](int X, int b) { return std::max(1, std::min(cap[b], ceil_div(pos[b] + 1, X))); };
    auto cost = [&](int X, int &longest) {
        long long ctas = 0;
        longest = 0;
        for (int b = 0; b < B; ++b) {
            const int n = count(X, b);
            ctas += n;
            longest = std::max(longest, ceil_div(pos[b] + 1, n));
        }
        return std::max<long long>(longest, (work + slots - 1) / slots) + kAttnCtaCost * ((ctas + slots - 1) / slots);
    };
    int bestX = pmax, longest = 0;
    long long best = cost(pmax, longest);
    for (int X = kMinChunk; X < pmax; X += std::max(kMinChunk / 4, X / 8)) {
        const long long v = cost(X, longest);
        if (v < best) {
            best = v;
            bestX = X;
        }
    }
    int len[kMaxBatch];
    for (int b = 0; b < B; ++b) {
        out[b] = (unsigned short)count(bestX, b);
        len[b] = ceil_div(pos[b] + 1, out[b]);
        order[b] = (unsigned char)b;
    }
    std::stable_sort(order, order + B, [&](unsigned char x, unsigned char y) { return len[x] > len[y]; });
}

// ---- batched GEMV plans: grid, tensor maps and tiles per batch size ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Row-major fp32 matrix [rows][cols] seen as 2-D tiles of box_rows x box_cols.
bool encode_matrix(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                   uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major fp32 matrix [rows][cols] seen as tiles of box_rows x 32 columns
// (128-byte lines) with the 128-byte swizzle the tensor-core operands use.
bool encode_matrix_sw128(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 4};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of ss_part a residual plan (Wo: 1, W2: 3) writes: one per tile, or per
// tile and cluster rank with the cluster split.
int tc_ss_parts(const BatchSet &set, int k) {
    const TcParams &tp = set.tcp[k];
    return tp.ntiles * (tp.csplit > 1 ? tp.csplit : 1);
}

// A weight matrix [rows][cols] for the tensor-core GEMV: fp32 in boxes of
// box_rows x 32 columns, or (the handle's bf16 copies) bf16 in boxes of
// box_rows x 64 columns -- 128-byte lines with the 128-byte swizzle either way.
bool encode_weights_sw128(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows, int wt) {
    if (!wt) return encode_matrix_sw128(m, base, cols, rows, box_rows);
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor-core plans of a batch size (16..64 rows): tiles of 128 output
// rows (64 of W1 over 64 of W3), the work split evenly over the SMs.
int build_tc_set(l2_ctx *c, int batch) {
    const L2Config &p = c->cfg;
    BatchSet &set = c->bsets[batch];
    const uint64_t L = p.n_layers, D = p.dim, H = p.hidden_dim, KVD = c->kv_dim, V = p.vocab_size;
    const int bpad = (batch + 15) / 16 * 16;
    const int wt = c->wt;
    // the weights a plan streams: the caller's fp32 matrices, or the handle's bf16 copies
    auto W = [&](const float *f32, const unsigned short *b16) { return wt ? (const void *)b16 : (const void *)f32; };
    set.tc_ws_floats = 0;
    set.tc_tiles = 0;
    // the inputs as fp32 (bf16 weights: split into bf16 parts in the kernel), or as their
    // tf32 hi and lo parts written by the producing kernel (fp32 weights)
    auto xmaps = [&](TcParams &tp, const float *f32, const float *hi, const float *lo, uint64_t cols) {
        tp.xsplit = hi && lo ? 1 : 0;
        if (!tp.xsplit) return encode_matrix_sw128(&tp.xmap, f32, cols, c->max_rows, bpad);
        return encode_matrix_sw128(&tp.xmap, hi, cols, c->max_rows, bpad) &&
               encode_matrix_sw128(&tp.xmap_lo, lo, cols, c->max_rows, bpad);
    };
    for (int k = 0; k < 5; ++k) {
        TcParams &tp = set.tcp[k];
        memset(&tp, 0, sizeof(tp));
        tp.bpad = bpad;
        tp.wt = c->wt;
        tp.stages = gemv_tc_stages(bpad, c->wt);
        bool ok = true;
        int n = 0;
        switch (k) {
            case 0:
                tp.mrows[0] = p.dim;
                tp.mrows[1] = tp.mrows[2] = c->kv_dim;
                for (int m = 0; m < 3; ++m) tp.tiles[m] = ceil_div(tp.mrows[m], 128);
                ok = encode_weights_sw128(&tp.wmap[0], W(c->w.wq, c->b16q), D, L * D, 128, wt) &&
                     encode_weights_sw128(&tp.wmap[1], W(c->w.wk, c->b16k), D, L * KVD, 128, wt) &&
                     encode_weights_sw128(&tp.wmap[2], W(c->w.wv, c->b16v), D, L * KVD, 128, wt) &&
                     xmaps(tp, c->xg, c->xg_hi, c->xg_lo, D);
                n = p.dim;
                break;
            case 1:
                tp.mrows[0] = p.dim;
                tp.tiles[0] = ceil_div(p.dim, 128);
                ok = encode_weights_sw128(&tp.wmap[0], W(c->w.wo, c->b16o), D, L * D, 128, wt) &&
                     encode_matrix_sw128(&tp.xmap, c->xb, D, c->max_rows, bpad);
                n = p.dim;
                break;
            case 2:
                tp.mrows[0] = p.hidden_dim;
                tp.tiles[0] = ceil_div(p.hidden_dim, 64);
                ok = encode_weights_sw128(&tp.wmap[0], W(c->w.w1, c->b16w1), D, L * H, 64, wt) &&
                     encode_weights_sw128(&tp.wmap[1], W(c->w.w3, c->b16w3), D, L * H, 64, wt) &&
                     xmaps(tp, c->xg, c->xg_hi, c->xg_lo, D);
                n = p.dim;
                break;
            case 3:
                tp.mrows[0] = p.dim;
                tp.tiles[0] = ceil_div(p.dim, 128);
                ok = encode_weights_sw128(&tp.wmap[0], W(c->w.w2, c->b16w2), H, L * D, 128, wt) &&
                     xmaps(tp, c->hb, c->hb_hi, c->hb_lo, H);
                n = p.hidden_dim;
                break;
            case 4:
                tp.mrows[0] = p.vocab_size;
                tp.tiles[0] = ceil_div(p.vocab_size, 128);
                ok = encode_weights_sw128(&tp.wmap[0], W(c->w.wcls, c->b16cls), D, V, 128, wt) &&
                     xmaps(tp, c->xg, c->xg_hi, c->xg_lo, D);
                n = p.dim;
                break;
        }
        if (!ok) return fail(c, L2_ECUDA, "cuTensorMapEncodeTiled failed for a tensor-core GEMV plan");
        tp.ntiles = tp.tiles[0] + tp.tiles[1] + tp.tiles[2];
        static const int modes[5] = {GEMV_QKV, GEMV_RESID, GEMV_W13, GEMV_RESID, GEMV_CLS};
        tp.csplit = gemv_tc_cluster_split(modes[k], c->wt, tp.ntiles, n, bpad, c->num_sms);
        set.tc_grid[k] = tp.csplit > 1 ? tp.ntiles * tp.csplit : gemv_tc_grid(tp.ntiles, n, c->num_sms);
        set.tc_ws_floats = std::max(set.tc_ws_floats, gemv_tc_ws_floats(set.tc_grid[k], bpad));
        set.tc_tiles = std::max(set.tc_tiles, tp.ntiles);
    }
    if (tc_ss_parts(set, 1) > kMaxParts || tc_ss_parts(set, 3) > kMaxParts)
        return fail(c, L2_EINVAL, "too many residual tiles for the sum-of-squares parts");
    set.tc = true;
    return L2_OK;
}

// Builds the five batched GEMV plans (QKV, Wo, W1/W3, W2, classifier) for
// `batch` sequences.  Returns L2_OK or an error code.
int build_batch_set(l2_ctx *c, int batch) {
    const L2Config &p = c->cfg;
    BatchSet &set = c->bsets[batch];
    const int cap = gemv_batched_rows_cap(batch);
    const GemvPlan *plans[5] = {&c->plan_qkv, &c->plan_wo, &c->plan_w13, &c->plan_w2, &c->plan_cls};
    const size_t L = p.n_layers;
    for (int k = 0; k < 5; ++k) {
        const GemvPlan &pl = *plans[k];
        BatchPlan &bpl = set.plan[k];
        BatchParams &bp = bpl.bp;
        memset(&bp, 0, sizeof(bp));
        const int npc = pl.mode == GEMV_W13 ? 2 : 1;
        // one CTA per SM, each owning a balanced row range that it walks in
        // blocks of at most cap / npc rows (whole units)
        int grid = 0, rows_max = 0;
        if (pl.mode == GEMV_QKV) {
            const int u[3] = {p.dim / 2, c->kv_dim / 2, c->kv_dim / 2};
            const int total = u[0] + u[1] + u[2];
            const int target = c->num_sms > 3 ? c->num_sms : 3;
            for (int m = 0; m < 3; ++m) {
                int g = (int)(((long long)target * u[m] + total / 2) / total);
                if (g > u[m]) g = u[m];
                if (g < 1) g = 1;
                bp.part_ctas[m] = g;
                bp.part_units[m] = u[m];
                grid += g;
                const int r = ceil_div(u[m], g) * 2;
                if (r > rows_max) rows_max = r;
            }
        } else {
            grid = pl.units < c->num_sms ? pl.units : c->num_sms;
            bp.part_ctas[0] = grid;
            bp.part_units[0] = pl.units;
            rows_max = ceil_div(pl.units, grid) * pl.unit_rows;
        }
        int block_cap = (cap / npc) / pl.unit_rows * pl.unit_rows;  // whole units per block
        if (block_cap < pl.unit_rows) block_cap = pl.unit_rows;
        const int nblocks = ceil_div(rows_max, block_cap);
        int rows_box = ceil_div(ceil_div(rows_max, nblocks), pl.unit_rows) * pl.unit_rows;
        bp.rows_box = rows_box;
        bpl.grid = grid;
        bpl.smem = gemv_batched_smem(npc * rows_box, batch, pl.base.n, pl.mode != GEMV_RESID, &bp.stages, &bp.tk);
        if (bpl.smem > 227 * 1024 || npc * rows_box > cap)
            return fail(c, L2_EINVAL, "a batched GEMV of %d sequences does not fit one CTA", batch);
        if (pl.mode == GEMV_RESID && grid > kMaxParts)
            return fail(c, L2_EINVAL, "a batched residual GEMV of %d sequences needs too many CTAs", batch);
        // weight tensor maps: all layers stacked as one tall matrix
        const uint32_t tk = (uint32_t)bp.tk, rb = (uint32_t)rows_box;
        bool ok = true;
        const uint64_t D = p.dim, H = p.hidden_dim, KVD = c->kv_dim;
        switch (k) {
            case 0:
                ok = encode_matrix(&bp.wmap[0], c->w.wq, D, L * D, tk, rb) &&
                     encode_matrix(&bp.wmap[1], c->w.wk, D, L * KVD, tk, rb) &&
                     encode_matrix(&bp.wmap[2], c->w.wv, D, L * KVD, tk, rb) &&
                     encode_matrix(&bp.xmap, c->x, D, c->max_rows, tk, batch);
                break;
            case 1:
                ok = encode_matrix(&bp.wmap[0], c->w.wo, D, L * D, tk, rb) &&
                     encode_matrix(&bp.xmap, c->xb, D, c->max_rows, tk, batch);
                break;
            case 2:
                ok = encode_matrix(&bp.wmap[0], c->w.w1, D, L * H, tk, rb) &&
                     encode_matrix(&bp.wmap[1], c->w.w3, D, L * H, tk, rb) &&
                     encode_matrix(&bp.xmap, c->x, D, c->max_rows, tk, batch);
                break;
            case 3:
                ok = encode_matrix(&bp.wmap[0], c->w.w2, H, L * D, tk, rb) &&
                     encode_matrix(&bp.xmap, c->hb, H, c->max_rows, tk, batch);
                break;
            case 4:
                ok = encode_matrix(&bp.wmap[0], c->w.wcls, D, (uint64_t)p.vocab_size, tk, rb) &&
                     encode_matrix(&bp.xmap, c->x, D, c->max_rows, tk, batch);
                break;
        }
        if (!ok) return fail(c, L2_ECUDA, "cuTensorMapEncodeTiled failed for a batched GEMV plan");
    }
    set.built = true;
    return L2_OK;
}

cudaError_t launch_batched(l2_ctx *c, int k, const GemvPlan &pl, int layer, int batch, cudaStream_t s, bool pdl) {
    const BatchSet &set = c->bsets[batch];
    if (set.tc) {
        TcParams tp = set.tcp[k];
        tp.g = layer_params(c, pl, layer);
        tp.g.batch = batch;
        tp.g.ss_part = c->ss_part;
        // the sums of squares come from the embedding kernel (layer 0), Wo (for W1/W3) or W2
        tp.g.ss_parts = (k == 0 && layer == 0) ? 1 : tc_ss_parts(set, k == 2 ? 1 : 3);
        tp.ws = c->tc_ws;
        tp.tickets = c->tc_tickets;
        tp.xg = c->xg;
        tp.xg_hi = c->xg_hi;
        tp.xg_lo = c->xg_lo;
        tp.hb_hi = c->hb_hi;
        tp.hb_lo = c->hb_lo;
        const L2Config &cf = c->cfg;
        if (k == 1) tp.next_gain = c->w.rms_ffn_weight + (size_t)layer * cf.dim;
        if (k == 3)
            tp.next_gain = layer + 1 < cf.n_layers ? c->w.rms_att_weight + (size_t)(layer + 1) * cf.dim
                                                   : c->w.rms_final_weight;
        if (k == 0 && layer == 0) {
            cudaError_t e = launch_tc_embed(tp, batch, s, pdl);
            if (e != cudaSuccess) return e;
        }
        return launch_gemv_tc(pl.mode, tp, set.tc_grid[k], s, pdl);
    }
    const BatchPlan &bpl = c->bsets[batch].plan[k];
    BatchParams bp = bpl.bp;
    bp.g = layer_params(c, pl, layer);
    bp.g.batch = batch;
    bp.g.ss_part = c->ss_part;
    bp.g.ss_parts = c->bsets[batch].plan[1].grid;  // the residual kernels' grid
    return launch_gemv_batched(pl.mode, bp, bpl.grid, bpl.smem, s, pdl);
}

// The persistent batch-1 step kernel (L2_FLAG_PERSIST): used when the device
// launches cooperative kernels, one CTA per SM fits (shared memory for the
// largest phase), the attention items of a step fit the grid and two cache
// rows fit one ring buffer; not with L2_FLAG_DEBUG (it keeps no
// probabilities).
int plan_persistent(l2_ctx *c) {
    c->persist = false;
    if (!(c->flags & L2_FLAG_PERSIST) || (c->flags & L2_FLAG_DEBUG)) return L2_OK;
    const L2Config &p = c->cfg;
    const int G = c->num_sms;
    int coop = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, c->device) != cudaSuccess) {
        cudaGetLastError();
        return L2_OK;
    }
    if (!coop || p.n_kv_heads > G) return L2_OK;
    auto per_cta = [&](int units) { return ceil_div(units, G); };
    int ys = 2 * per_cta((p.dim + 2 * c->kv_dim) / 2);
    ys = std::max(ys, per_cta(p.dim));
    ys = std::max(ys, 2 * per_cta(p.hidden_dim));
    ys = std::max(ys, per_cta(p.vocab_size));
    const int xs = std::max(p.dim, p.hidden_dim);
    const int gq = c->attn.gq;
    int stages = L2_STEP_STAGES, ch4 = step_kernel_ring(gq, c->head_size, xs, ys, stages, L2_STEP_MAX_CHUNK_WORDS);
    if (!ch4) {
        stages = 2;
        ch4 = step_kernel_ring(gq, c->head_size, xs, ys, stages, L2_STEP_MAX_CHUNK_WORDS);
    }
    if (!ch4) return L2_OK;
    const size_t smem = step_kernel_smem(gq, c->head_size, xs, ys, stages, ch4);
    if (smem > 227 * 1024) return L2_OK;
    cudaError_t e = step_kernel_init();
    if (e != cudaSuccess) return cuda_fail(c, e, "step_kernel_init()");
    if (step_kernel_ctas_per_sm(gq, smem) < 1) return L2_OK;
    int nc = G / p.n_kv_heads;
    nc = std::min(nc, ceil_div(p.seq_len, kMinChunk));
    nc = std::min(nc, c->attn_chunks);
    if (nc < 1) return L2_OK;

    StepKParams &k = c->sp;
    k = StepKParams{};
    k.emb = c->w.token_embedding_table;
    k.rms_att = c->w.rms_att_weight;
    k.rms_ffn = c->w.rms_ffn_weight;
    k.rms_final = c->w.rms_final_weight;
    k.wq = c->w.wq;
    k.wk = c->w.wk;
    k.wv = c->w.wv;
    k.wo = c->w.wo;
    k.w1 = c->w.w1;
    k.w2 = c->w.w2;
    k.w3 = c->w.w3;
    k.wcls = c->w.wcls;
    k.x = c->x;
    k.xb = c->xb;
    k.q = c->q;
    k.hb = c->hb;
    k.logits = c->logits;
    k.kcache = c->kcache;
    k.vcache = c->vcache;
    k.rope = c->rope;
    k.ws_ml = c->ws_ml;
    k.ws_acc = c->ws_acc;
    k.tickets = c->tickets;
    k.step = c->step_dev;
    k.err = c->err;
    k.dim = p.dim;
    k.hidden_dim = p.hidden_dim;
    k.n_layers = p.n_layers;
    k.n_heads = p.n_heads;
    k.n_kv_heads = p.n_kv_heads;
    k.head_size = c->head_size;
    k.kv_dim = c->kv_dim;
    k.vocab = p.vocab_size;
    k.seq_len = p.seq_len;
    k.n_chunks = nc;
    k.min_chunk = kMinChunk;
    // one 16-byte word of a cache row per lane (the decode attention kernel may
    // give a lane several; this kernel's attention phase does not)
    k.lp = 1;
    while (k.lp < c->head_size / 4) k.lp <<= 1;
    k.xs_floats = xs;
    k.ys_floats = ys;
    k.evict_first = c->evict_first ? 1 : 0;
    k.stages = stages;
    k.ch4 = ch4;
    k.scale = (float)(1.0 / std::sqrt((double)c->head_size));
    c->persist_gq = gq;
    c->persist_smem = smem;
    c->persist = true;
    return L2_OK;
}

// The one-block step kernel (step_cta.cu) for batch-1 steps of a model whose
// weights fit a few MB (L2-resident: a step of per-matrix launches costs its
// kernel boundaries, not its bytes): the default unless L2_FLAG_NO_ONE_CTA,
// L2_FLAG_PERSIST or L2_FLAG_BF16_WEIGHTS is set, when its shared memory fits.
// With L2_FLAG_DEBUG it exports the probabilities as the attention kernel does.
constexpr double kCtaMaxWeightBytes = 4.0 * 1024 * 1024;

int plan_cta(l2_ctx *c) {
    c->cta = false;
    if (c->flags & (L2_FLAG_NO_ONE_CTA | L2_FLAG_PERSIST | L2_FLAG_BF16_WEIGHTS)) return L2_OK;
    const L2Config &p = c->cfg;
    const double d = p.dim, h = p.hidden_dim, kv = c->kv_dim, L = p.n_layers, V = p.vocab_size;
    const double bytes = 4.0 * (L * (2 * d * d + 2 * kv * d + 3 * d * h + 2 * d) + V * d + d);
    if (bytes > kCtaMaxWeightBytes) return L2_OK;
    const size_t smem = step_cta_smem(p.dim, p.hidden_dim, c->kv_dim, p.n_heads, p.seq_len, p.n_layers);
    if (smem > 227 * 1024) return L2_OK;
    cudaError_t e = step_cta_init();
    if (e != cudaSuccess) return cuda_fail(c, e, "step_cta_init()");
    CtaStepParams &k = c->ctap;
    k = CtaStepParams{};
    k.emb = c->w.token_embedding_table;
    k.rms_att = c->w.rms_att_weight;
    k.rms_ffn = c->w.rms_ffn_weight;
    k.rms_final = c->w.rms_final_weight;
    k.wq = c->w.wq;
    k.wk = c->w.wk;
    k.wv = c->w.wv;
    k.wo = c->w.wo;
    k.w1 = c->w.w1;
    k.w2 = c->w.w2;
    k.w3 = c->w.w3;
    k.wcls = c->w.wcls;
    k.x = c->x;
    k.logits = c->logits;
    k.kcache = c->kcache;
    k.vcache = c->vcache;
    k.rope = c->rope;
    k.dbg = c->dbg;
    k.step = c->step_dev;
    k.err = c->err;
    k.ext = c->ext_dev;
    k.dim = p.dim;
    k.hidden_dim = p.hidden_dim;
    k.n_layers = p.n_layers;
    k.n_heads = p.n_heads;
    k.n_kv_heads = p.n_kv_heads;
    k.head_size = c->head_size;
    k.kv_dim = c->kv_dim;
    k.vocab = p.vocab_size;
    k.seq_len = p.seq_len;
    k.scale = (float)(1.0 / std::sqrt((double)c->head_size));
    c->cta_smem = smem;
    c->cta = true;
    return L2_OK;
}

// The prompt-chunk attention reads each K/V tile once per 16 query vectors but
// walks all of a block's positions in one CTA: it beats the per-row kernel
// (which shares a tile among a group's query heads and splits positions over
// the SMs) when groups are small and the chunk gives enough CTAs.
bool attn_prefill_pays(const l2_ctx *c, int batch) {
    if (!c->attn_pf || batch < 2) return false;
    const int gq = c->cfg.n_heads / c->cfg.n_kv_heads;
    const int ctas = ceil_div(batch, 16 / gq) * c->cfg.n_kv_heads;
    return gq <= 2 && 2 * ctas >= c->num_sms;
}

// prefill: the step is a prompt chunk (rows of one slot at consecutive positions).
cudaError_t launch_op(l2_ctx *c, int op, int layer, int batch, cudaStream_t s, bool pdl, bool prefill = false) {
    if (batch > 1 && op != 1) {
        const GemvPlan *pl[] = {&c->plan_qkv, nullptr, &c->plan_wo, &c->plan_w13, &c->plan_w2, &c->plan_cls};
        const int k = op == 0 ? 0 : op - 1;  // index into the batch set's plans
        return launch_batched(c, k, *pl[op], op == 5 ? 0 : layer, batch, s, pdl);
    }
    switch (op) {
        case 0: {
            GemvParams g = layer_params(c, c->plan_qkv, layer);
            return launch_gemv(GEMV_QKV, c->plan_qkv.shape, g, c->plan_qkv.grid, c->plan_qkv.smem, s, pdl, c->wt);
        }
        case 1: {
            AttnParams a = attn_params(c, layer, batch);
            if (prefill && attn_prefill_pays(c, batch)) return launch_attn_prefill(a, batch, s, pdl);
            return launch_attn(c->attn, a, batch, s, pdl);
        }
        case 2: {
            GemvParams g = layer_params(c, c->plan_wo, layer);
            return launch_gemv(GEMV_RESID, c->plan_wo.shape, g, c->plan_wo.grid, c->plan_wo.smem, s, pdl, c->wt);
        }
        case 3: {
            GemvParams g = layer_params(c, c->plan_w13, layer);
            return launch_gemv(GEMV_W13, c->plan_w13.shape, g, c->plan_w13.grid, c->plan_w13.smem, s, pdl, c->wt);
        }
        case 4: {
            GemvParams g = layer_params(c, c->plan_w2, layer);
            return launch_gemv(GEMV_RESID, c->plan_w2.shape, g, c->plan_w2.grid, c->plan_w2.smem, s, pdl, c->wt);
        }
        case 5: {
            GemvParams g = layer_params(c, c->plan_cls, 0);
            return launch_gemv(GEMV_CLS, c->plan_cls.shape, g, c->plan_cls.grid, c->plan_cls.smem, s, pdl, c->wt);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t enqueue_step(l2_ctx *c, int batch, cudaStream_t s, bool prefill = false) {
    const bool pdl = !(c->flags & L2_FLAG_NO_PDL);
    cudaError_t e;
    for (int l = 0; l < c->cfg.n_layers; ++l)
        for (int op = 0; op < 5; ++op)
            if ((e = launch_op(c, op, l, batch, s, pdl, prefill)) != cudaSuccess) return e;
    return launch_op(c, 5, 0, batch, s, pdl, prefill);
}

int get_graph(l2_ctx *c, int batch, bool prefill, cudaGraphExec_t *out) {
    cudaGraphExec_t *slot = prefill ? &c->graph_pf[batch] : &c->graph[batch];
    if (*slot) {
        *out = *slot;
        return L2_OK;
    }
    cudaGraph_t g = nullptr;
    L2_CUDA(c, cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    cudaError_t e = enqueue_step(c, batch, c->cap_stream, prefill);
    cudaError_t e2 = cudaStreamEndCapture(c->cap_stream, &g);
    if (e != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return cuda_fail(c, e, "kernel launch during graph capture");
    }
    if (e2 != cudaSuccess) return cuda_fail(c, e2, "cudaStreamEndCapture");
    if (g_fail_graph_at > 0 && --g_fail_graph_at == 0) {
        cudaGraphDestroy(g);
        return fail(c, L2_ECUDA, "cudaGraphInstantiate failed (injected)");
    }
    cudaGraphExec_t ex = nullptr;
    e = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGraphInstantiate");
    *slot = ex;
    *out = ex;
    return L2_OK;
}

// Failure-path check (l2_debug_wait_timeout): one CTA completes a bulk copy
// into stage 0 of a two-stage ring, then waits on stage 1, which nothing ever
// fills, with a short limit.  The wait gives up and sets the error word; the
// CTA then waits (bounded) for its copy in flight and returns, as the decode
// kernels do.  It also leaves every attention ticket counted once, as a chunk
// merge that stopped before resetting its ticket would.
__global__ void __launch_bounds__(32)
    debug_wait_kernel(const float *src, uint32_t bytes, int *err, unsigned *tickets, int n_tickets,
                      unsigned long long limit_ns) {
    __shared__ __align__(128) float buf[32];
    __shared__ __align__(8) uint64_t bars[2];
    if (threadIdx.x == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&bars[0], bytes);
        bulk_g2s_nohint(buf, src, bytes, &bars[0]);
    }
    const bool filled = mbar_wait_limit(&bars[1], 0, err, limit_ns);  // nothing arrives: gives up
    if (!filled) (void)mbar_wait_limit(&bars[0], 0, err, kWaitLimitNs);
    for (int i = threadIdx.x; i < n_tickets; i += 32) atomicAdd(&tickets[i], 1u);
}

// Copies B tokens from device memory into the step block, each checked
// against the vocabulary (an out-of-range token sets L2_DEV_ERR_BOUNDS in the
// error word and token 0 is used in its place).
__global__ void set_step_tokens(StepDev *step, const int *tokens, int B, int vocab, int *err) {
    const int b = threadIdx.x;
    if (b < B) {
        int t = tokens[b];
        if (t < 0 || t >= vocab) {
            atomicOr(err, L2_DEV_ERR_BOUNDS);
            t = 0;
        }
        step->token[b] = t;
    }
}

// tokens_dev: when not NULL, the step's tokens are read from this device
// array when the step runs (tokens is then ignored).  prefill_slot >= 0: the
// B rows are consecutive positions pos[0].. of that one slot (a prompt
// chunk, checked by the caller) instead of one position of each of slots
// 0..B-1.
int submit(l2_ctx *c, int B, const int *tokens, const int *pos, float *logits_out, const int *tokens_dev = nullptr,
           int prefill_slot = -1) {
    const int cap = prefill_slot >= 0 ? c->max_rows : c->max_batch;
    if (B < 1 || B > cap) return fail(c, L2_EINVAL, "batch %d outside 1..%d", B, cap);
    for (int b = 0; b < B; ++b) {
        if (!tokens_dev && (tokens[b] < 0 || tokens[b] >= c->cfg.vocab_size))
            return fail(c, L2_EINVAL, "token %d of slot %d outside [0, %d)", tokens[b], b, c->cfg.vocab_size);
        if (prefill_slot >= 0) continue;
        if (pos[b] < 0 || pos[b] >= c->cfg.seq_len)
            return fail(c, L2_EINVAL, "pos %d of slot %d outside [0, %d)", pos[b], b, c->cfg.seq_len);
        if (pos[b] > c->written[b])
            return fail(c, L2_ESTATE, "pos %d of slot %d skips cache rows (only %d written)", pos[b], b, c->written[b]);
    }
    if (logits_out && (reinterpret_cast<uintptr_t>(logits_out) & 3u))
        return fail(c, L2_EINVAL, "logits_out must be 4-byte aligned");

    const int i = c->ring_next;
    c->ring_next = (i + 1) % kRing;
    if (c->ring_used[i]) L2_CUDA(c, cudaEventSynchronize(c->ring_ev[i]));
    StepDev &sh = c->step_host[i];
    for (int b = 0; b < B; ++b) {
        sh.token[b] = tokens_dev ? 0 : tokens[b];
        sh.pos[b] = pos[b];
        sh.slot[b] = prefill_slot >= 0 ? prefill_slot : b;
        sh.stable[b] = prefill_slot >= 0 ? pos[0] : pos[b];
    }
    if (B > 1) attn_chunk_plan(c, B, pos, sh.nchunk, sh.row_order);
    sh.logits_out = logits_out;
    sh.B = B;
    sh.sync_count = 0;
    c->last_rows = B;
    c->last_prefill = prefill_slot >= 0;
    L2_CUDA(c, cudaMemcpyAsync(c->step_dev, &sh, sizeof(StepDev), cudaMemcpyHostToDevice, c->stream));
    L2_CUDA(c, cudaEventRecord(c->ring_ev[i], c->stream));
    c->ring_used[i] = true;
    if (tokens_dev) {
        set_step_tokens<<<1, kMaxBatch, 0, c->stream>>>(c->step_dev, tokens_dev, B, c->cfg.vocab_size, c->err);
        L2_CUDA(c, cudaGetLastError());
    }

    if (B == 1 && c->cta && prefill_slot < 0) {
        L2_CUDA(c, launch_step_cta(c->ctap, c->cta_smem, c->stream));
    } else if (B == 1 && c->persist && sh.slot[0] == 0) {
        L2_CUDA(c, launch_step_kernel(c->persist_gq, c->sp, c->num_sms, c->persist_smem, c->stream));
    } else if (c->flags & L2_FLAG_NO_GRAPH) {
        L2_CUDA(c, enqueue_step(c, B, c->stream, prefill_slot >= 0));
    } else {
        cudaGraphExec_t g = nullptr;
        int rc = get_graph(c, B, prefill_slot >= 0, &g);
        if (rc != L2_OK) return rc;
        L2_CUDA(c, cudaGraphLaunch(g, c->stream));
    }
    if (prefill_slot >= 0)
        c->written[prefill_slot] = pos[B - 1] + 1;
    else
        for (int b = 0; b < B; ++b) c->written[b] = pos[b] + 1;
    return L2_OK;
}

}  // namespace

// Attention scratch of l2_forward_static: accumulators, (max, sum) pairs and
// tickets, 512 KiB.  Every GPU that loads the library holds it until exit.  In
// host code this name is only a stand-in: kernels get the address that
// cudaGetSymbolAddress returns for the current device, looked up by l2_create
// (so the module that holds the array is loaded, and the array allocated,
// when the first handle on a device is created, not by a later decode call).
constexpr size_t kStaticScratchFloats = size_t(1) << 17;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
float *g_static_scratch_ptr[kMaxDevices] = {};  // device address, per device

// The array's device address on `device`, which must be current; looked up
// once per device.
int static_scratch_address(l2_ctx *c, int device, float **out) {
    *out = nullptr;
    if (device < 0 || device >= kMaxDevices) return fail(c, L2_EINVAL, "device index %d too large", device);
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_ptr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetSymbolAddress(static attention scratch)");
        g_static_scratch_ptr[device] = static_cast<float *>(p);
    }
    *out = g_static_scratch_ptr[device];
    return L2_OK;
}

}  // namespace

extern "C" {

int l2_create(const L2Config *config, const L2Weights *weights, int max_batch, unsigned flags, void *cuda_stream,
              l2_ctx **out) {
    g_create_error.clear();
    if (!out) return fail(nullptr, L2_EINVAL, "out is NULL");
    *out = nullptr;
    if (!config || !weights) return fail(nullptr, L2_EINVAL, "config and weights must not be NULL");
    if (max_batch < 1 || max_batch > kMaxBatch)
        return fail(nullptr, L2_EINVAL, "max_batch %d outside 1..%d", max_batch, kMaxBatch);
    if (flags & ~(L2_FLAG_DEBUG | L2_FLAG_NO_GRAPH | L2_FLAG_NO_PDL | L2_FLAG_PERSIST | L2_FLAG_NO_TC |
                  L2_FLAG_BF16_WEIGHTS | L2_FLAG_NO_ONE_CTA))
        return fail(nullptr, L2_EINVAL, "unknown flags 0x%x", flags);
    if (flags & L2_FLAG_BF16_WEIGHTS) {
        if ((flags & L2_FLAG_NO_TC) && max_batch != 1)
            return fail(nullptr, L2_EINVAL,
                        "L2_FLAG_BF16_WEIGHTS streams steps of several rows through the tensor cores: with "
                        "L2_FLAG_NO_TC it serves one sequence (max_batch 1)");
        if (flags & L2_FLAG_PERSIST) return fail(nullptr, L2_EINVAL, "L2_FLAG_BF16_WEIGHTS excludes L2_FLAG_PERSIST");
        if (config->dim % 8 || config->hidden_dim % 8)
            return fail(nullptr, L2_EINVAL, "L2_FLAG_BF16_WEIGHTS needs dim and hidden_dim divisible by 8");
    }
    int rc = check_config(*config);
    if (rc) return rc;
    rc = check_weights(*weights);
    if (rc) return rc;

    l2_ctx *c = new l2_ctx();
    c->cfg = *config;
    c->w = *weights;
    c->max_batch = max_batch;
    // Prompt chunks use up to 64 rows whatever max_batch is (the per-row
    // buffers are small); with L2_FLAG_DEBUG the per-row probability export
    // keeps them at max_batch.
    c->max_rows = (flags & L2_FLAG_DEBUG) ? max_batch : kMaxBatch;
    // bf16 weights without the tensor cores: batch-1 steps only, a prompt one token per step
    if ((flags & L2_FLAG_BF16_WEIGHTS) && (flags & L2_FLAG_NO_TC)) c->max_rows = 1;
    c->flags = flags;
    const L2Config &p = c->cfg;
    c->head_size = p.dim / p.n_heads;
    c->kv_dim = p.dim * p.n_kv_heads / p.n_heads;
    c->written.assign(max_batch, 0);

    auto bail = [&](int code) {
        g_create_error = c->error;
        free_all(c);
        delete c;
        return code;
    };
#define CREATE_CUDA(call)                                 \
    do {                                                  \
        cudaError_t e_ = (call);                          \
        if (e_ != cudaSuccess) return bail(cuda_fail(c, e_, #call)); \
    } while (0)

    CREATE_CUDA(cudaGetDevice(&c->device));
    if ((rc = static_scratch_address(c, c->device, &c->static_scratch))) return bail(rc);
    CREATE_CUDA(cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device));
    int l2_bytes = 0;
    CREATE_CUDA(cudaDeviceGetAttribute(&l2_bytes, cudaDevAttrL2CacheSize, c->device));
    c->attn = attn_plan(c->head_size, p.n_heads, p.n_kv_heads);
    if (!c->attn.ok) return bail(fail(c, L2_EINVAL, "unsupported head_size / GQA grouping"));
    CREATE_CUDA(gemv_init());
    CREATE_CUDA(gemv_batched_init());
    CREATE_CUDA(attn_init());
    c->attn_pf = !(flags & L2_FLAG_DEBUG) && attn_prefill_supported(c->head_size, p.n_heads, p.n_kv_heads);
    if (c->attn_pf) CREATE_CUDA(attn_prefill_init());
    c->attn_per_sm = attn_ctas_per_sm(c->attn);

    if (cuda_stream) {
        c->stream = static_cast<cudaStream_t>(cuda_stream);
    } else {
        CREATE_CUDA(cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking));
        c->own_stream = true;
    }
    CREATE_CUDA(cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));

    const size_t B = (size_t)c->max_rows, L = p.n_layers, S = p.seq_len, hs = c->head_size;
    const size_t cache = (size_t)max_batch * L * p.n_kv_heads * S * hs;
    c->attn_chunks = attn_chunks_for(c, 1);
    if (c->max_rows > 1 && ceil_div(p.seq_len, kMinChunk) > c->attn_chunks) c->attn_chunks = ceil_div(p.seq_len, kMinChunk);
    c->attn_chunks = std::min(c->attn_chunks, c->attn.max_chunks);
    // Steps of one row merge their attention chunks through distributed shared memory
    // when the chunks of every KV head fit one cluster and all clusters are resident.
#ifndef L2_ATTN_CLUSTER
#define L2_ATTN_CLUSTER 1
#endif
    {
        const int nc1 = std::min(attn_chunks_for(c, 1), c->attn_chunks);
        c->attn_cluster = L2_ATTN_CLUSTER && attn_cluster_fits(c->attn, nc1, p.n_kv_heads) ? nc1 : 0;
    }
    const size_t ws = B * p.n_heads * (size_t)c->attn_chunks;
    if ((rc = alloc_n(c, &c->x, B * p.dim, "x")) || (rc = alloc_n(c, &c->xb, B * p.dim, "xb")) ||
        (rc = alloc_n(c, &c->q, B * p.dim, "q")) || (rc = alloc_n(c, &c->hb, B * p.hidden_dim, "hb")) ||
        (rc = alloc_n(c, &c->logits, B * p.vocab_size, "logits")) || (rc = alloc_n(c, &c->kcache, cache, "key cache")) ||
        (rc = alloc_n(c, &c->vcache, cache, "value cache")) || (rc = alloc_n(c, &c->ws_ml, ws * 2, "attention workspace")) ||
        (rc = alloc_n(c, &c->ws_acc, ws * hs, "attention workspace")) ||
        (rc = alloc_n(c, &c->tickets, B * p.n_kv_heads, "attention tickets")) ||
        (rc = alloc_n(c, &c->rope, S * (hs / 2), "RoPE table")) || (rc = alloc_n(c, &c->step_dev, 1, "step inputs")) ||
        (rc = alloc_n(c, &c->err, 1, "error word")) ||
        (rc = alloc_n(c, &c->ss_part, (size_t)kMaxParts * B, "sum-of-squares partials")) ||
        (rc = alloc_n(c, &c->ext_dev, 1, "buffer extents")) || (rc = alloc_n(c, &c->ext_static_dev, 1, "buffer extents")))
        return bail(rc);
    if (flags & L2_FLAG_DEBUG) {
        if ((rc = alloc_n(c, &c->dbg, B * L * p.n_heads * S, "attention probabilities"))) return bail(rc);
        CREATE_CUDA(cudaMemset(c->dbg, 0, B * L * p.n_heads * S * sizeof(float)));
    }
    CREATE_CUDA(cudaMemset(c->tickets, 0, B * p.n_kv_heads * sizeof(unsigned)));
    CREATE_CUDA(cudaMemset(c->err, 0, sizeof(int)));
    CREATE_CUDA(cudaMemset(c->kcache, 0, cache * sizeof(float)));
    CREATE_CUDA(cudaMemset(c->vcache, 0, cache * sizeof(float)));
    CREATE_CUDA(cudaMemset(c->x, 0, B * p.dim * sizeof(float)));
    CREATE_CUDA(cudaMemset(c->step_dev, 0, sizeof(StepDev)));

    // RoPE table: theta = pos * 10000^(-2j/head_size) for pair j of a head,
    // evaluated in double and rounded once to fp32.
    {
        std::vector<float2> tab(S * (hs / 2));
        for (size_t t = 0; t < S; ++t)
            for (size_t j = 0; j < hs / 2; ++j) {
                const double inv_freq = std::pow(10000.0, -(double)(2 * j) / (double)hs);
                const double th = (double)t * inv_freq;
                tab[t * (hs / 2) + j] = make_float2((float)std::cos(th), (float)std::sin(th));
            }
        CREATE_CUDA(cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice));
    }
    CREATE_CUDA(cudaMallocHost(reinterpret_cast<void **>(&c->step_host), sizeof(StepDev) * kRing));
    memset(c->step_host, 0, sizeof(StepDev) * kRing);
    for (auto &e : c->ring_ev) CREATE_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));

    // Stream the weights with an evict-first L2 hint only when they cannot stay
    // resident in L2 between steps anyway.
    const double wbytes = 4.0 * ((double)L * (2.0 * p.dim * p.dim + 2.0 * c->kv_dim * p.dim + 3.0 * p.dim * p.hidden_dim) +
                                 (double)p.vocab_size * p.dim);
    c->evict_first = wbytes > 0.75 * (double)l2_bytes;
    if (flags & L2_FLAG_BF16_WEIGHTS) {
        // the handle's bf16 copies of the matrices (round to nearest even), converted once here
        const size_t L_ = p.n_layers, dd = L_ * p.dim * p.dim, kd = L_ * c->kv_dim * p.dim,
                     hd = L_ * p.hidden_dim * p.dim, cls = (size_t)p.vocab_size * p.dim;
        if ((rc = alloc_n(c, &c->w16, 2 * dd + 2 * kd + 3 * hd + cls, "bf16 weights"))) return bail(rc);
        unsigned short *at = c->w16;
        auto take = [&](const float *src, size_t n, const unsigned short *&dst) -> cudaError_t {
            dst = at;
            cudaError_t e = convert_to_bf16(src, at, n, c->stream);
            at += n;
            return e;
        };
        CREATE_CUDA(take(c->w.wq, dd, c->b16q));
        CREATE_CUDA(take(c->w.wk, kd, c->b16k));
        CREATE_CUDA(take(c->w.wv, kd, c->b16v));
        CREATE_CUDA(take(c->w.wo, dd, c->b16o));
        CREATE_CUDA(take(c->w.w1, hd, c->b16w1));
        CREATE_CUDA(take(c->w.w2, hd, c->b16w2));
        CREATE_CUDA(take(c->w.w3, hd, c->b16w3));
        CREATE_CUDA(take(c->w.wcls, cls, c->b16cls));
        CREATE_CUDA(cudaStreamSynchronize(c->stream));
        c->wt = 1;
    }
    make_plans(c);
    for (const GemvPlan *pl : {&c->plan_qkv, &c->plan_wo, &c->plan_w13, &c->plan_w2, &c->plan_cls})
        if (pl->shape < 0)
            return bail(fail(c, L2_EINVAL, "a GEMV stage needs %zu bytes of shared memory (> 227 KB); dim or hidden_dim too large",
                             pl->smem));
    if (c->attn.smem > 227 * 1024) return bail(fail(c, L2_EINVAL, "attention needs too much shared memory"));
    c->bsets.resize(c->max_rows + 1);
    // CUDA-core plans for steps of several rows (fp32 weights only: a bf16 handle's
    // steps of several rows all run on the tensor cores)
    for (int b = 2; b <= c->max_rows && !c->wt; ++b)
        if ((rc = build_batch_set(c, b))) {
            if (b <= max_batch) return bail(rc);
            c->max_rows = b - 1;  // prompt chunks stop at the widest step that could be planned
            c->error.clear();
            break;
        }
    // tensor-core plans for 16..64 rows (2..64 with bf16 weights), with one workspace and
    // ticket array for all
    const int tc_min = c->wt ? 2 : L2_TC_MIN_BATCH;
    if (!(flags & L2_FLAG_NO_TC) && c->max_rows >= tc_min) {
        CREATE_CUDA(gemv_tc_init());
        if ((rc = alloc_n(c, &c->xg, (size_t)c->max_rows * p.dim, "x * gain"))) return bail(rc);
        if (!c->wt && ((rc = alloc_n(c, &c->xg_hi, (size_t)c->max_rows * p.dim, "x * gain, tf32 hi")) ||
                       (rc = alloc_n(c, &c->xg_lo, (size_t)c->max_rows * p.dim, "x * gain, tf32 lo")) ||
                       (rc = alloc_n(c, &c->hb_hi, (size_t)c->max_rows * p.hidden_dim, "hb, tf32 hi")) ||
                       (rc = alloc_n(c, &c->hb_lo, (size_t)c->max_rows * p.hidden_dim, "hb, tf32 lo"))))
            return bail(rc);
        size_t ws = 0;
        int tiles = 0;
        for (int b = tc_min; b <= c->max_rows && b <= gemv_tc_max_batch(); ++b) {
            if ((rc = build_tc_set(c, b))) return bail(rc);
            ws = std::max(ws, c->bsets[b].tc_ws_floats);
            tiles = std::max(tiles, c->bsets[b].tc_tiles);
        }
        if (tiles > 0) {
            c->tc_ws_n = ws ? ws : 1;
            if ((rc = alloc_n(c, &c->tc_ws, c->tc_ws_n, "tensor-core GEMV workspace")) ||
                (rc = alloc_n(c, &c->tc_tickets, (size_t)tiles, "tensor-core GEMV tickets")))
                return bail(rc);
            CREATE_CUDA(cudaMemset(c->tc_tickets, 0, (size_t)tiles * sizeof(unsigned)));
            c->tc_tickets_n = (size_t)tiles;
        }
    }
    if ((rc = plan_persistent(c))) return bail(rc);
    if ((rc = plan_cta(c))) return bail(rc);
    // buffer sizes, read by the bounds-checked build only
    {
        Extents &e = c->ext;
        const size_t R = (size_t)c->max_rows;
        e.emb = (size_t)p.vocab_size * p.dim;
        e.x = e.xb = e.q = R * p.dim;
        e.hb = R * p.hidden_dim;
        e.logits = R * p.vocab_size;
        e.cache = cache;
        e.rope = S * (hs / 2);
        e.ws_rows = ws;
        e.tickets = R * p.n_kv_heads;
        e.dbg = c->dbg ? R * L * p.n_heads * S : 0;
        e.ss_part = (size_t)kMaxParts * R;
        e.xg = c->xg ? R * p.dim : 0;
        e.tc_ws = c->tc_ws_n;
        e.tc_tickets = c->tc_tickets_n;
        // l2_forward_static: its attention partials and tickets live in the static array
        c->ext_static = e;
        const AttnParams probe = attn_params(c, 0, 1);
        c->ext_static.ws_rows = (size_t)p.n_heads * probe.n_chunks;
        c->ext_static.tickets = (size_t)p.n_kv_heads;
        CREATE_CUDA(cudaMemcpy(c->ext_dev, &c->ext, sizeof(Extents), cudaMemcpyHostToDevice));
        CREATE_CUDA(cudaMemcpy(c->ext_static_dev, &c->ext_static, sizeof(Extents), cudaMemcpyHostToDevice));
    }
    CREATE_CUDA(cudaDeviceSynchronize());
#undef CREATE_CUDA
    *out = c;
    return L2_OK;
}

int l2_reset(l2_ctx *c, int slot) {
    if (!c) return L2_EINVAL;
    if (slot < -1 || slot >= c->max_batch) return fail(c, L2_EINVAL, "slot %d outside -1..%d", slot, c->max_batch - 1);
    if (slot < 0)
        for (int &w : c->written) w = 0;
    else
        c->written[slot] = 0;
    return L2_OK;
}

int l2_forward(l2_ctx *c, int token, int pos, float *logits_out) {
    if (!c) return L2_EINVAL;
    return submit(c, 1, &token, &pos, logits_out);
}

int l2_forward_batch(l2_ctx *c, int B, const int *tokens, const int *pos, float *logits_out) {
    if (!c) return L2_EINVAL;
    if (!tokens || !pos) return fail(c, L2_EINVAL, "tokens and pos must not be NULL");
    return submit(c, B, tokens, pos, logits_out);
}

int l2_prefill(l2_ctx *c, int slot, int T, const int *tokens, int pos0, float *logits_out) {
    if (!c) return L2_EINVAL;
    if (!tokens) return fail(c, L2_EINVAL, "tokens must not be NULL");
    if (slot < 0 || slot >= c->max_batch) return fail(c, L2_EINVAL, "slot %d outside 0..%d", slot, c->max_batch - 1);
    if (T < 1) return fail(c, L2_EINVAL, "T must be >= 1 (got %d)", T);
    if (pos0 < 0 || (long long)pos0 + T > c->cfg.seq_len)
        return fail(c, L2_EINVAL, "positions %d..%lld outside [0, %d)", pos0, (long long)pos0 + T - 1, c->cfg.seq_len);
    if (pos0 > c->written[slot])
        return fail(c, L2_ESTATE, "pos0 %d of slot %d skips cache rows (only %d written)", pos0, slot, c->written[slot]);
    if (logits_out && (reinterpret_cast<uintptr_t>(logits_out) & 3u))
        return fail(c, L2_EINVAL, "logits_out must be 4-byte aligned");
    for (int i = 0; i < T; ++i)
        if (tokens[i] < 0 || tokens[i] >= c->cfg.vocab_size)
            return fail(c, L2_EINVAL, "token %d at index %d outside [0, %d)", tokens[i], i, c->cfg.vocab_size);
    int pos[kMaxBatch];
    for (int i0 = 0; i0 < T; i0 += c->max_rows) {
        const int n = std::min(c->max_rows, T - i0);
        for (int b = 0; b < n; ++b) pos[b] = pos0 + i0 + b;
        const int rc = submit(c, n, tokens + i0, pos, logits_out ? logits_out + (size_t)i0 * c->cfg.vocab_size : nullptr,
                              nullptr, slot);
        if (rc) return rc;
    }
    return L2_OK;
}

int l2_forward_dev_tokens(l2_ctx *c, int B, const int *tokens_dev, const int *pos, float *logits_out) {
    if (!c) return L2_EINVAL;
    if (!tokens_dev || !pos) return fail(c, L2_EINVAL, "tokens_dev and pos must not be NULL");
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, tokens_dev) != cudaSuccess ||
        (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)) {
        cudaGetLastError();
        return fail(c, L2_EINVAL, "tokens_dev must be device memory");
    }
    return submit(c, B, nullptr, pos, logits_out, tokens_dev);
}

int l2_forward_host(l2_ctx *c, int token, int pos, float *logits_host) {
    if (!c) return L2_EINVAL;
    if (!logits_host) return fail(c, L2_EINVAL, "logits_host must not be NULL");
    int rc = submit(c, 1, &token, &pos, nullptr);
    if (rc) return rc;
    L2_CUDA(c, cudaMemcpyAsync(logits_host, c->logits, sizeof(float) * c->cfg.vocab_size, cudaMemcpyDeviceToHost,
                               c->stream));
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    return L2_OK;
}

const float *l2_logits(const l2_ctx *c) { return c ? c->logits : nullptr; }

int l2_position(const l2_ctx *c, int slot) {
    if (!c || slot < 0 || slot >= c->max_batch) return L2_EINVAL;
    return c->written[slot];
}

int l2_debug_attention(l2_ctx *c, int slot, int layer, float *att_out) {
    if (!c) return L2_EINVAL;
    if (!(c->flags & L2_FLAG_DEBUG)) return fail(c, L2_EINVAL, "created without L2_FLAG_DEBUG");
    if (slot < 0 || slot >= c->max_batch || layer < 0 || layer >= c->cfg.n_layers || !att_out)
        return fail(c, L2_EINVAL, "bad slot, layer or output pointer");
    const int n = c->written[slot];
    if (n == 0) return fail(c, L2_ESTATE, "slot %d has no step yet", slot);
    const size_t S = c->cfg.seq_len, H = c->cfg.n_heads;
    const float *src = c->dbg + (((size_t)slot * c->cfg.n_layers + layer) * H) * S;
    L2_CUDA(c, cudaMemcpy2DAsync(att_out, n * sizeof(float), src, S * sizeof(float), n * sizeof(float), H,
                                 cudaMemcpyDeviceToHost, c->stream));
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    return L2_OK;
}

int l2_kv_export(l2_ctx *c, int slot, int layer, int n_pos, float *k_out, float *v_out) {
    if (!c) return L2_EINVAL;
    if (slot < 0 || slot >= c->max_batch || layer < 0 || layer >= c->cfg.n_layers || !k_out || !v_out)
        return fail(c, L2_EINVAL, "bad slot, layer or output pointer");
    if (n_pos < 0 || n_pos > c->written[slot]) return fail(c, L2_ESTATE, "only %d rows written", c->written[slot]);
    if (n_pos == 0) return L2_OK;
    const size_t S = c->cfg.seq_len, hs = c->head_size, KV = c->cfg.n_kv_heads;
    for (size_t g = 0; g < KV; ++g) {
        const size_t off = (((size_t)slot * c->cfg.n_layers + layer) * KV + g) * S * hs;
        L2_CUDA(c, cudaMemcpy2DAsync(k_out + g * hs, c->kv_dim * sizeof(float), c->kcache + off, hs * sizeof(float),
                                     hs * sizeof(float), n_pos, cudaMemcpyDeviceToHost, c->stream));
        L2_CUDA(c, cudaMemcpy2DAsync(v_out + g * hs, c->kv_dim * sizeof(float), c->vcache + off, hs * sizeof(float),
                                     hs * sizeof(float), n_pos, cudaMemcpyDeviceToHost, c->stream));
    }
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    return L2_OK;
}

int l2_kv_import(l2_ctx *c, int slot, int n_pos, const float *k_in, const float *v_in) {
    if (!c) return L2_EINVAL;
    if (slot < 0 || slot >= c->max_batch || !k_in || !v_in) return fail(c, L2_EINVAL, "bad slot or input pointer");
    if (n_pos < 0 || n_pos > c->cfg.seq_len) return fail(c, L2_EINVAL, "n_pos %d outside 0..seq_len", n_pos);
    const size_t S = c->cfg.seq_len, hs = c->head_size, KV = c->cfg.n_kv_heads, L = c->cfg.n_layers;
    for (size_t l = 0; l < L && n_pos > 0; ++l)
        for (size_t g = 0; g < KV; ++g) {
            const size_t off = (((size_t)slot * L + l) * KV + g) * S * hs;
            const size_t src = l * (size_t)n_pos * c->kv_dim + g * hs;
            L2_CUDA(c, cudaMemcpy2DAsync(c->kcache + off, hs * sizeof(float), k_in + src, c->kv_dim * sizeof(float),
                                         hs * sizeof(float), n_pos, cudaMemcpyHostToDevice, c->stream));
            L2_CUDA(c, cudaMemcpy2DAsync(c->vcache + off, hs * sizeof(float), v_in + src, c->kv_dim * sizeof(float),
                                         hs * sizeof(float), n_pos, cudaMemcpyHostToDevice, c->stream));
        }
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    c->written[slot] = n_pos;
    return L2_OK;
}

int l2_sync(l2_ctx *c) {
    if (!c) return L2_EINVAL;
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    int word = 0;
    L2_CUDA(c, cudaMemcpy(&word, c->err, sizeof(int), cudaMemcpyDeviceToHost));
    if (word) {
        // A kernel that gave up may have left a ticket counted (the tensor-core
        // GEMV's CTAs take theirs only after their last tile): start the next
        // step from zero.
        L2_CUDA(c, cudaMemset(c->tickets, 0, (size_t)c->max_rows * c->cfg.n_kv_heads * sizeof(unsigned)));
        if (c->tc_tickets) L2_CUDA(c, cudaMemset(c->tc_tickets, 0, c->tc_tickets_n * sizeof(unsigned)));
        L2_CUDA(c, cudaMemset(c->err, 0, sizeof(int)));
        if (word & L2_DEV_ERR_TIMEOUT) return fail(c, L2_ETIMEOUT, "a device-side wait gave up (error word 0x%x)", word);
        return fail(c, L2_EDEVICE, "a kernel reported an error (error word 0x%x)", word);
    }
    return L2_OK;
}

const char *l2_last_error(const l2_ctx *c) { return c ? c->error.c_str() : g_create_error.c_str(); }

void l2_destroy(l2_ctx *c) {
    if (!c) return;
    free_all(c);
    delete c;
}

int l2_launch_op(l2_ctx *c, int op, int layer, int count) { return l2_launch_op_batch(c, op, layer, 1, count); }

int l2_launch_op_batch(l2_ctx *c, int op, int layer, int batch, int count) {
    if (!c) return L2_EINVAL;
    if (op < 0 || op > 5 || layer < 0 || layer >= c->cfg.n_layers || count < 0)
        return fail(c, L2_EINVAL, "bad op, layer or count");
    if (batch < 1 || batch > c->max_rows) return fail(c, L2_EINVAL, "batch %d outside 1..%d", batch, c->max_rows);
    if (c->written[0] == 0) return fail(c, L2_ESTATE, "run a step first");
    if (batch > 1 && batch != c->last_rows)
        return fail(c, L2_ESTATE, "the last step had %d rows: run a step of %d rows first", c->last_rows, batch);
    // Standalone launches write the classifier's output only to the handle's buffer.
    L2_CUDA(c, cudaMemsetAsync(reinterpret_cast<char *>(c->step_dev) + offsetof(StepDev, logits_out), 0,
                               sizeof(float *), c->stream));
    // as in the step: consecutive launches linked by programmatic dependent launch
    // unless the handle was created with L2_FLAG_NO_PDL
    const bool pdl = !(c->flags & L2_FLAG_NO_PDL);
    for (int i = 0; i < count; ++i)
        L2_CUDA(c, launch_op(c, op, layer, batch, c->stream, pdl, batch > 1 && c->last_prefill));
    return L2_OK;
}

int l2_sample(const float *logits, int B, int vocab_size, float temperature, float topp,
              unsigned long long *rng_state, int *tokens_out, void *cuda_stream) {
    if (!logits || !rng_state || !tokens_out) return fail(nullptr, L2_EINVAL, "l2_sample: NULL pointer");
    if (B < 1 || B > 65535) return fail(nullptr, L2_EINVAL, "l2_sample: B = %d outside 1..65535", B);
    if (vocab_size < 1 || vocab_size > sample_max_vocab())
        return fail(nullptr, L2_EINVAL, "l2_sample: vocab_size %d outside 1..%d", vocab_size, sample_max_vocab());
    if (!(temperature >= 0.0f) || !std::isfinite(temperature))
        return fail(nullptr, L2_EINVAL, "l2_sample: temperature must be finite and >= 0");
    if (!std::isfinite(topp)) return fail(nullptr, L2_EINVAL, "l2_sample: topp must be finite");
    if (reinterpret_cast<uintptr_t>(logits) & 3u) return fail(nullptr, L2_EINVAL, "l2_sample: logits not 4-byte aligned");
    for (const void *ptr : {(const void *)logits, (const void *)rng_state, (const void *)tokens_out}) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess ||
            (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged)) {
            cudaGetLastError();
            return fail(nullptr, L2_EINVAL, "l2_sample: pointers must be device memory");
        }
    }
    cudaError_t e = sample_init();
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "sample_init()");
    SampleParams sp{};
    sp.logits = logits;
    sp.rng = rng_state;
    sp.out = tokens_out;
    sp.vocab = vocab_size;
    sp.temperature = temperature;
    sp.topp = topp;
    e = launch_sample(sp, B, static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "sample launch");
    return L2_OK;
}

int l2_kernels_per_step(const l2_ctx *c, int B) {
    if (!c || B < 1 || B > c->max_batch) return L2_EINVAL;
    if (B == 1 && (c->cta || c->persist)) return 1;
    return 5 * c->cfg.n_layers + 1 + (B > 1 && c->bsets[B].tc ? 1 : 0);
}

int l2_step_input_bytes(void) { return (int)sizeof(StepDev); }

void l2_debug_fail_alloc_at(int n) { g_fail_alloc_at = n > 0 ? n : 0; }

void l2_debug_fail_graph_at(int n) { g_fail_graph_at = n > 0 ? n : 0; }

int l2_debug_bounds_checked(void) { return L2_DEBUG_BOUNDS ? 1 : 0; }

int l2_debug_limit_cache(l2_ctx *c, unsigned long long floats) {
    if (!c) return L2_EINVAL;
    L2_CUDA(c, cudaStreamSynchronize(c->stream));
    c->ext.cache = std::min<size_t>(c->ext.cache, (size_t)floats);
    c->ext_static.cache = c->ext.cache;
    L2_CUDA(c, cudaMemcpy(c->ext_dev, &c->ext, sizeof(Extents), cudaMemcpyHostToDevice));
    L2_CUDA(c, cudaMemcpy(c->ext_static_dev, &c->ext_static, sizeof(Extents), cudaMemcpyHostToDevice));
    return L2_OK;
}

int l2_debug_wait_timeout(l2_ctx *c, int limit_us) {
    if (!c) return L2_EINVAL;
    if (limit_us < 1 || (unsigned long long)limit_us * 1000ull > kWaitLimitNs)
        return fail(c, L2_EINVAL, "limit_us %d outside 1..%llu", limit_us, kWaitLimitNs / 1000ull);
    // dim is a multiple of 4, so this is a multiple of 16 bytes, at most the kernel's buffer
    const uint32_t bytes = (uint32_t)std::min<size_t>(128, (size_t)c->cfg.dim * sizeof(float));
    debug_wait_kernel<<<1, 32, 0, c->stream>>>(c->x, bytes, c->err, c->tickets, c->max_rows * c->cfg.n_kv_heads,
                                               (unsigned long long)limit_us * 1000ull);
    L2_CUDA(c, cudaGetLastError());
    return L2_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// l2_forward_static: the decode step with nothing allocated on its path, for
// callers that cannot call cudaMalloc once decoding has started (a serving
// process that handed all device memory to its own pool at start-up, or a
// latency-critical loop that must not hit the implicit device synchronisation
// an allocation or free may cause).  l2_forward may build a CUDA graph on its
// first call for a batch size, which allocates; this entry point launches the
// kernels one by one instead, and gives the one kernel that needs scratch
// memory -- attention, for its cross-CTA partial results and tickets -- a
// static device array in place of the handle's workspace.

extern "C" int l2_forward_static(l2_ctx *c, int token, int pos, float *logits_out) {
    if (!c) return L2_EINVAL;
    int dev = -1;
    L2_CUDA(c, cudaGetDevice(&dev));
    if (dev != c->device) return fail(c, L2_EINVAL, "the handle's device (%d) must be current (is %d)", c->device, dev);
    if (token < 0 || token >= c->cfg.vocab_size)
        return fail(c, L2_EINVAL, "token %d outside [0, %d)", token, c->cfg.vocab_size);
    if (pos < 0 || pos >= c->cfg.seq_len) return fail(c, L2_EINVAL, "pos %d outside [0, %d)", pos, c->cfg.seq_len);
    if (pos > c->written[0]) return fail(c, L2_ESTATE, "pos %d skips cache rows (only %d written)", pos, c->written[0]);
    if (logits_out && (reinterpret_cast<uintptr_t>(logits_out) & 3u))
        return fail(c, L2_EINVAL, "logits_out must be 4-byte aligned");

    // Scratch layout: accumulators [n_heads][n_chunks][head_size] (16-byte
    // aligned), then (max, sum) pairs [n_heads][n_chunks][2], then one ticket
    // per KV head.
    const AttnParams probe = attn_params(c, 0, 1);
    const size_t slots = (size_t)c->cfg.n_heads * probe.n_chunks;
    const size_t acc_f = slots * c->head_size, ml_f = slots * 2, tick_f = (size_t)c->cfg.n_kv_heads;
    const size_t need = acc_f + ml_f + tick_f;
    if (need > kStaticScratchFloats)
        return fail(c, L2_EINVAL,
                    "attention needs %zu floats of scratch; l2_forward_static has a static array of %zu floats",
                    need, kStaticScratchFloats);
    float *scratch = c->static_scratch;  // looked up by l2_create on this device
    float *ws_acc = scratch, *ws_ml = scratch + acc_f;
    unsigned *tickets = reinterpret_cast<unsigned *>(scratch + acc_f + ml_f);

    const int i = c->ring_next;
    c->ring_next = (i + 1) % kRing;
    if (c->ring_used[i]) L2_CUDA(c, cudaEventSynchronize(c->ring_ev[i]));
    StepDev &sh = c->step_host[i];
    sh.token[0] = token;
    sh.pos[0] = pos;
    sh.slot[0] = 0;
    sh.stable[0] = pos;
    sh.logits_out = logits_out;
    sh.B = 1;
    L2_CUDA(c, cudaMemcpyAsync(c->step_dev, &sh, sizeof(StepDev), cudaMemcpyHostToDevice, c->stream));
    L2_CUDA(c, cudaEventRecord(c->ring_ev[i], c->stream));
    c->ring_used[i] = true;
    // The array keeps the previous call's contents: the tickets must start at zero.
    L2_CUDA(c, cudaMemsetAsync(tickets, 0, tick_f * sizeof(unsigned), c->stream));

    const bool pdl = !(c->flags & L2_FLAG_NO_PDL);
    for (int l = 0; l < c->cfg.n_layers; ++l) {
        L2_CUDA(c, launch_op(c, 0, l, 1, c->stream, pdl));
        AttnParams a = attn_params(c, l, 1);
        a.ws_acc = ws_acc;
        a.ws_ml = ws_ml;
        a.tickets = tickets;
        a.ext = c->ext_static_dev;
        L2_CUDA(c, launch_attn(c->attn, a, 1, c->stream, pdl));
        for (int op = 2; op < 5; ++op) L2_CUDA(c, launch_op(c, op, l, 1, c->stream, pdl));
    }
    L2_CUDA(c, launch_op(c, 5, 0, 1, c->stream, pdl));
    c->written[0] = pos + 1;
    return L2_OK;
}
