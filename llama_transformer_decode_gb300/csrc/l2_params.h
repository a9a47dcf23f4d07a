// Kernel parameter blocks shared by the host orchestrator and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace l2 {

constexpr int kMaxBatch = 64;
// A bounded device-side wait gives up after this much wall time.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// Bits of the device error word.
enum : int { L2_DEV_ERR_TIMEOUT = 1, L2_DEV_ERR_BOUNDS = 2 };

// Element counts of the buffers the kernels index, for the bounds-checked build
// (compiled with L2_DEBUG_BOUNDS=1): there every computed index into these buffers
// and every bulk-copy source range is checked, a violation sets
// L2_DEV_ERR_BOUNDS in the error word and the access is skipped.  A device copy
// lives with the handle; the release build never reads it.
struct Extents {
    size_t emb;              // token embedding table
    size_t x, xb, q, hb;     // activations (rows x width)
    size_t logits;           // the handle's logits buffer
    size_t cache;            // each of the K and V caches
    size_t rope;             // RoPE table entries (cos, sin pairs)
    size_t ws_rows;          // attention partials: (m, l) pairs and head_size-wide accumulators
    size_t tickets;          // attention tickets
    size_t dbg;              // probability export (0: none)
    size_t ss_part, xg;      // batched steps: sums-of-squares partials, x * gain
    size_t tc_ws, tc_tickets;  // tensor-core GEMV: partial tiles, tickets
};

// Per-step inputs, filled by one host->device copy before each step.
struct StepDev {
    int token[kMaxBatch];
    int pos[kMaxBatch];
    int slot[kMaxBatch];    // KV-cache slot row b reads and writes (b for ordinary steps)
    int stable[kMaxBatch];  // rows of that slot written before this step (pos[b] for
                            // ordinary steps; the first position of a prefill chunk)
    float *logits_out;  // caller's device buffer [B][vocab] or nullptr
    int B;
    unsigned sync_count;  // grid-barrier arrivals of the persistent step kernel (zero at the copy)
    // Steps of several rows (attn_chunk_plan, on the host): attention CTAs per KV head
    // for row b, and the order in which the attention grid takes the rows (most
    // positions per CTA first, so the longest CTAs start in the first wave).
    unsigned short nchunk[kMaxBatch];
    unsigned char row_order[kMaxBatch];
};

// The fused GEMV kernel's modes (prologue / epilogue around y = W v).
enum GemvMode : int {
    GEMV_QKV = 0,    // v = rmsnorm(x); rows of Wq|Wk|Wv; RoPE; q out, K/V rows into the cache
    GEMV_RESID = 1,  // v = an activation vector; x += y
    GEMV_W13 = 2,    // v = rmsnorm(x); rows of W1 and W3; hb = silu(h1) * h3
    GEMV_CLS = 3,    // v = rmsnorm(x); logits = y
};

struct GemvParams {
    int n;            // row length = input vector length
    int unit_rows;    // rows per unit of the CTA split (2 keeps RoPE pairs together)
    int total_units;  // units split evenly across the grid
    int layer;
    const float *mat0, *mat1, *mat2;  // this layer's matrices, row-major [rows][n]
    int rows0, rows1, rows2;
    const float *in_vec;  // GEMV_RESID input (xb or hb), [B][n]
    const float *norm_w;  // rmsnorm gain [n]
    const float *emb;     // embedding table (layer-0 QKV reads x from it)
    float *x;             // residual stream [B][dim]
    float *q;             // [B][dim]
    float *kcache, *vcache;  // [slot][layer][kv_head][seq_len][head_size]
    const float2 *rope;      // [seq_len][head_size/2] (cos, sin)
    float *hb;               // [B][hidden_dim]
    float *logits;           // handle's logits buffer [B][vocab]
    const StepDev *step;
    int *err;
    int dim, kv_dim, head_size, seq_len, n_kv_heads, n_layers, vocab;
    int evict_first;  // stream the weights with an L2 evict-first hint
    const Extents *ext;  // buffer sizes (read only by the bounds-checked build)
    // Batched steps (l2dec_matvec_batched_kernel) only:
    int batch;        // sequences in the step (slots 0..batch-1)
    float *ss_part;   // [kMaxParts][batch] partial sums of x^2 written by the residual kernels
    int ss_parts;     // rows of ss_part the RMSNorm modes add up (grid of the residual kernels)
};

constexpr int kMaxParts = 1024;

// Batched GEMV launch (gemv_batched.cu): tensor maps for 2-D tile copies of
// the weights (rows x columns boxes) and of the B input rows.
struct alignas(128) BatchParams {
    CUtensorMap wmap[3];  // QKV: Wq, Wk, Wv; W1/W3: W1, W3; otherwise [0]
    CUtensorMap xmap;     // input activations [slots][n], box = tk columns x batch rows
    GemvParams g;
    int part_ctas[3];     // CTAs per matrix (QKV), or [0] = grid
    int part_units[3];    // units per matrix
    int rows_box;         // rows per weight box = rows per block (a CTA walks its rows in blocks)
    int tk;               // columns per K tile
    int stages;           // ring depth
};

// Persistent step kernel (step_kernel.cu, batch 1): everything one step
// reads and writes.  Weights are the model's base pointers (layer l of a
// per-layer tensor starts l * its per-layer size further on).
struct StepKParams {
    const float *emb, *rms_att, *rms_ffn, *rms_final;
    const float *wq, *wk, *wv, *wo, *w1, *w2, *w3, *wcls;
    float *x, *xb, *q, *hb, *logits;
    float *kcache, *vcache;   // slot 0: [layer][kv_head][seq_len][head_size]
    const float2 *rope;
    float *ws_ml, *ws_acc;    // attention partials [n_heads][n_chunks][2] / [..][head_size]
    unsigned *tickets;        // [n_kv_heads], zero between steps
    StepDev *step;
    int *err;
    int dim, hidden_dim, n_layers, n_heads, n_kv_heads, head_size, kv_dim, vocab, seq_len;
    int n_chunks;    // most attention CTAs per KV head (n_chunks * n_kv_heads <= grid)
    int min_chunk;   // fewest cache positions per attention CTA
    int lp;          // lanes per cache row (power of two >= head_size / 4)
    int xs_floats;   // shared input-vector region (largest row length)
    int ys_floats;   // shared output region (most outputs one CTA produces in a phase)
    int evict_first;
    int stages;      // ring buffers per warp (<= 4)
    int ch4;         // 16-byte words per ring buffer (a multiple of 8)
    float scale;     // 1 / sqrt(head_size)
};

// Whole batch-1 step of a small model in one CTA (step_cta.cu): the model's
// base pointers (layer l of a per-layer tensor starts l * its per-layer size
// further on) and the handle's buffers for slot 0.
struct CtaStepParams {
    const float *emb, *rms_att, *rms_ffn, *rms_final;
    const float *wq, *wk, *wv, *wo, *w1, *w2, *w3, *wcls;
    float *x;                 // residual stream [dim], left as the step ends it
    float *logits;            // handle's logits buffer [vocab]
    float *kcache, *vcache;   // slot 0: [layer][kv_head][seq_len][head_size]
    const float2 *rope;       // [seq_len][head_size/2] (cos, sin)
    float *dbg;               // [n_layers][n_heads][seq_len] probabilities (slot 0), or nullptr
    const StepDev *step;
    int *err;
    const Extents *ext;       // buffer sizes (read only by the bounds-checked build)
    int dim, hidden_dim, n_layers, n_heads, n_kv_heads, head_size, kv_dim, vocab, seq_len;
    float scale;              // 1 / sqrt(head_size)
};

// Token sampler (sample.cu): one CTA per sequence.
struct SampleParams {
    const float *logits;       // [B][vocab]
    unsigned long long *rng;   // [B] xorshift* states, advanced by one draw when temperature > 0
    int *out;                  // [B] sampled token ids
    int vocab;
    float temperature;         // 0: argmax
    float topp;                // in (0, 1): nucleus sampling; otherwise none
    int cand_cap;              // top-p candidate list capacity (set at launch)
};

// Tensor-core batched GEMV (gemv_tc.cu): output tiles of 128 rows (64 rows
// of W1 over the same 64 rows of W3) x bpad sequences, the (tile, K stage)
// work split evenly over the grid; tensor maps with 128-byte swizzle, boxes of
// 32 columns.
struct alignas(128) TcParams {
    CUtensorMap wmap[3];  // QKV: Wq, Wk, Wv; W1/W3: W1, W3; otherwise [0]
    CUtensorMap xmap;     // inputs [max rows][n] (x * gain for the RMSNorm modes), box 32 columns x bpad rows
    GemvParams g;
    int tiles[3];         // output tiles per matrix (QKV), or [0]
    int mrows[3];         // rows of each matrix in one layer
    int ntiles;           // all tiles
    int bpad;             // sequences rounded up to a multiple of 16 (MMA N)
    int wt;               // weights: 0 fp32 (3xTF32 products), 1 bf16 (kind::f16, inputs in three bf16 parts)
    int stages;           // ring stages for this width
    // > 1: each tile's K range is split over a thread-block cluster of csplit CTAs
    // (grid ntiles * csplit) whose parts are added through distributed shared
    // memory; 0: the stream-K split with the workspace and tickets below.
    int csplit;
    float *ws;            // partial tiles [grid][2][bpad][128]
    unsigned *tickets;    // [ntiles], zero between launches
    float *xg;            // x * gain of the next RMSNorm [max rows][dim], written by the residual kernels
    const float *next_gain;  // residual kernels: the gain vector of the next RMSNorm
    // fp32 weights: the inputs' tf32 split made once by the kernel that writes them
    // (hi = the tf32 value nearest to v, lo = the tf32 value nearest to v - hi) instead of
    // by every CTA for every tile.  xsplit: this launch's inputs come as xmap (hi) and
    // xmap_lo (lo); xg_hi/xg_lo (residual and embedding kernels) and hb_hi/hb_lo (W1/W3)
    // receive the split of what they write, or are null.
    CUtensorMap xmap_lo;
    int xsplit;
    float *xg_hi, *xg_lo;  // [max rows][dim]
    float *hb_hi, *hb_lo;  // [max rows][hidden_dim]
};

struct AttnParams {
    const float *q;                  // [B][dim]
    const float *kcache, *vcache;    // [slot][layer][kv_head][seq_len][head_size]
    float *out;                      // [B][dim]
    float *ws_ml;                    // [B][n_heads][n_chunks][2] (running max, sum)
    float *ws_acc;                   // [B][n_heads][n_chunks][head_size]
    unsigned *tickets;               // [B][n_kv_heads], zero between launches
    float *dbg;                      // [B][n_layers][n_heads][seq_len] scores -> probabilities, or nullptr
    const StepDev *step;
    int *err;
    int layer, n_layers, n_heads, n_kv_heads, head_size, seq_len, dim;
    int n_chunks;   // grid.x: CTAs per (slot, KV head)
    int min_chunk;  // fewest positions a CTA takes before more CTAs join
    int capacity;   // batches: CTAs resident at once; the chunk grows so the
                    // positions of all slots fill about that many (0: fixed chunk)
    int cluster;    // > 1: the n_chunks CTAs of a (row, KV head) form one thread-block
                    // cluster and merge their chunks through distributed shared memory
    float scale;    // 1 / sqrt(head_size)
    const Extents *ext;  // buffer sizes (read only by the bounds-checked build)
};

}  // namespace l2
