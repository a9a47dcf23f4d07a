/*
 * l2decode -- single-token Llama-2 decode step on one GB300 (sm_103a), fp32.
 *
 * The operation is llama2.c's forward(token, pos) -> logits, as stated by
 * the page "run.c" (play_with_baby_llama2 mirror of llama2.c), function
 * transformer(), and by the page "run.c 逐行解讀" (line-by-line walkthrough
 * of the later run.c), §4 forward() steps 1-3:
 *   x = emb[token];
 *   per layer l: xb = rmsnorm(x, rms_att[l]); q = Wq xb; k = Wk xb; v = Wv xb;
 *     RoPE(q over dim, k over kv_dim; theta = pos*10000^(-(i mod hs)/hs));
 *     K[l][pos] = k; V[l][pos] = v;
 *     per query head h with KV head g(h): softmax(q_h.K_t/sqrt(hs), t<=pos)
 *       weighted sum of V_t -> xb;
 *     x += Wo xb; xb = rmsnorm(x, rms_ffn[l]);
 *     x += W2 (silu(W1 xb) * (W3 xb));
 *   logits = Wcls rmsnorm(x, rms_final).
 * g(h) = floor(h * n_kv_heads / n_heads), which is the pages' h / kv_mul
 * whenever n_heads is a multiple of n_kv_heads.
 *
 * Conventions for every entry point:
 *   - Calls return an L2_* status; they never exit or abort the process.
 *     After a failure, l2_last_error() describes it.
 *   - Device pointers are borrowed: the caller keeps them alive and
 *     unchanged until l2_destroy().  The handle owns everything it
 *     allocates (KV cache, activations, workspaces, CUDA graphs, pinned
 *     staging) and frees it in l2_destroy().
 *   - Work is enqueued on the stream given to l2_create() and the call
 *     returns without waiting, except where a function says it blocks.
 *   - One handle must not be used from two host threads at once.
 */
#ifndef L2_DECODE_H
#define L2_DECODE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define L2_OK 0
#define L2_EINVAL (-1)   /* invalid argument (config, pointer, token, pos, batch, slot) */
#define L2_ESTATE (-2)   /* KV-cache precondition violated: pos beyond the written rows */
#define L2_ENOMEM (-3)   /* a device or pinned allocation failed */
#define L2_ECUDA (-4)    /* a CUDA runtime call failed */
#define L2_EDEVICE (-5)  /* a kernel reported an error through the device error word */
#define L2_ETIMEOUT (-6) /* a bounded device-side wait gave up */

/* l2_create flags. */
#define L2_FLAG_DEBUG 0x1u    /* keep per-layer attention probabilities (l2_debug_attention) */
#define L2_FLAG_NO_GRAPH 0x2u /* launch the step's kernels one by one instead of a CUDA graph */
#define L2_FLAG_NO_PDL 0x4u   /* no programmatic dependent launch between the step's kernels */
/* Run batch-1 steps as ONE persistent cooperative kernel (one CTA per SM,
 * grid-wide barriers between the phases of a layer) instead of one kernel
 * per matmul group and one attention kernel per layer.  Used when the device
 * supports cooperative launch and the shape fits (l2_kernels_per_step then
 * reports 1); ignored with L2_FLAG_DEBUG.  Measured on GB300 it is slower
 * than the default graph of kernels with programmatic dependent launch. */
#define L2_FLAG_PERSIST 0x8u
/* Batched steps and prompt chunks of 16 or more rows normally run their
 * matrix products on the tensor cores (tf32 with the 3-way split hi*hi +
 * hi*lo + lo*hi, fp32-level accuracy); with this flag they stay on the CUDA
 * cores. */
#define L2_FLAG_NO_TC 0x10u
/* Reduced-precision weight streaming: the handle converts the weight
 * matrices (Wq, Wk, Wv, Wo, W1, W2, W3, Wcls) once to bf16 (round to nearest
 * even) in its own device memory, and each step streams those -- half the
 * bytes of fp32.  Products and sums stay fp32 (each bf16 weight widens
 * exactly), as do the embedding table, the RMSNorm gains, activations and the
 * KV cache; the results are those of the model with bf16-rounded matrices.
 * Steps of one row read the bf16 words on the CUDA cores; batched steps and
 * prompt chunks of 16 or more rows multiply them on the tensor cores
 * (kind::f16, each fp32 input split exactly into three bf16 parts).  With
 * L2_FLAG_NO_TC max_batch must be 1 (else L2_EINVAL) and prompts are fed one
 * token per step; L2_FLAG_PERSIST is refused; dim and hidden_dim must be
 * divisible by 8. */
#define L2_FLAG_BF16_WEIGHTS 0x20u
/* Batch-1 steps of a model whose weights take at most 4 MiB (they stay in L2,
 * so a step of one kernel per matrix product costs its kernel boundaries, not
 * its bytes) normally run as ONE kernel of one thread block that does every
 * phase of the step with block-wide barriers between them (l2_kernels_per_step
 * then reports 1; with L2_FLAG_DEBUG it exports the probabilities too).  This
 * flag keeps such models on the graph of per-matrix kernels.  Larger models,
 * L2_FLAG_PERSIST and L2_FLAG_BF16_WEIGHTS always use the other paths. */
#define L2_FLAG_NO_ONE_CTA 0x40u

/* Model shape: the pages' Config struct ("run.c", Config; walkthrough §2).
 * head_size = dim / n_heads, kv_dim = dim * n_kv_heads / n_heads. */
typedef struct {
    int dim;        /* transformer width */
    int hidden_dim; /* FFN width */
    int n_layers;
    int n_heads;    /* query heads */
    int n_kv_heads; /* key/value heads, 1 <= n_kv_heads <= n_heads */
    int vocab_size;
    int seq_len;    /* KV-cache capacity in positions */
} L2Config;

/* Weights: the pages' TransformerWeights (walkthrough §2), fp32, row-major
 * [out][in], layers stacked first.  All are DEVICE pointers, 16-byte
 * aligned.  wcls may equal token_embedding_table (a shared classifier). */
typedef struct {
    const float *token_embedding_table; /* [vocab_size][dim] */
    const float *rms_att_weight;        /* [n_layers][dim] */
    const float *rms_ffn_weight;        /* [n_layers][dim] */
    const float *wq;                    /* [n_layers][dim][dim] */
    const float *wk;                    /* [n_layers][kv_dim][dim] */
    const float *wv;                    /* [n_layers][kv_dim][dim] */
    const float *wo;                    /* [n_layers][dim][dim] */
    const float *w1;                    /* [n_layers][hidden_dim][dim] */
    const float *w2;                    /* [n_layers][dim][hidden_dim] */
    const float *w3;                    /* [n_layers][hidden_dim][dim] */
    const float *rms_final_weight;      /* [dim] */
    const float *wcls;                  /* [vocab_size][dim] */
} L2Weights;

typedef struct l2_ctx l2_ctx;

/*
 * Creates a decoder on the current CUDA device.  max_batch (1..64) is the
 * number of independent sequences ("slots"), each with its own KV cache of
 * seq_len positions.  cuda_stream is a cudaStream_t (NULL: the library
 * creates its own stream).  The shape limits of this implementation, on top
 * of the pages' own (dim % n_heads == 0, even head_size): dim, hidden_dim and
 * head_size are multiples of 4, head_size <= 128, and at most 8 query heads
 * share one KV head.  Blocks while it allocates and uploads the RoPE table.
 * Returns L2_EINVAL, L2_ENOMEM or L2_ECUDA on failure (then *out is NULL).
 */
int l2_create(const L2Config *config, const L2Weights *weights, int max_batch, unsigned flags,
              void *cuda_stream, l2_ctx **out);

/* Rewinds the KV cache of one slot (-1: all slots) to zero written rows.
 * The cache is the pages' key_cache / value_cache of the run state, one per
 * slot ("run.c 逐行解讀" §3 memory management, malloc_run_state: n_layers x
 * seq_len x kv_dim floats each; "run.c", RunState and malloc_run_state), which
 * forward() fills one row per position; rewinding starts a new sequence at
 * position 0 without clearing memory (rows are always written before they
 * are read).  Host bookkeeping only; no device work.  L2_EINVAL on a bad slot. */
int l2_reset(l2_ctx *ctx, int slot);

/*
 * One decode step of slot 0: enqueues forward(token, pos) ("run.c 逐行解讀"
 * §4 forward(), steps 1-3; "run.c", transformer(token, pos, ...)) and writes
 * the vocab_size logits to logits_out (a DEVICE pointer, or NULL to keep them
 * only in the handle's buffer, see l2_logits).  Preconditions checked on
 * the host: 0 <= token < vocab_size, 0 <= pos < seq_len, and pos <= the
 * number of rows already written to the slot's cache (rows 0..pos-1 must
 * exist).  After the call the slot holds rows 0..pos; rows beyond pos are
 * stale.  L2_EINVAL / L2_ESTATE on a failed check (nothing enqueued).
 */
int l2_forward(l2_ctx *ctx, int token, int pos, float *logits_out);

/*
 * One decode step of slots 0..B-1 at once (1 <= B <= max_batch).  tokens and
 * pos are HOST arrays of B entries; slot b steps tokens[b] at pos[b] under the
 * same checks as l2_forward.  logits_out is a DEVICE array [B][vocab_size]
 * or NULL.  Every weight is read once per call for all B sequences.
 */
int l2_forward_batch(l2_ctx *ctx, int B, const int *tokens, const int *pos, float *logits_out);

/* l2_forward for callers without device buffers: logits_host is HOST memory
 * (vocab_size floats).  Blocks until the logits have arrived. */
int l2_forward_host(l2_ctx *ctx, int token, int pos, float *logits_host);

/* Device pointer to the handle's logits buffer [max_batch][vocab_size],
 * holding the last step's logits.  NULL on a bad handle. */
const float *l2_logits(const l2_ctx *ctx);

/* Number of cache rows written for a slot (the next pos it may step), or
 * L2_EINVAL.  forward() at pos reads rows 0..pos of the layer's cache and
 * writes row pos ("run.c 逐行解讀" §4 forward() step 2e and the K/V write
 * into key_cache / value_cache), so pos may not exceed this count. */
int l2_position(const l2_ctx *ctx, int slot);

/*
 * Attention probabilities of the last step of `slot` at `layer`: the
 * softmax outputs (not the scores) as a HOST array [n_heads][pos+1], where
 * pos is that step's position.  Needs L2_FLAG_DEBUG.  Blocks.
 */
int l2_debug_attention(l2_ctx *ctx, int slot, int layer, float *att_out);

/*
 * KV-cache transfer in the pages' layout ([pos][kv_dim] per layer; K after
 * RoPE).  Both block.
 * l2_kv_export copies rows 0..n_pos-1 of one layer of a slot into HOST
 * arrays k_out, v_out [n_pos][kv_dim]; n_pos <= l2_position(slot).
 * l2_kv_import writes HOST arrays k_in, v_in [n_layers][n_pos][kv_dim] into
 * rows 0..n_pos-1 of every layer of a slot and sets its position to n_pos.
 */
int l2_kv_export(l2_ctx *ctx, int slot, int layer, int n_pos, float *k_out, float *v_out);
int l2_kv_import(l2_ctx *ctx, int slot, int n_pos, const float *k_in, const float *v_in);

/* Waits for the handle's stream and reports asynchronous failures:
 * L2_ECUDA for a CUDA error, L2_EDEVICE / L2_ETIMEOUT for a kernel that set
 * the device error word (the word is cleared, and so are the attention and
 * tensor-core tickets, which a kernel that gave up may have left counted).
 * Blocks.  The pages have no asynchronous work and so no counterpart; their
 * failures end the process ("run.c", malloc_run_state: exit(1) after a failed
 * calloc), which this library never does. */
int l2_sync(l2_ctx *ctx);

/* Text of the last failure on this handle ("" if none).  With a NULL
 * handle, the last failure of l2_create on this thread. */
const char *l2_last_error(const l2_ctx *ctx);

/* Frees everything the handle owns (the pages' free_run_state: "run.c",
 * the activations, logits and the KV cache).  Waits for its stream first. */
void l2_destroy(l2_ctx *ctx);

/*
 * Profiling hook: enqueues `count` launches of one kernel of the step,
 * exactly as the step launches it (consecutive launches linked by
 * programmatic dependent launch, as the step's kernels are, unless the handle
 * has L2_FLAG_NO_PDL), for timing it alone.  op: 0 = fused
 * rmsnorm+QKV+RoPE+KV write, 1 = attention, 2 = Wo+residual, 3 = rmsnorm +
 * W1/W3 + SwiGLU, 4 = W2+residual, 5 = final rmsnorm + classifier.  Uses
 * slot 0's last token and position.  It overwrites activations and the
 * cache row at that position, so re-run the step afterwards if its result
 * matters.
 */
int l2_launch_op(l2_ctx *ctx, int op, int layer, int count);

/*
 * l2_launch_op for the kernels of a step of `batch` rows (batched sequences,
 * or a prompt chunk when the last step was one), as that step launches them
 * (the tensor-core GEMV for 16-64 rows unless L2_FLAG_NO_TC).  The handle's
 * last step must have had `batch` rows (else L2_ESTATE); its step block (rows'
 * tokens, positions, slots, attention chunk plan) is reused.  batch 1 is
 * l2_launch_op.  Profiling only: it overwrites activations and the cache rows
 * of that step.  The pages have no counterpart.
 */
int l2_launch_op_batch(l2_ctx *ctx, int op, int layer, int batch, int count);

/*
 * Prefill: the T tokens of a prompt, at positions pos0..pos0+T-1 of one
 * sequence (KV-cache slot `slot`), with the pages' causal attention (token
 * i attends to positions 0..pos0+i).  Cache rows pos0.. of the slot are
 * written; rows before pos0 must exist (pos0 <= l2_position(slot), else
 * L2_ESTATE); pos0 + T <= seq_len and every token in [0, vocab_size), else
 * L2_EINVAL.  logits_out (DEVICE, [T][vocab_size], or NULL) receives the
 * logits after each token, each equal to what l2_forward gives for that
 * token at that position.  The tokens are processed 64 at a time (max_batch
 * at a time with L2_FLAG_DEBUG) as one batched step each: the rows of a
 * chunk share the weights read and read the cache rows the chunk's earlier
 * rows write.  Any handle can prefill in 64-row chunks: the per-row buffers
 * are sized for 64 rows, the KV cache for max_batch slots.  Chunks of 16 or
 * more rows run their matrix products on the tensor cores (unless
 * L2_FLAG_NO_TC), and where it pays their attention reads each cache tile
 * once per 16 query vectors instead of once per row.  The pages have no
 * counterpart (their loop feeds a prompt one token per step); the R/Keras
 * page's full-sequence causal forward computes the same values.
 */
int l2_prefill(l2_ctx *ctx, int slot, int T, const int *tokens, int pos0, float *logits_out);

/*
 * l2_forward_batch with the tokens read from DEVICE memory when the step
 * runs (for instance the tokens_out of the previous l2_sample), so a
 * generation loop need not wait for the host: tokens_dev [B] ints on the
 * device, pos [B] host ints (checked on the host as in l2_forward_batch).
 * A token outside [0, vocab_size) cannot be checked on the host: the step
 * then uses token 0 for that slot and the next l2_sync returns L2_EDEVICE.
 * Enqueues one extra one-thread kernel before the step.  The pages have no
 * counterpart (their loop keeps the token on the host).
 */
int l2_forward_dev_tokens(l2_ctx *ctx, int B, const int *tokens_dev, const int *pos, float *logits_out);

/* Number of kernel launches one step of batch B enqueues, or L2_EINVAL:
 * 5 * n_layers + 1, plus one (the embedding kernel) when the step's matrix
 * products run on the tensor cores, or 1 for the persistent step kernel. */
int l2_kernels_per_step(const l2_ctx *ctx, int B);

/* Bytes each step copies from host to device: the step block (per row its
 * token, position, cache slot and the slot's rows written before the step;
 * the output pointer; the row count; the step's total attention rows). */
int l2_step_input_bytes(void);

/*
 * l2_forward without allocating anything, for callers that cannot call
 * cudaMalloc once decoding has started: a serving process that handed all of
 * the device memory to its own pool at start-up, or a latency-critical loop
 * that must not hit the implicit device synchronisation an allocation or a
 * free may cause.  (l2_forward may build a CUDA graph on its first call for a
 * batch size, and building one allocates.)  The pages have no counterpart of
 * this entry point.
 * Same arguments, checks, status codes and result as l2_forward, for slot 0.
 * The step's kernels are launched one by one, and the attention kernel keeps
 * its cross-CTA partial results and tickets in one static device array of
 * 512 KiB (131072 floats) compiled into the library, which every GPU that
 * loads the library holds until the process exits.  A handle whose attention
 * needs more, n_heads * n_chunks * (head_size + 2) + n_kv_heads floats with
 * n_chunks = min(floor(c * SMs / n_kv_heads), ceil(seq_len / 128)) and c the
 * attention CTAs that fit on one SM (at most 4), is refused
 * with L2_EINVAL before anything is enqueued.  (With one attention CTA per
 * SM on 152 SMs: 16.6 k floats at the Llama-2-7B shape; 8 query heads per KV
 * head of size 128 need 158 k and are refused.)  l2_create looks up the
 * array's device address (once per device, with that device current), which
 * loads the module that holds it: the array is resident on a device from the
 * first handle created there, so this entry point itself never makes the
 * runtime allocate.  The handle's device must be current.  Every call shares
 * the array and clears its tickets first: calls whose kernels overlap on the
 * GPU (handles on different streams) race and give wrong results.
 */
int l2_forward_static(l2_ctx *ctx, int token, int pos, float *logits_out);

/*
 * Next-token sampling on the device: the sampler of the generation loop on
 * the pages ("run.c": argmax(), sample() and the main loop; "run.c 逐行解讀"
 * §6 Sampler: random_u32() xorshift* and sample() with temperature and
 * top-p).  For each of B sequences, from logits[b][0..vocab_size):
 *   temperature == 0: the index of the first maximum; rng_state[b] unchanged;
 *   temperature > 0: one xorshift* draw from rng_state[b] (advanced in
 *     place), its top 24 bits k the coin; the tempered softmax weights
 *     q_i = floor(E(l_i / T - max_j l_j / T) * 2^48), E a specified fp32
 *     exponential (Cody-Waite reduction, degree-7 Taylor polynomial, within
 *     1 ulp of exp, 0 below -87); the first index whose running total of q
 *     exceeds floor(k * total / 2^24);
 *   0 < topp < 1: the same draw restricted to the nucleus, the shortest
 *     prefix of the weights sorted descending (ties: lower index first)
 *     whose total P has P * 2^24 >= floor(topp * 2^24) * total, walked in
 *     that order against floor(k * P / 2^24).
 * All sums are exact integer arithmetic, so the result is a function of the
 * inputs alone (bit-for-bit reproducible).  Tokens whose weight is below
 * 2^-48 of the largest are never drawn.
 * logits (fp32, row-major [B][vocab_size], 4-byte aligned), rng_state
 * ([B] 64-bit states, non-zero) and tokens_out ([B] ints) are DEVICE
 * pointers owned by the caller; rows of logits are not modified.  The work
 * is enqueued on cuda_stream (NULL: the legacy default stream) and the call
 * returns without waiting.  L2_EINVAL for NULL pointers, host pointers,
 * B < 1, vocab_size outside 1..49152, a negative or non-finite temperature
 * or a non-finite topp (l2_last_error(NULL) describes it); L2_ECUDA if the
 * launch fails.  Not for logits containing NaN.
 */
int l2_sample(const float *logits, int B, int vocab_size, float temperature, float topp,
              unsigned long long *rng_state, int *tokens_out, void *cuda_stream);

/*
 * Fault injection for tests: makes the n-th device allocation from now on
 * (n >= 1) fail as if out of memory; 0 disables.  Process-wide.
 */
void l2_debug_fail_alloc_at(int n);

/*
 * Fault injection for tests: makes the n-th CUDA graph instantiation from now
 * on (n >= 1) fail; the step that needed the graph returns L2_ECUDA with
 * nothing run and the cache position unchanged, and the next call builds the
 * graph again.  0 disables.  Process-wide.
 */
void l2_debug_fail_graph_at(int n);

/*
 * Failure-path check for tests: enqueues one kernel on the handle's stream
 * that waits, with a limit of limit_us microseconds (1..2000000), on an
 * mbarrier that nothing arrives on, through the same bounded wait the decode
 * kernels use.  When the wait gives up it sets the device error word, waits
 * (bounded) for its own bulk copy in flight and returns; it also leaves the
 * handle's attention tickets counted, as a chunk merge that stopped early
 * would.  The next l2_sync then returns L2_ETIMEOUT, clears the error word and
 * the tickets, and the handle steps normally again.  Nothing faults or hangs.
 * L2_EINVAL for a bad handle or limit.  The pages have no counterpart.
 */
int l2_debug_wait_timeout(l2_ctx *ctx, int limit_us);

/*
 * The bounds-checked build of this library (compiled with L2_DEBUG_BOUNDS=1;
 * the Python binding loads it when L2DECODE_BOUNDS_CHECKED=1): every index the
 * kernels compute into the handle's buffers, and every bulk copy's source
 * range, is checked against the buffer's size; a violation sets the device
 * error word (l2_sync then returns L2_EDEVICE) and the access is skipped, so
 * nothing is read or written out of range.  The persistent step kernel
 * (L2_FLAG_PERSIST) is not instrumented.  l2_debug_bounds_checked returns 1
 * in that build and 0 in the release build.  l2_debug_limit_cache lowers the
 * size the checks assume for each KV cache to `floats` (never above the
 * real size; blocks): steps that then read or write cache rows past it are
 * flagged, which lets a test see the checks fire without any access out of
 * range.  It has no effect in the release build.  L2_EINVAL on a NULL handle.
 */
int l2_debug_bounds_checked(void);
int l2_debug_limit_cache(l2_ctx *ctx, unsigned long long floats);

#ifdef __cplusplus
}
#endif
#endif /* L2_DECODE_H */
