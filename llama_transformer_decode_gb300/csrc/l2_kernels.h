// Launch entry points of the decode kernels (host side).
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

#include "l2_params.h"

namespace l2 {

// Fused streaming GEMV (gemv.cu), in one of kGemvShapes launch shapes.
constexpr int kGemvShapes = 3;
cudaError_t gemv_init();
int gemv_threads(int shape);
// Dynamic shared memory of one CTA for input length n and at most ymax local outputs.
size_t gemv_smem_bytes(int shape, int n, int ymax);
// The first launch shape whose shared memory fits (its size in *smem), or -1
// (*smem then holds the smallest shape's need).
int gemv_pick_shape(int n, int ymax, size_t *smem);
cudaError_t launch_gemv(int mode, int shape, const GemvParams &p, int grid, size_t smem, cudaStream_t stream,
                        bool pdl, int wt = 0);
// Device copy of n fp32 values as bf16 (round to nearest even), on `stream`.
cudaError_t convert_to_bf16(const float *src, unsigned short *dst, size_t n, cudaStream_t stream);

// Batched fused GEMV, B >= 2 sequences per step (gemv_batched.cu).
cudaError_t gemv_batched_init();
// Most weight rows (all pieces) one CTA holds in registers for `batch` sequences.
int gemv_batched_rows_cap(int batch);
// Dynamic shared memory for stage_rows weight rows per block, `batch`
// sequences and rows of n floats (norm: the mode has an RMSNorm prologue);
// *stages and *tk receive the ring depth and K-tile width.
size_t gemv_batched_smem(int stage_rows, int batch, int n, bool norm, int *stages, int *tk);
cudaError_t launch_gemv_batched(int mode, const BatchParams &bp, int grid, size_t smem, cudaStream_t stream, bool pdl);

// Persistent step kernel for batch 1 (step_kernel.cu), one CTA per SM,
// launched cooperatively.
int step_kernel_threads();
size_t step_kernel_smem(int gq, int head_size, int xs_floats, int ys_floats, int stages, int ch4);
// 16-byte words per ring buffer (a multiple of 8, at most max_ch4) that fill
// the shared memory left by the largest phase with `stages` buffers per warp,
// or 0 if two cache rows do not fit one buffer.
int step_kernel_ring(int gq, int head_size, int xs_floats, int ys_floats, int stages, int max_ch4);
cudaError_t step_kernel_init();
int step_kernel_ctas_per_sm(int gq, size_t smem);
cudaError_t launch_step_kernel(int gq, const StepKParams &p, int grid, size_t smem, cudaStream_t stream);

// Whole batch-1 step of a small model in one thread block (step_cta.cu): its
// dynamic shared memory, the one-time attribute set-up, and the launch.
size_t step_cta_smem(int dim, int hidden, int kv_dim, int n_heads, int seq_len, int n_layers);
cudaError_t step_cta_init();
cudaError_t launch_step_cta(const CtaStepParams &p, size_t smem, cudaStream_t stream);

// Token sampler (sample.cu).
int sample_max_vocab();
size_t sample_smem_bytes(int vocab);
cudaError_t sample_init();
cudaError_t launch_sample(const SampleParams &p, int batch, cudaStream_t stream);

// Tensor-core batched GEMV (gemv_tc.cu), 16..64 sequences.
int gemv_tc_max_batch();
int gemv_tc_stages(int bpad, int wt);
size_t gemv_tc_smem(int bpad, int wt);
int gemv_tc_grid(int ntiles, int n, int ctas);
// Cluster size for the cluster split of a plan (0: stream-K), see gemv_tc.cu.
// wt: 0 fp32 weights, 1 bf16 weights.
int gemv_tc_cluster_split(int mode, int wt, int ntiles, int n, int bpad, int num_sms);
size_t gemv_tc_ws_floats(int grid, int bpad);
cudaError_t gemv_tc_init();
cudaError_t launch_tc_embed(const TcParams &tp, int batch, cudaStream_t stream, bool pdl);
cudaError_t launch_gemv_tc(int mode, const TcParams &tp, int grid, cudaStream_t stream, bool pdl);

// Flash-decoding attention (attention.cu).
struct AttnLaunch {
    int lp;       // lanes per cache row (power of two; a lane takes 4 / 2 / 1 of its 16-byte words
                  // with 1 / 2 / more query heads per KV head)
    int gq;       // query heads per KV head, rounded up to a power of two
    int rl;       // 1: row-per-lane layout (head size 64, 4 or 8 heads per KV head)
    int threads;
    size_t smem;
    int max_chunks;  // CTAs per KV head the last CTA's merge can stage in its ring
    bool ok;      // this head size / grouping is supported
};
AttnLaunch attn_plan(int head_size, int n_heads, int n_kv_heads);
// Attention of a prompt chunk (attn_prefill.cu): rows of one slot at consecutive positions.
bool attn_prefill_supported(int head_size, int n_heads, int n_kv_heads);
cudaError_t attn_prefill_init();
cudaError_t launch_attn_prefill(const AttnParams &p, int rows, cudaStream_t stream, bool pdl);
cudaError_t attn_init();
// Attention CTAs that can be resident on one SM (registers, shared memory, threads).
int attn_ctas_per_sm(const AttnLaunch &a);
// Whether `clusters` thread-block clusters of n_chunks attention CTAs (2..8) can all
// be resident at once.
bool attn_cluster_fits(const AttnLaunch &a, int n_chunks, int clusters);
cudaError_t launch_attn(const AttnLaunch &a, const AttnParams &p, int batch, cudaStream_t stream, bool pdl);

}  // namespace l2
