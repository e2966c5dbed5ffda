/*
 * swin_block -- the whole Swin Transformer block around the shifted-window
 * attention of swin_wattn.h: LayerNorm, the two residual connections and the
 * MLP, on one GB300 (sm_103a), behind a plain C ABI.
 *
 * Pages: "Swin Transformer V2" (neura.market), How It Works: the original
 * Swin normalises before each sub-layer (pre-norm); V2 normalises the output
 * of each residual branch before adding it back to the main branch
 * (residual post-norm):
 *   V1  z = x + attn(LN1(x));  y = z + MLP(LN2(z))
 *   V2  z = x + LN1(attn(x));  y = z + LN2(MLP(z))
 * attn is the swin_wattn block (cyclic shift, windows, QKV, logits + bias +
 * mask, softmax, P.V, reverse, roll back, projection).  Readings where the
 * pages give no formula: LayerNorm over a token's C channels with the biased
 * variance and eps = 1e-5, per-channel gain and shift; MLP(u) =
 * GELU(u W1^T + b1) W2^T + b2 with hidden width mlp_ratio * C and the exact
 * GELU u * Phi(u).  The extra LayerNorm that V2 inserts every six blocks of
 * its largest models belongs to the stage, not to a block: swin_stage_norm.
 *
 * bf16 tensors, fp32 arithmetic inside each step; the residual stream z, the
 * LayerNorm outputs and the MLP hidden activations are rounded to bf16
 * between steps.  Same conventions as swin_wattn.h: device pointers,
 * asynchronous on `stream`, the caller owns every tensor, status codes
 * SWIN_WATTN_*, no CPU fallback.
 */
#ifndef SWIN_BLOCK_H
#define SWIN_BLOCK_H

#include "swin_wattn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct swin_block_s *swin_block_t;

/* The block's parameters, all device pointers, bf16 unless stated:
 *   ln1_gamma, ln1_beta, ln2_gamma, ln2_beta  [C]
 *   Wqkv [3C, C], bqkv [3C], bias_table [(2M-1)^2, heads], logit_scale (fp32,
 *   [heads], tau; V2 only), Wproj [C, C], bproj [C]: as swin_wattn_forward
 *   W1 [rC, C], b1 [rC], W2 [C, rC], b2 [C]   (r = mlp_ratio)
 * Biases may be NULL (zero); every other pointer is required, 16-byte
 * aligned. */
typedef struct swin_block_params {
    const void *ln1_gamma, *ln1_beta;
    const void *Wqkv, *bqkv, *bias_table;
    const float *logit_scale;
    const void *Wproj, *bproj;
    const void *ln2_gamma, *ln2_beta;
    const void *W1, *b1, *W2, *b2;
} swin_block_params;

/* A block of C channels, `heads` heads of C/heads = 32 channels, M x M
 * windows shifted by `shift` (0 <= shift < M), mode SWIN_WATTN_V1 (pre-norm,
 * dot-product logits) or SWIN_WATTN_V2 (residual post-norm, scaled-cosine
 * logits); bf16 only (SWIN_WATTN_FP32 is refused with EUNSUPPORTED).
 * mlp_ratio: hidden width of the MLP in units of C (1..8).  *out receives
 * the handle (NULL on failure).  The handle owns a workspace of
 * (3 + mlp_ratio) * B*H*W*C bf16 elements, allocated on the first forward
 * of a given size and freed by swin_block_destroy. */
int swin_block_create(swin_block_t *out, int C, int heads, int M, int shift, int mode, int mlp_ratio);

/* y = block(x) for x [B, H, W, C] bf16 (H % M == 0, W % M == 0), written to
 * out [B, H, W, C] (must not overlap x).  EINVAL for bad shapes, NULL or
 * misaligned pointers; ENOMEM if the workspace cannot be allocated; ECUDA
 * for launch failures (asynchronous kernel errors and bounded-wait timeouts
 * surface at swin_block_sync_status).  B = 0 is a no-op. */
int swin_block_forward(swin_block_t h, const void *x, int B, int H, int W, const swin_block_params *p, void *out,
                       swin_stream_t stream);

/* Synchronises `stream` and reports an error the block's kernels recorded
 * since the last call (SWIN_WATTN_ETIMEOUT), else SWIN_WATTN_OK. */
int swin_block_sync_status(swin_block_t h, swin_stream_t stream);

/* Number of kernel launches the last swin_block_forward on this handle
 * enqueued (C = 96 or 64 with windows of 7 or 8: 2 -- the attention with
 * LayerNorm 1 and the first residual folded in, the MLP with LayerNorm 2 and
 * the second residual -- in either mode; more where those kernels do not
 * apply); 0 before the first forward or after one that failed its checks, -1
 * for a NULL handle. */
int swin_block_last_launches(swin_block_t h);

/* Options for swin_block_set_option. */
enum {
    SWIN_BLOCK_OPT_OVERLAP_CALLS = 1 /* 0 (default) or 1: the block's fused kernels
                                        (the attention with LayerNorm 1 folded in
                                        and the MLP) may start while the kernels
                                        queued before them on the stream finish
                                        (programmatic dependent launch): each loads
                                        its parameters during that time and waits
                                        for the earlier work before it reads its
                                        input or writes its output.  With 1 the
                                        caller guarantees that no work queued before
                                        a forward writes that forward's parameters
                                        (fixed weights, as in serving). */
};

/* Sets an option (see SWIN_BLOCK_OPT_*).  EINVAL for a NULL handle, unknown
 * options or values. */
int swin_block_set_option(swin_block_t h, int option, int64_t value);

/* Frees the handle and its workspace (NULL is a no-op). */
int swin_block_destroy(swin_block_t h);

/* The LayerNorm step on its own, for tests: per token of C channels,
 *   flags 0: out_ln = LN(a)
 *   flags 1: s = a + b; out_sum = s (if not NULL); out_ln = LN(s)
 *   flags 2: out_ln = b + LN(a)
 * a, b, out_sum, out_ln [rows, C] bf16; gamma, beta [C] bf16.  C a multiple
 * of 8 and at most 2048. */
int swin_block_test_layernorm(const void *a, const void *b, const void *gamma, const void *beta, void *out_sum,
                              void *out_ln, int rows, int C, int flags, swin_stream_t stream);

/* The extra LayerNorm of V2's largest models ("Swin Transformer V2"
 * (neura.market), How It Works: a layer normalisation inserted every six
 * blocks), applied to the main branch between blocks of a stage: per token of
 * C channels, out = LN(x) (biased variance, eps = 1e-5, gain gamma, shift
 * beta).  Reading (the page gives no more): it follows blocks 6, 12, ... of
 * a stage, before the merging step, with a gain and shift of its own.
 * x, out [rows, C] bf16 (out may be x itself, not a partial overlap); gamma,
 * beta [C] bf16; C a multiple of 8, at most 2048.  EINVAL for bad sizes,
 * NULL, misaligned or partly overlapping pointers; ECUDA for a launch
 * failure.  rows = 0 is a no-op. */
int swin_stage_norm(const void *x, int rows, int C, const void *gamma, const void *beta, void *out,
                    swin_stream_t stream);

/* ---- merging step between stages ----------------------------------------------
 * Between stages of the hierarchy ("Boosting Swin Transformer Speed",
 * Introduction: a pyramid of stages) the resolution halves and the channels
 * double.  Reading (the pages give no formula): each 2 x 2 neighbourhood is
 * concatenated in the order (0,0), (1,0), (0,1), (1,1) (row offset first),
 * normalised over its 4C channels (as the block's LayerNorm) and mapped by a
 * linear layer without bias:
 *   out[b, i, j, :] = LN(concat(x[b, 2i, 2j], x[b, 2i+1, 2j], x[b, 2i, 2j+1],
 *                               x[b, 2i+1, 2j+1])) Wm^T
 * A stage is `depth` blocks with shifts 0, M/2, 0, ... (one swin_block handle
 * per shift) followed by this step. */
typedef struct swin_merge_s *swin_merge_t;

/* C input channels (multiple of 8, 4C <= 2048).  The handle owns a workspace
 * of B*H*W*C bf16 elements (allocated on first use). */
int swin_merge_create(swin_merge_t *out, int C);

/* x [B, H, W, C] bf16 (H, W even) -> out [B, H/2, W/2, 2C] bf16; gamma, beta
 * [4C] bf16; Wm [2C, 4C] bf16.  EINVAL for odd H or W, NULL or misaligned
 * pointers, overlap of x and out; ENOMEM if the workspace cannot be
 * allocated; ECUDA for launch failures.  B = 0 is a no-op. */
int swin_merge_forward(swin_merge_t h, const void *x, int B, int H, int W, const void *gamma, const void *beta,
                       const void *Wm, void *out, swin_stream_t stream);

/* Frees the handle and its workspace (NULL is a no-op). */
int swin_merge_destroy(swin_merge_t h);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_BLOCK_H */
