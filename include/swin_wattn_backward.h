/*
 * swin_wattn_backward -- gradients of the shifted-window attention block
 * (V1 and V2 logits) on one GB300, behind a plain C ABI.
 *
 * Page "Boosting Swin Transformer Speed: Profiling, Mixed Precision, and
 * Kernel Fusion Secrets", Training Optimization: training runs the block's
 * backward pass through the fused attention kernel and through the
 * index-mapping kernels of window partition, cyclic shift and reverse.  The
 * pages give no formula for the gradients; they are those of the forward of
 * swin_wattn.h (V1), by the chain rule:
 *   dy_w = gather(dy)                 (window order: cyclic shift -s, partition)
 *   dWproj = dy_w^T o, dbproj = sum_t dy_w, do = dy_w Wproj
 *   per window and head:  dP = do v^T, D_i = sum_j P_ij dP_ij,
 *     dS = P (dP - D), dq = dS k / sqrt(d), dk = dS^T q / sqrt(d), dv = P^T do,
 *     dtable[idx(i, j), head] += dS_ij  (masked pairs have P = 0, so dS = 0)
 *   dWqkv = dqkv^T xs, dbqkv = sum_t dqkv, dx = scatter(dqkv Wqkv)
 * (o, P, q, k, v as in the forward; xs = gather(x); scatter = window
 * reverse then roll by +s, the inverse map of gather).
 *
 * The call recomputes q, k and v from x (nothing of the forward is kept) and
 * runs: the QKV GEMM and the do GEMM, each gathering its rows into window
 * order in its loads; the attention backward, which recomputes S and P,
 * yields o, dq, dk, dv (written back in token order) and the table
 * gradient; the dx GEMM; two weight-gradient GEMMs (split-K over all
 * tokens, which do not depend on the token order; each also yields its
 * bias gradient, the column sums of dy and dqkv, and adds its per-CTA
 * partial sums in a fixed order).
 *
 * Windows of more than 64 tokens (up to 24 x 24): the large-window forward
 * kernel runs first and keeps, besides o, the log2 of each row's softmax
 * normaliser (lse), so that P = exp2(logit * log2 e - lse) needs no row pass;
 * D_i = do_i . o_i (equal to sum_j P_ij dP_ij); the attention backward then
 * runs over (head, window, tile of 128 keys) units, summing dq over the key
 * tiles in fp32 and the table gradient as fixed-point integers on a 2^-19
 * grid (terms of magnitude 4 or more in fp32).
 *
 * Conventions of swin_wattn.h: device pointers, asynchronous on `stream`,
 * caller-owned tensors, status codes SWIN_WATTN_*, no CPU fallback.
 */
#ifndef SWIN_WATTN_BACKWARD_H
#define SWIN_WATTN_BACKWARD_H

#include "swin_wattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Gradients of sum(out * dy), out = the handle's block applied to x.
 * Inputs (bf16, as swin_wattn_forward): x [B, H, W, C], Wqkv [3C, C],
 * bqkv [3C] (NULL = zero), bias_table [(2M-1)^2, heads], logit_scale (fp32
 * [heads], tau; V2 only, NULL in V1), Wproj [C, C], bproj [C] (NULL = zero;
 * does not enter any gradient), dy [B, H, W, C].
 * Outputs, overwritten: dx [B, H, W, C] bf16; dWqkv [3C, C], dbqkv [3C],
 * dtable [(2M-1)^2, heads], dlogit_scale [heads] (V2; may be NULL in V1),
 * dWproj [C, C], dbproj [C], all fp32.
 * V2 (page "Swin Transformer V2" (neura.market), How It Works: cosine
 * logits over a learned tau clipped at 0.01): with q^ = q / max(|q|, 1e-12)
 * and sigma = 1 / max(tau, 0.01) per head, logit = sigma q^.k^ + table, and
 *   dq^ = sigma dS k^, dk^ = sigma dS^T q^,
 *   dq = (dq^ - q^ (q^ . dq^)) / |q| (likewise k),
 *   dtau = -sum(dS q^.k^) / tau^2 where tau > 0.01, else 0;
 * the table gradient flows on to G's weights through swin_wattn_cpb_backward.
 * Every pointer 16-byte aligned; dx overlaps neither x nor dy.
 * Errors: EINVAL for NULL or misaligned pointers (logit_scale and
 * dlogit_scale are required in V2), bad shapes, overlap; EUNSUPPORTED for an
 * fp32 handle, windows of more than 24 x 24 tokens, C != 32 heads, or
 * B*H*W >= 2^31; ENOMEM if the workspace (8 * B*H*W*C bf16 elements plus
 * 4C^2, plus 2 B*H*W*heads fp32 in V2, plus (2 heads + C) B*H*W fp32 for
 * windows of more than 64 tokens, plus the weight gradients' partial sums)
 * cannot be allocated; ECUDA for launch failures.
 * B = 0 zeroes the parameter gradients and returns. */
int swin_wattn_backward(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        const void *bias_table, const float *logit_scale, const void *Wproj, const void *bproj,
                        const void *dy, void *dx, float *dWqkv, float *dbqkv, float *dtable, float *dlogit_scale,
                        float *dWproj, float *dbproj, swin_stream_t stream);

/* V2: the gradients of G's weights (as swin_wattn_cpb_table: W1 [hidden, 2],
 * b1 [hidden] (may be NULL), W2 [heads, hidden], fp32) from the gradient of
 * its table, dtable [(2M-1)^2, heads] fp32 (swin_wattn_backward's output):
 * dW2[h, k] = sum_idx dtable[idx, h] relu(a_k(idx)), and through the ReLU
 * (a_k > 0) da_k = sum_h dtable[idx, h] W2[h, k], dW1[k] = sum_idx da_k u(idx),
 * db1[k] = sum_idx da_k, with a_k(idx) = W1[k] . u(idx) + b1[k] over the
 * log-spaced coordinates u.  Outputs overwritten: dW1 [hidden, 2], db1
 * [hidden] (may be NULL), dW2 [heads, hidden], fp32 device pointers.
 * Errors: EINVAL for NULL pointers or hidden outside 1..4096; EUNSUPPORTED
 * for more than 16 heads. */
int swin_wattn_cpb_backward(swin_wattn_t h, const float *W1, const float *b1, const float *W2, int hidden,
                            const float *dtable, float *dW1, float *db1, float *dW2, swin_stream_t stream);

/* Number of kernels the last successful swin_wattn_backward enqueued. */
int swin_wattn_backward_launches(swin_wattn_t h);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_WATTN_BACKWARD_H */
