/*
 * Stage hooks of libswin_wattn, for tests: each runs one kernel of the
 * three-kernel path on caller buffers, so that every step of the block can be
 * compared with the float64 oracle on its own.  Same conventions as
 * swin_wattn.h (device pointers, bf16 tensors, asynchronous on `stream`,
 * status codes).  Intermediate layout, window order: row r = win*N + t with
 * win = (b*(H/M) + wi)*(W/M) + wj and t = ti*M + tj (N = M*M tokens per
 * window).
 */
#ifndef SWIN_WATTN_TEST_H
#define SWIN_WATTN_TEST_H

#include "swin_wattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Cyclic shift by -s, window partition and QKV projection with bias
 * (pages: "Boosting Swin Transformer Speed", Training Optimization -- the
 * partition/shift index maps; Inference Optimization -- QKV GEMM with bias).
 *   qkv[r, o] = sum_c x[b, (wi*M+ti+s) mod H, (wj*M+tj+s) mod W, c] * Wqkv[o, c] + bqkv[o]
 * qkv is [B*H*W, 3C] bf16 in window order.  In V2 mode every q and k head
 * (32 columns) is scaled to unit L2 norm (norm clamped at 1e-12) after the
 * bias, before rounding, as the attention stage expects.  bf16 mode only. */
int swin_wattn_test_qkv(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv,
                        const void *bqkv, void *qkv, swin_stream_t stream);

/* Per-window, per-head attention on a window-ordered qkv buffer: logits (V1 or
 * V2) + relative bias + shift mask, softmax, P.V.  In V2 mode q and k must
 * already be unit vectors (as swin_wattn_test_qkv writes them), so q.k is the
 * cosine.  attn is [B*H*W, C] bf16 in window order, channel head*d + e.  bf16
 * mode only. */
int swin_wattn_test_attn(swin_wattn_t h, const void *qkv, int B, int H, int W,
                         const void *bias_table, const float *logit_scale, void *attn,
                         swin_stream_t stream);

/* Output projection with bias, window reverse and roll by +s:
 *   out[b, (wi*M+ti+s) mod H, (wj*M+tj+s) mod W, :] = attn[r, :] Wproj^T + bproj
 * bf16 mode only. */
int swin_wattn_test_proj(swin_wattn_t h, const void *attn, int B, int H, int W,
                         const void *Wproj, const void *bproj, void *out, swin_stream_t stream);

/* The tensor-core GEMM building block alone, no index maps:
 *   D[m, n] = sum_k A[m, k] * Bw[n, k] + bias[n]
 * A [rows, K], Bw [N, K], D [rows, N], bias [N] (may be NULL), bf16,
 * row-major.  K and N multiples of 16 (N <= 2048), rows >= 0.
 * swizzle_bytes selects the operand layout: 128 (K blocks of 64 in 128-byte
 * swizzled shared memory, as the three-kernel path), 64 (K blocks of 32 in
 * 64-byte swizzled shared memory, as the fused kernel) or 0 (A staged in
 * tensor memory, the MMA form that reads A from TMEM; K <= 128, N <= 256) or
 * -64 (Bw given as [K, N] row-major and used as an N-major operand, 64-byte
 * swizzle; N = 32 or 64, K <= 128) or 1 (lane-masked MMA pair: Bw is [2N, K]
 * and D is [rows, 2N]; within every block of 128 rows, rows 0..63 use
 * Bw[0:N] and rows 64..127 use Bw[N:2N], the two products written into the
 * same accumulator columns by MMAs that mask each other's rows; D columns
 * 0..N-1 come from the shared-memory-A form and N..2N-1 from the TMEM-A form;
 * bias ignored; K <= 128 and a multiple of 32, N <= 128). */
int swin_wattn_test_gemm(const void *A, const void *Bw, const void *bias, void *D, int rows, int N,
                         int K, int swizzle_bytes, swin_stream_t stream);

/* Overwrites one byte of a guard band of the handle's forward workspace
 * (side 0: the band before it, 1: the band after it), so that the
 * SWIN_WATTN_DEBUG check can be tested.  EINVAL unless the workspace was
 * allocated with guard bands. */
int swin_wattn_test_corrupt_workspace(swin_wattn_t h, int side);

/* Runs a one-block kernel that waits on a barrier nothing completes, with the
 * handle's wait limit, so that the bounded-wait path can be tested: the
 * kernel records a timeout in the handle's error word and returns; the
 * caller then reads ETIMEOUT from swin_wattn_sync_status. */
int swin_wattn_test_watchdog(swin_wattn_t h, swin_stream_t stream);

/* The same kernel, reporting into the status word of the fixed array of
 * swin_wattn_forward_noalloc, with a wait limit of wait_limit_us (1 us to
 * 60 s): swin_wattn_noalloc_sync_status then returns ETIMEOUT once. */
int swin_wattn_test_noalloc_watchdog(int64_t wait_limit_us, swin_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_WATTN_TEST_H */
