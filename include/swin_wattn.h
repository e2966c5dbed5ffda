/*
 * swin_wattn -- the Swin shifted-window multi-head self-attention block on
 * one GB300 (sm_103a), behind a plain C ABI.
 *
 * The block (pages "Boosting Swin Transformer Speed: Profiling, Mixed
 * Precision, and Kernel Fusion Secrets", Introduction and Training
 * Optimization; "Swin Transformer V2" (neura.market), How It Works):
 *   cyclic shift by -s, partition into M x M windows, QKV projection with
 *   bias, per-window per-head logits plus relative position bias, the
 *   shift-region mask, softmax, multiplication by V, window reverse, roll
 *   back by +s, output projection with bias.
 * Two logit modes:
 *   V1  q.k / sqrt(d) + table[idx, head]   (learned (2M-1)^2 x heads table)
 *   V2  cos(q, k) / max(tau_head, 0.01) + table[idx, head]   (table from the
 *       meta-network G over log-spaced coordinates, built once)
 * Readings where the pages give no formula: roll by -s moves the element at
 * (i+s) mod n to i; tokens row-major in a window, windows row-major per
 * image; idx = (ri-rj+M-1)*(2M-1) + (ci-cj+M-1) for query i, key j (in-window
 * coordinates); shifted frame cut into bands [0,H-M), [H-M,H-s), [H-s,H) per
 * axis and pairs from different (row band, column band) regions get weight
 * exactly 0; V2 cos uses max(|v|, 1e-12) norms and no 1/sqrt(d).
 *
 * Every call is host code; device work is enqueued on the caller's stream
 * and is asynchronous.  Pointers are device pointers unless the name says
 * host.  The caller owns every tensor; the library frees only what it
 * allocated itself.  One handle must not be used from two host threads at
 * once.  No call falls back to the CPU.
 */
#ifndef SWIN_WATTN_H
#define SWIN_WATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct swin_wattn_s *swin_wattn_t;
typedef struct CUstream_st *swin_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* mode: the logit mode, optionally OR-ed with SWIN_WATTN_FP32. */
enum {
    SWIN_WATTN_V1 = 0,    /* dot-product logits, learned bias table */
    SWIN_WATTN_V2 = 1,    /* scaled-cosine logits, table from G */
    SWIN_WATTN_FP32 = 0x10 /* fp32 tensors and fp32 arithmetic (default: bf16
                              tensors, fp32 accumulation) */
};

/* Status codes (every call returns one). */
enum {
    SWIN_WATTN_OK = 0,
    SWIN_WATTN_EINVAL = -1,       /* bad argument: shape, NULL, alignment, aliasing */
    SWIN_WATTN_EUNSUPPORTED = -2, /* valid block, but no kernel for this shape */
    SWIN_WATTN_ECUDA = -3,        /* a CUDA runtime call failed (launch, copy, alloc) */
    SWIN_WATTN_ENOMEM = -4,       /* device allocation of the handle's workspace failed */
    SWIN_WATTN_ETIMEOUT = -5,     /* a kernel gave up a bounded wait (reported by
                                     swin_wattn_sync_status) */
    SWIN_WATTN_ESCRATCH = -6,     /* the call needs more intermediate memory than the
                                     fixed scratch of swin_wattn_forward_noalloc holds */
    SWIN_WATTN_ECORRUPT = -7      /* with SWIN_WATTN_DEBUG set only: a guard band
                                     around a handle's workspace was overwritten */
};

/* Environment switches (read whenever a handle allocates or grows a device
 * workspace; no effect on calls that need no new workspace):
 *   SWIN_WATTN_FAIL_ALLOC  set and not "0": every such allocation fails as if
 *       the device were out of memory, and the call returns SWIN_WATTN_ENOMEM
 *       (the handle stays usable; a later call with the switch unset
 *       allocates normally).  For testing a caller's error path.
 *   SWIN_WATTN_DEBUG       set and not "0": each such workspace is allocated
 *       with a 4 KiB guard band on either side, filled with a byte pattern.
 *       After every call that used the workspace the library synchronises the
 *       call's stream and reads the bands back; a changed byte returns
 *       SWIN_WATTN_ECORRUPT.  For debugging only (it serialises the stream). */

/* Options for swin_wattn_set_option. */
enum {
    SWIN_WATTN_OPT_PATH = 1,       /* 0 = automatic, 1 = three kernels (QKV GEMM,
                                      window attention, projection GEMM),
                                      2 = the fused single-kernel block */
    SWIN_WATTN_OPT_WAIT_LIMIT_US = 2, /* limit of every device-side wait, microseconds
                                         (default 2,000,000) */
    SWIN_WATTN_OPT_HOST_CHUNKS = 3,  /* chunks of whole images that
                                        swin_wattn_forward_host overlaps (1..16,
                                        default 8; fewer when B is smaller) */
    SWIN_WATTN_OPT_OVERLAP_CALLS = 4 /* 0 (default) or 1: swin_wattn_forward's
                                        kernels may start while the kernels
                                        queued before it on the stream finish
                                        (programmatic dependent launch): they load
                                        the parameters (Wqkv, bqkv, the bias table,
                                        logit_scale, Wproj, bproj) during that time
                                        and wait for the earlier work before they
                                        read x or write out.  With 1 the caller
                                        guarantees that no work queued before a
                                        call writes that call's parameters (fixed
                                        weights, as in serving).  The three-kernel
                                        path's kernels overlap the same way, each
                                        with the one before it; the host-buffer
                                        forward is unaffected.  swin_wattn_backward
                                        then overlaps its own kernels after the
                                        recompute GEMM (all but the large-window
                                        attention ones), never the work queued
                                        before the call, so it needs no such
                                        guarantee. */
};

/* Creates a handle for blocks with C channels, `heads` heads (d = C/heads),
 * M x M windows and shift s.  Allocates the handle's 4-byte device error
 * word; no kernel runs.
 * Errors: EINVAL if out is NULL, C, heads or M <= 0, C % heads != 0,
 * s < 0 or s >= M, or mode has unknown bits.  EUNSUPPORTED for bf16 mode when
 * d != 32 or M > 64 (the tensor-core kernels are written for d = 32), and for
 * fp32 mode when one window does not fit in shared memory. */
int swin_wattn_create(swin_wattn_t *out, int C, int heads, int M, int shift, int mode);

/* Frees the handle and its workspace.  Synchronises the device first.
 * NULL is accepted (no-op). */
int swin_wattn_destroy(swin_wattn_t h);

/* One forward pass of the block.
 *   x           [B, H, W, C]            bf16 (fp32 in FP32 mode), contiguous
 *   Wqkv        [3C, C] row-major       output channel o = part*C + head*d + e,
 *                                       part 0,1,2 = q,k,v
 *   bqkv        [3C]                    may be NULL (zero)
 *   bias_table  [(2M-1)^2, heads]       row idx, column head (same dtype as x)
 *   logit_scale [heads] fp32            tau per head (V2; clipped at 0.01 inside);
 *                                       ignored (may be NULL) in V1
 *   Wproj       [C, C] row-major        (out x in)
 *   bproj       [C]                     may be NULL (zero)
 *   out         [B, H, W, C]            same dtype as x; must not overlap x
 * All device pointers must be 16-byte aligned.
 * Errors (checked before any launch): EINVAL for NULL h/x/Wqkv/bias_table/
 * Wproj/out, NULL logit_scale in V2, B < 0, H or W not a positive multiple
 * of M, misaligned pointers, out overlapping x.  B == 0 is a no-op.  ECUDA if
 * a launch fails.  ENOMEM if the workspace of the three-kernel path cannot be
 * allocated.  A device-side timeout is reported by swin_wattn_sync_status. */
int swin_wattn_forward(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv,
                       const void *bqkv, const void *bias_table, const float *logit_scale,
                       const void *Wproj, const void *bproj, void *out, swin_stream_t stream);

/* The same forward with x and out in HOST memory (pinned memory gives
 * asynchronous copies).  The batch is cut into up to 8 chunks of whole images
 * (SWIN_WATTN_OPT_HOST_CHUNKS sets the count)
 * (windows never cross images, so each chunk is an exact forward of its
 * images), and each chunk is copied host->device into a buffer the handle
 * owns, run, and copied device->host into out_host; the three steps of
 * different chunks overlap on three streams the handle owns, so the two copy
 * directions and the kernels run at the same time.  The call is ordered on
 * `stream` as if it ran there: the handle's streams wait for the work already
 * on `stream`, and `stream` waits for the last chunk's copy back.  The
 * weights, biases, table and logit_scale are device pointers, as in
 * swin_wattn_forward.  Returns once the work is enqueued; synchronise the
 * stream before reading out_host.  Errors as swin_wattn_forward, plus ENOMEM
 * when the staging buffers cannot be allocated. */
int swin_wattn_forward_host(swin_wattn_t h, const void *x_host, int B, int H, int W,
                            const void *Wqkv, const void *bqkv, const void *bias_table,
                            const float *logit_scale, const void *Wproj, const void *bproj,
                            void *out_host, swin_stream_t stream);

/* V2: the relative-bias table of the meta-network G over log-spaced
 * coordinates ("Swin Transformer V2" (neura.market), How It Works: a small
 * network G maps relative coordinates to bias values; log-spaced
 * coordinates).  For dr, dc in [-(M-1), M-1]:
 *   u = (sign(dr) ln(1+|dr|), sign(dc) ln(1+|dc|))
 *   table[idx, :] = W2 relu(W1 u + b1),  idx = (dr+M-1)*(2M-1) + (dc+M-1)
 * W1 [hidden, 2], b1 [hidden] (may be NULL), W2 [heads, hidden], all fp32
 * device pointers; table [(2M-1)^2, heads] in the handle's dtype.  Computed
 * in fp32 and rounded once.  Call once per weight set, not per forward.
 * Errors: EINVAL for NULL pointers or hidden <= 0 or hidden > 4096. */
int swin_wattn_cpb_table(swin_wattn_t h, const float *W1, const float *b1, const float *W2,
                         int hidden, void *table, swin_stream_t stream);

/* Synchronises `stream`, then reads and clears the handle's device error
 * word.  Returns OK, ETIMEOUT if a kernel gave up a bounded wait since the
 * last call, or ECUDA if the stream reports an error. */
int swin_wattn_sync_status(swin_wattn_t h, swin_stream_t stream);

/* Sets an option (see SWIN_WATTN_OPT_*).  EINVAL for unknown options or values. */
int swin_wattn_set_option(swin_wattn_t h, int option, int64_t value);

/* Which path swin_wattn_forward takes for a B x H x W input: 1 = three
 * kernels, 2 = fused, 3 = fp32 kernel; a negative status if it would fail. */
int swin_wattn_path(swin_wattn_t h, int B, int H, int W);

/* Number of kernel launches the last swin_wattn_forward enqueued. */
int swin_wattn_last_launches(swin_wattn_t h);

/* Static text for a status code. */
const char *swin_wattn_strerror(int code);

/* Text of the CUDA runtime error behind the handle's most recent ECUDA from a
 * launch in swin_wattn_forward (or "no CUDA error recorded").  Static string. */
const char *swin_wattn_last_cuda_error(swin_wattn_t h);

/* Size of the scratch array compiled into the library for
 * swin_wattn_forward_noalloc (64 MiB per GPU that loads the library, held
 * until the process exits), and the part of it that holds the intermediates
 * (the first 256 bytes are a status word). */
#define SWIN_WATTN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
#define SWIN_WATTN_NOALLOC_MAX_INTERMEDIATE_BYTES (SWIN_WATTN_NOALLOC_SCRATCH_BYTES - 256)

/* The forward pass of swin_wattn_forward for callers that cannot allocate
 * device memory.  None of the sources describes one: this is a deployment
 * convenience of this library.
 *
 * Who needs it: code that runs where it does not own the device allocator
 * (inside a framework whose caching allocator must see every allocation,
 * or an embedded runtime that fixes its memory budget at start-up), and code
 * that must not allocate after start-up (a latency-critical serving loop,
 * where cudaMalloc would synchronise the device).  swin_wattn_create
 * allocates an error word and swin_wattn_forward a workspace for the q/k/v
 * and attention intermediates; this entry point takes no handle and calls
 * no cudaMalloc, cudaFree or other allocating routine.  Its intermediates
 * live in a fixed array compiled into the library (see
 * SWIN_WATTN_NOALLOC_SCRATCH_BYTES).
 *
 * Arguments: the block parameters of swin_wattn_create (C, heads, M, shift,
 * mode; bf16 mode only, d = 32, M <= 64), then those of swin_wattn_forward
 * with the same layouts and rules.  The caller still owns and passes every
 * input and the output.
 * Limit: 8 * B * H * W * C bytes of intermediates must fit in
 * SWIN_WATTN_NOALLOC_MAX_INTERMEDIATE_BYTES (for C = 96 that is about 87,000
 * tokens, e.g. B = 27 at 56 x 56); larger calls return SWIN_WATTN_ESCRATCH
 * before any launch.
 * Set-up: the first call on a device looks up the device address of the
 * array (this can load the library's device code on that device); make that
 * first call before any stream capture.  Later calls reuse the address while
 * the device's context stays the same; after a device reset (a new context)
 * the next call looks it up again, and counts as a first call.
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents; the call clears the status word it needs itself.  Calls
 * whose work overlaps on the GPU (different streams, or several host threads)
 * race on the array and corrupt each other's results: serialise them.
 * A bounded-wait timeout inside the kernels is recorded in the array's status
 * word and read back by swin_wattn_noalloc_sync_status.
 * Errors: EINVAL / EUNSUPPORTED as swin_wattn_create and swin_wattn_forward
 * (fp32 mode is EUNSUPPORTED), ESCRATCH as above, ECUDA if a launch fails.
 * B == 0 is a no-op. */
int swin_wattn_forward_noalloc(int C, int heads, int M, int shift, int mode, const void *x, int B, int H,
                               int W, const void *Wqkv, const void *bqkv, const void *bias_table,
                               const float *logit_scale, const void *Wproj, const void *bproj, void *out,
                               swin_stream_t stream);

/* Status of the swin_wattn_forward_noalloc calls made on the current device
 * so far: waits for `stream` (the stream of those calls), reads the status
 * word of the fixed array (one small device-to-host copy, no allocation) and
 * clears it.  Returns SWIN_WATTN_ETIMEOUT if a kernel of one of those calls
 * gave up a bounded wait (its output is then incomplete), SWIN_WATTN_OK if
 * none did, SWIN_WATTN_ECUDA if the wait or the copy failed.  Like the entry
 * point itself, it has no counterpart in the sources. */
int swin_wattn_noalloc_sync_status(swin_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIN_WATTN_H */
