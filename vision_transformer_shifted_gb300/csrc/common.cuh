// Internal declarations shared by the kernels and the C ABI of libswin_wattn.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

struct swin_wattn_s;   // a forward handle (swin_wattn.h)

namespace swin {

using bf16 = __nv_bfloat16;

// Geometry of one forward call: a [B, H, W, C] token grid cut into M x M
// windows after a cyclic shift by -s.
struct Geom {
    int B, H, W, C, M, s;
    int nh, nw, N; // windows per column / row, tokens per window
    int64_t T;     // B*H*W tokens
    int64_t nwin;  // B*nh*nw windows
};

inline Geom make_geom(int B, int H, int W, int C, int M, int s)
{
    Geom g;
    g.B = B; g.H = H; g.W = W; g.C = C; g.M = M; g.s = s;
    g.nh = H / M; g.nw = W / M; g.N = M * M;
    g.T = (int64_t)B * H * W;
    g.nwin = (int64_t)B * g.nh * g.nw;
    return g;
}

// Window-order row r = win*N + t (win = (b*nh + wi)*nw + wj, t = ti*M + tj)
// -> token index b*H*W + i*W + j of its place in the original frame, where
// (i, j) = (wi*M+ti+s mod H, wj*M+tj+s mod W).  The cyclic shift by -s reads
// the token at (i+s, j+s) into shifted position (i, j); the window reverse
// followed by the roll by +s writes the result back to that same place, so
// one map serves the gather in front of the QKV projection and the scatter
// behind the output projection.
__device__ __forceinline__ int64_t window_row_to_token(const Geom &g, int64_t r)
{
    const int64_t win = r / g.N;
    const int t = (int)(r - win * g.N);
    const int per = g.nh * g.nw;
    const int b = (int)(win / per);
    const int rem = (int)(win - (int64_t)b * per);
    const int wi = rem / g.nw, wj = rem - (rem / g.nw) * g.nw;
    const int ti = t / g.M, tj = t - (t / g.M) * g.M;
    int i = wi * g.M + ti + g.s;
    if (i >= g.H) i -= g.H;
    int j = wj * g.M + tj + g.s;
    if (j >= g.W) j -= g.W;
    return ((int64_t)b * g.H + i) * g.W + j;
}

// The inverse map: token t = b*H*W + i*W + j -> its window-order row (the
// token sits at shifted position (i-s mod H, j-s mod W)).
__device__ __forceinline__ int64_t token_to_window_row(const Geom &g, int64_t t)
{
    const int64_t hw = (int64_t)g.H * g.W;
    const int64_t b = t / hw;
    const int rem = (int)(t - b * hw);
    const int i = rem / g.W, j = rem - (rem / g.W) * g.W;
    int si = i - g.s;
    if (si < 0) si += g.H;
    int sj = j - g.s;
    if (sj < 0) sj += g.W;
    const int wi = si / g.M, wj = sj / g.M;
    return ((b * g.nh + wi) * g.nw + wj) * g.N + (si - wi * g.M) * g.M + (sj - wj * g.M);
}

// 32-bit form of window_row_to_token for callers that know B*H*W < 2^31.
__device__ __forceinline__ int window_row_to_token32(const Geom &g, int r)
{
    const int win = r / g.N;
    const int t = r - win * g.N;
    const int per = g.nh * g.nw;
    const int b = win / per;
    const int rem = win - b * per;
    const int wi = rem / g.nw, wj = rem - (rem / g.nw) * g.nw;
    const int ti = t / g.M, tj = t - (t / g.M) * g.M;
    int i = wi * g.M + ti + g.s;
    if (i >= g.H) i -= g.H;
    int j = wj * g.M + tj + g.s;
    if (j >= g.W) j -= g.W;
    return (b * g.H + i) * g.W + j;
}

// Band of a shifted-frame coordinate p on an axis of length n (shift s > 0):
// 0 for [0, n-M), 1 for [n-M, n-s), 2 for [n-s, n).  Pairs of tokens whose
// (row band, column band) differ are masked.
__device__ __forceinline__ int shift_band(int p, int n, int M, int s)
{
    return p < n - M ? 0 : (p < n - s ? 1 : 2);
}

// Device error word bits.
enum : int { ERR_TIMEOUT = 1 };

struct DeviceStatus {
    int *err;          // device error word (atomicOr of ERR_* bits)
    uint64_t wait_ns;  // limit of every bounded wait
};

// ---- handle-owned workspaces (workspace.cu) ------------------------------------

// Grows *buf to at least `need` bytes (freeing the old buffer): SWIN_WATTN_OK,
// SWIN_WATTN_ENOMEM (also whenever the environment sets SWIN_WATTN_FAIL_ALLOC)
// or SWIN_WATTN_ECUDA.  With SWIN_WATTN_DEBUG set the buffer gets guard bands.
int ws_ensure(void **buf, size_t *have, size_t need);
void ws_free(void **buf, size_t *have);
// For a buffer with guard bands: synchronises `stream` and returns
// SWIN_WATTN_ECORRUPT if a band changed; SWIN_WATTN_OK at once otherwise.
int ws_check(const void *buf, cudaStream_t stream);
// Test hook: overwrites one byte of a guard band (side 0: before, 1: after).
int ws_test_corrupt(const void *buf, int side);

// ---- kernel launchers (return cudaSuccess or the error) ----------------------

enum { LOAD_PLAIN = 0, LOAD_GATHER = 1 };
enum { STORE_PLAIN = 0, STORE_SCATTER = 1 };
// (inside launch_gemm: LOAD_GATHER + STORE_PLAIN on the resident-weight kernel
// runs as plain token-order loads whose output rows go to their window-order
// places, STORE_WINDOW: the same result, without gathered loads)
enum { STORE_WINDOW = 2 };

struct GemmArgs {
    const bf16 *A;   // LOAD_PLAIN: [rows, lda]; LOAD_GATHER: x [B, H, W, K]
    int64_t lda;
    const bf16 *Bw;  // [N, K] row-major
    const bf16 *bias; // [N] or null
    bf16 *D;         // STORE_PLAIN: [rows, ldd]; STORE_SCATTER: out [B, H, W, N]
    int64_t ldd;
    int64_t rows;
    int N, K;
    Geom g;          // index maps of LOAD_GATHER / STORE_SCATTER
    int norm_cols;   // > 0: output columns below it are scaled, 32 at a time, to
                     // unit L2 norm (V2 q and k heads); 0: none
    float *norms;    // norm_cols > 0 and not null: the clamped norm max(|v|, 1e-12) of each
                     // normalised 32-column chunk, [rows, norms_ld] fp32
    int norms_ld;    // row stride of norms (0: norm_cols / 32)
    int epi;         // EPI_NONE, EPI_GELU (GELU after the bias), EPI_RESID (add R after the bias)
    const bf16 *R;   // EPI_RESID: [rows, ldr] row-major (plain store only)
    int64_t ldr;
    int overlap;     // launched to overlap the kernels before it (programmatic dependent
                     // launch): its prologue reads Bw and bias before they finish
};
enum { EPI_NONE = 0, EPI_GELU = 1, EPI_RESID = 2 };

cudaError_t launch_gemm(const GemmArgs &a, int load_mode, int store_mode, DeviceStatus st,
                        cudaStream_t stream);
// Plain GEMM with 32-wide K blocks in the 64-byte-swizzled layout (tests the
// layout the fused kernel uses).
cudaError_t launch_gemm_sw64(const GemmArgs &a, DeviceStatus st, cudaStream_t stream);
// Plain GEMM with the A operand staged in TMEM (K <= 128, N <= 256): tests the
// TMEM-A MMA form.
cudaError_t launch_gemm_ts_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream);
// Plain GEMM with B given [K, N] (N-major, N = 32 or 64, K <= 128): tests the
// MN-major 64-byte-swizzled B operand form.
cudaError_t launch_gemm_mn_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream);
// Lane-masked MMA forms: rows 0..63 of each 128-row block against Bw[0:N], rows
// 64..127 against Bw[N:2N], A from shared memory (D columns 0..N-1) and from
// TMEM (D columns N..2N-1); D is [rows, 2N].
cudaError_t launch_gemm_pair_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream);

struct AttnArgs {
    const bf16 *qkv;      // [T, 3C] window order
    bf16 *attn;           // [T, C] window order (token order with o_token_order)
    const bf16 *table;    // [(2M-1)^2, heads]
    const float *tau;     // [heads] (V2)
    int heads, mode;      // mode 0 = V1, 1 = V2
    Geom g;
    float *lse;           // windows of more than 64 tokens, not null: log2 of each row's softmax
                          // normaliser over the log2-scaled logits, [T, heads] (window order)
    int o_token_order;    // windows of more than 64 tokens: write attn in token order
    int overlap;          // launched to overlap the kernels before it (programmatic dependent
                          // launch): its prologue reads table and tau before they finish
};

cudaError_t launch_attention(const AttnArgs &a, DeviceStatus st, cudaStream_t stream);
// The persistent large-window kernel (attn_window.cu): M = 12, 16, 20, 24 and
// every head's bias table within shared memory.
bool attn_window_supported(int M, int heads);
cudaError_t launch_attn_window(const AttnArgs &a, DeviceStatus st, cudaStream_t stream);

struct Fp32Args {
    const float *x, *Wqkv, *bqkv, *table, *tau, *Wproj, *bproj;
    float *out;
    int heads, mode;
    Geom g;
};

// fp32 block, one CTA per window; returns cudaErrorInvalidConfiguration if
// the window does not fit in shared memory.
cudaError_t launch_fp32_block(const Fp32Args &a, cudaStream_t stream);
size_t fp32_block_smem_bytes(int N, int C);

// The whole block in one persistent kernel (windows of <= 64 tokens, C = 64, 96 or 128).
bool fused_supported(int M, int C, int heads);
// With the transformer block's LayerNorm (gamma ln_g, beta ln_b) and residual
// folded in: fold 1 = pre-norm (V1), out = x + attn(LN(x)); 2 = residual
// post-norm (V2), out = x + LN(attn(x)); 0 = attn(x) alone.
bool fused_fold_supported(int M, int C, int heads, int fold);
// The same through a forward handle (its path choice, status word and wait
// limit); SWIN_WATTN_EUNSUPPORTED where that handle would not fuse the grid.
int attn_forward_folded(::swin_wattn_s *h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        const void *bias_table, const float *logit_scale, const void *Wproj, const void *bproj,
                        const void *ln_g, const void *ln_b, int fold, void *out, cudaStream_t stream);
// The block's MLP sub-layer in one kernel (hidden activation kept on chip),
// on the residual stream z [T, C]: out = z + GELU(LN(z) W1^T + b1) W2^T + b2
// (V1 pre-norm, post false) or out = z + LN(GELU(z W1^T + b1) W2^T + b2) (V2,
// post true); LN with gain ln_g and shift ln_b; W1 [R, C], W2 [C, R].  Where
// mlp_fused_supported(C, R).
bool mlp_fused_supported(int C, int R);
cudaError_t launch_mlp_fused(const bf16 *z, const bf16 *W1, const bf16 *b1, const bf16 *W2, const bf16 *b2,
                             const bf16 *ln_g, const bf16 *ln_b, bool post, bf16 *out, int64_t T, int C, int R,
                             DeviceStatus st, cudaStream_t stream, int overlap = 0);

// sched: two device ints, zero before the first launch (the kernel's tile
// counter; each launch leaves them zero); one launch at a time per pair.
cudaError_t launch_fused(const bf16 *x, const bf16 *Wqkv, const bf16 *bqkv, const bf16 *table, const float *tau,
                         const bf16 *Wproj, const bf16 *bproj, bf16 *out, int mode, const Geom &g, DeviceStatus st,
                         int *sched, cudaStream_t stream, const bf16 *ln_g = nullptr, const bf16 *ln_b = nullptr,
                         int fold = 0, int overlap = 0);

// Tensor map over a row-major bf16 matrix [rows, cols] (16-byte aligned base,
// cols * 2 a multiple of 16): boxes of 32 columns x box_rows rows (<= 256),
// 64-byte swizzle in shared memory, zero fill past the last row.  L2 fetches
// are promoted to 128 bytes, or kept at 64 (promote128 false) when the
// neighbouring 64 bytes of a row are not read soon after.
cudaError_t make_tensor_map_sw64(CUtensorMap *map, const void *ptr, int64_t rows, int cols, int box_rows,
                                 bool promote128 = true);
// Tensor map over a row-major bf16 matrix [rows, cols] with row stride ld
// (elements): boxes of 64 columns x box_rows rows, 128-byte swizzle, zero
// fill past the last row or column.
cudaError_t make_tensor_map_sw128(CUtensorMap *map, const void *ptr, int64_t rows, int cols, int64_t ld,
                                  int box_rows);
// Tensor map over a bf16 image batch [rows, width, cols] (rows = B*H image rows,
// width = W, cols = C; strides multiples of 16 bytes): boxes of 32 channels x
// box_w tokens x box_h image rows, 64-byte swizzle, zero fill outside.
cudaError_t make_tensor_map_sw64_3d(CUtensorMap *map, const void *ptr, int64_t rows, int width, int cols, int box_w,
                                    int box_h);

cudaError_t launch_cpb_table(const float *W1, const float *b1, const float *W2, int hidden, int M,
                             int heads, bool out_bf16, void *table, cudaStream_t stream);

// G's weight gradients from its table gradient (fp32; heads <= 16).
cudaError_t launch_cpb_backward(const float *W1, const float *b1, const float *W2, const float *dtable, int hidden,
                                int M, int heads, float *dW1, float *db1, float *dW2, cudaStream_t stream);

cudaError_t launch_watchdog(DeviceStatus st, cudaStream_t stream);

// ---- backward (V1) ----------------------------------------------------------
// dW [n_out, n_in] = G^T X and db [n_out] = the column sums of G (fp32,
// overwritten; db may be null) for bf16 row-major G [T, n_out] and X [T,
// n_in] (n_in a multiple of 32, n_out of 8): split-K tcgen05 GEMM into
// `workspace` (wgrad_workspace_bytes), then a fixed-order sum; three
// launches.  overlap: each of the three may start while the kernel before it
// finishes (programmatic dependent launch); they touch global memory only
// after it has completed.
size_t wgrad_workspace_bytes(int n_out, int n_in, int64_t T);
cudaError_t launch_wgrad(const bf16 *G, int n_out, const bf16 *X, int n_in, int64_t T, float *dW, float *db,
                         float *workspace, DeviceStatus st, cudaStream_t stream, int overlap = 0);
// out [cols, rows] = in [rows, cols]^T.
cudaError_t launch_transpose(const bf16 *in, bf16 *out, int rows, int cols, cudaStream_t stream);
// Windows of <= 64 tokens and 32 channels per head.
bool attn_backward_supported(int M, int C, int heads);
// From qkv [T, 3C] and do [T, C] (window order): the attention output
// attn [T, C] and dqkv [T, 3C] in token order, and dtable += ([(2M-1)^2,
// heads] fp32).  v2: qkv holds unit-length q and k, norms [T, 2 heads] their
// norms (the QKV GEMM's), tau [heads]; dqkv is then the gradient of the raw
// q and k, and dtau += ([heads] fp32).  overlap as for launch_wgrad (the
// prologue reads no global memory).
cudaError_t launch_attn_backward(const bf16 *qkv, const bf16 *dO, const bf16 *table, const float *tau, int heads,
                                 int v2, const Geom &g, bf16 *attn, bf16 *dqkv, float *dtable, const float *norms,
                                 float *dtau, DeviceStatus st, cudaStream_t stream, int overlap = 0);
// Windows of more than 64 tokens (up to 24 x 24) and 32 channels per head.
bool attn_flash_backward_supported(int M, int C, int heads);
// The same gradients for large windows from the forward's outputs: attn
// [T, C] (token order) and lse [T, heads] (window order; log2 of each row's
// softmax normaliser over the log2-scaled logits).  D [T, heads] is
// scratch; dq_acc [T, C] fp32 must be zero on entry.  Three launches.
cudaError_t launch_attn_flash_backward(const bf16 *qkv, const bf16 *dO, const bf16 *attn, const bf16 *table,
                                       const float *tau, int heads, int v2, const Geom &g, const float *lse, float *D,
                                       const float *norms, bf16 *dqkv, float *dq_acc, float *dtable, float *dtau,
                                       DeviceStatus st, cudaStream_t stream);
// The forward attention step alone on the same kernel (windows of <= 64
// tokens): attn [T, C] (window order) = P v from qkv [T, 3C] (window order);
// v2: cosine logits over the already normalised q, k, scaled by 1/max(tau, 0.01).
cudaError_t launch_attn_forward_tc(const bf16 *qkv, const bf16 *table, const float *tau, int heads, int v2,
                                   const Geom &g, bf16 *attn, DeviceStatus st, cudaStream_t stream,
                                   int overlap = 0);

} // namespace swin
