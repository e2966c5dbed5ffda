// The whole Swin Transformer block around the shifted-window attention:
// LayerNorm, residual connections, MLP ("Swin Transformer V2" (neura.market),
// How It Works: pre-norm in the original Swin, residual post-norm in V2):
//   V1  z = x + attn(LN1(x));  y = z + MLP(LN2(z))
//   V2  z = x + LN1(attn(x));  y = z + LN2(MLP(z))
// Steps: the swin_wattn forward for attn; one LayerNorm kernel that also
// does the residual add (add-then-normalise for V1, normalise-then-add for
// V2); the MLP as one kernel that keeps the hidden activation on chip where
// its weights fit an SM's shared memory (mlp_fused.cu; V2 with its LayerNorm
// and residual), else as two tcgen05 GEMMs whose epilogues apply GELU and the
// residual add.  Where the attention is the fused kernel, LayerNorm 1 and
// the first residual are folded into it (its x tiles' prologue, V1; its
// output rows' epilogue, V2) and z is its output.
#include <cmath>
#include <new>

#include "swin_block.h"
#include "swin_wattn.h"
#include "common.cuh"
#include "ptx.cuh"

using namespace swin;

namespace {

constexpr float LN_EPS = 1e-5f;

// LayerNorm over rows of C bf16 channels.  A row is spread over `lpr` lanes
// (a power of two <= 32) of 16-byte chunks; a warp handles 32 / lpr rows.
//   flags 0: out_ln = LN(a)
//   flags 1: s = a + b (fp32, then bf16); out_sum = s; out_ln = LN(s)
//   flags 2: out_ln = b + LN(a)
// With mH > 0, row r of `a` is not stored: it is the 2 x 2 neighbourhood
// concatenation of a [B, mH, mW, C/4] image (merging step between stages):
// row r = (b, i, j) of the half-resolution grid, channel part q (of four)
// from pixel (2i + (q & 1), 2j + (q >> 1)).
template <int CPL>   // 16-byte chunks per lane
__global__ void __launch_bounds__(256) layernorm_kernel(const bf16 *a, const bf16 *b, const bf16 *gamma,
                                                        const bf16 *beta, bf16 *out_sum, bf16 *out_ln, int64_t rows,
                                                        int C, int lpr, int flags, int mH, int mW)
{
    const int lane = threadIdx.x & 31;
    const int sub = lane / lpr, li = lane % lpr;
    const int64_t row = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * (32 / lpr) + sub;
    const int chunks = C / 8;
    const bool row_ok = row < rows;
    float v[CPL][8];
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = li + k * lpr;
        const bool ok = row_ok && c < chunks;
#pragma unroll
        for (int e = 0; e < 8; ++e) v[k][e] = 0.f;
        if (ok) {
            const bf16 *src = a + row * C + c * 8;
            if (mH > 0) {
                const int Cs = C / 4, cps = Cs / 8;   // source channels, 16-byte chunks per source pixel
                const int q = c / cps, cc = c - q * cps;
                const int Wh = mW / 2, Hh = mH / 2;
                const int64_t bi = row / ((int64_t)Hh * Wh);
                const int rem = (int)(row - bi * Hh * Wh);
                const int i = rem / Wh, j = rem - (rem / Wh) * Wh;
                src = a + ((bi * mH + 2 * i + (q & 1)) * (int64_t)mW + 2 * j + (q >> 1)) * Cs + cc * 8;
            }
            const uint4 ua = *reinterpret_cast<const uint4 *>(src);
            const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16x2(wa[e]);
                v[k][2 * e] = f.x;
                v[k][2 * e + 1] = f.y;
            }
            if (flags == 1) {
                const uint4 ub = *reinterpret_cast<const uint4 *>(b + row * C + c * 8);
                const uint32_t wb[4] = {ub.x, ub.y, ub.z, ub.w};
                uint32_t ws[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = unpack_bf16x2(wb[e]);
                    ws[e] = pack_bf16x2(v[k][2 * e] + f.x, v[k][2 * e + 1] + f.y);
                    // the stored (rounded) sum is what the LayerNorm sees
                    const float2 r = unpack_bf16x2(ws[e]);
                    v[k][2 * e] = r.x;
                    v[k][2 * e + 1] = r.y;
                }
                if (out_sum) *reinterpret_cast<uint4 *>(out_sum + row * C + c * 8) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sum += v[k][e];
        }
    }
    // mean and (biased) variance over the row's lanes
    for (int o = lpr / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float mean = sum / (float)C;
    float sq = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = li + k * lpr;
        if (row_ok && c < chunks) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = v[k][e] - mean;
                sq = fmaf(d, d, sq);
            }
        }
    }
    for (int o = lpr / 2; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const float rstd = rsqrtf(sq / (float)C + LN_EPS);
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const int c = li + k * lpr;
        if (!(row_ok && c < chunks)) continue;
        const uint4 ug = *reinterpret_cast<const uint4 *>(gamma + c * 8);
        const uint4 ub = *reinterpret_cast<const uint4 *>(beta + c * 8);
        const uint32_t wg[4] = {ug.x, ug.y, ug.z, ug.w}, wbt[4] = {ub.x, ub.y, ub.z, ub.w};
        float r[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 g = unpack_bf16x2(wg[e]), bt = unpack_bf16x2(wbt[e]);
            r[2 * e] = (v[k][2 * e] - mean) * rstd * g.x + bt.x;
            r[2 * e + 1] = (v[k][2 * e + 1] - mean) * rstd * g.y + bt.y;
        }
        if (flags == 2) {
            const uint4 ur = *reinterpret_cast<const uint4 *>(b + row * C + c * 8);
            const uint32_t wr[4] = {ur.x, ur.y, ur.z, ur.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_bf16x2(wr[e]);
                r[2 * e] += f.x;
                r[2 * e + 1] += f.y;
            }
        }
        *reinterpret_cast<uint4 *>(out_ln + row * C + c * 8) =
            make_uint4(pack_bf16x2(r[0], r[1]), pack_bf16x2(r[2], r[3]), pack_bf16x2(r[4], r[5]),
                       pack_bf16x2(r[6], r[7]));
    }
}

cudaError_t launch_layernorm(const bf16 *a, const bf16 *b, const bf16 *gamma, const bf16 *beta, bf16 *out_sum,
                             bf16 *out_ln, int64_t rows, int C, int flags, cudaStream_t stream, int mH = 0, int mW = 0)
{
    // lanes per row: a power of two with at least three 16-byte chunks per
    // lane (several loads in flight per thread), at most 32; a row's lanes
    // reduce its statistics by shuffles
    const int chunks = C / 8;
    int lpr = 1;
    while (lpr < 32 && 2 * lpr * 3 <= chunks) lpr <<= 1;
    const int cpl = (chunks + lpr - 1) / lpr;
    const int rows_per_block = (256 / 32) * (32 / lpr);
    const unsigned grid = (unsigned)((rows + rows_per_block - 1) / rows_per_block);
    if (grid == 0) return cudaSuccess;
#define SWIN_LN_CASE(n)                                                                                       \
    case n:                                                                                                   \
        layernorm_kernel<n><<<grid, 256, 0, stream>>>(a, b, gamma, beta, out_sum, out_ln, rows, C, lpr, flags, mH, mW); \
        break;
    switch (cpl) {
        SWIN_LN_CASE(1)
        SWIN_LN_CASE(2)
        SWIN_LN_CASE(3)
        SWIN_LN_CASE(4)
        SWIN_LN_CASE(5)
        SWIN_LN_CASE(6)
        SWIN_LN_CASE(7)
        SWIN_LN_CASE(8)
    default:
        return cudaErrorInvalidValue;
    }
#undef SWIN_LN_CASE
    return cudaGetLastError();
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SWIN_WATTN_OK : SWIN_WATTN_ECUDA; }

} // namespace

struct swin_block_s {
    swin_wattn_t attn;
    int C, heads, M, shift, mode, ratio;
    int *d_err;
    void *ws;   // z, t1, t2 [T, C] and m1 [T, rC], bf16
    size_t ws_bytes;
    int last_launches;   // of the last forward
    int overlap;         // SWIN_BLOCK_OPT_OVERLAP_CALLS
};

extern "C" {

int swin_block_create(swin_block_t *out, int C, int heads, int M, int shift, int mode, int mlp_ratio)
{
    if (!out) return SWIN_WATTN_EINVAL;
    *out = nullptr;
    if (mode & SWIN_WATTN_FP32) return SWIN_WATTN_EUNSUPPORTED;
    if (mlp_ratio < 1 || mlp_ratio > 8 || C <= 0 || C % 16 || C > 2048) return SWIN_WATTN_EINVAL;
    swin_wattn_t attn = nullptr;
    int rc = swin_wattn_create(&attn, C, heads, M, shift, mode);
    if (rc != SWIN_WATTN_OK) return rc;
    swin_block_s *h = new (std::nothrow) swin_block_s{};
    if (!h) {
        swin_wattn_destroy(attn);
        return SWIN_WATTN_ENOMEM;
    }
    h->attn = attn;
    h->C = C;
    h->heads = heads;
    h->M = M;
    h->shift = shift;
    h->mode = mode;
    h->ratio = mlp_ratio;
    if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess || cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        swin_wattn_destroy(attn);
        delete h;
        return SWIN_WATTN_ENOMEM;
    }
    *out = h;
    return SWIN_WATTN_OK;
}

int swin_block_last_launches(swin_block_t h) { return h ? h->last_launches : -1; }

int swin_block_set_option(swin_block_t h, int option, int64_t value)
{
    if (!h) return SWIN_WATTN_EINVAL;
    switch (option) {
    case SWIN_BLOCK_OPT_OVERLAP_CALLS: {
        if (value < 0 || value > 1) return SWIN_WATTN_EINVAL;
        const int rc = swin_wattn_set_option(h->attn, SWIN_WATTN_OPT_OVERLAP_CALLS, value);
        if (rc != SWIN_WATTN_OK) return rc;
        h->overlap = (int)value;
        return SWIN_WATTN_OK;
    }
    default:
        return SWIN_WATTN_EINVAL;
    }
}

int swin_block_destroy(swin_block_t h)
{
    if (!h) return SWIN_WATTN_OK;
    ws_free(&h->ws, &h->ws_bytes);
    if (h->d_err) cudaFree(h->d_err);
    swin_wattn_destroy(h->attn);
    delete h;
    return SWIN_WATTN_OK;
}

int swin_block_sync_status(swin_block_t h, swin_stream_t stream)
{
    if (!h) return SWIN_WATTN_EINVAL;
    int rc = swin_wattn_sync_status(h->attn, stream);
    if (rc != SWIN_WATTN_OK) return rc;
    int err = 0;
    if (cudaMemcpy(&err, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SWIN_WATTN_ECUDA;
    if (err) {
        if (cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) return SWIN_WATTN_ECUDA;
        return SWIN_WATTN_ETIMEOUT;
    }
    return SWIN_WATTN_OK;
}

int swin_block_forward(swin_block_t h, const void *x, int B, int H, int W, const swin_block_params *p, void *out,
                       swin_stream_t stream)
{
    if (!h || !p || !x || !out) return SWIN_WATTN_EINVAL;
    if (B < 0 || H <= 0 || W <= 0 || H % h->M || W % h->M) return SWIN_WATTN_EINVAL;
    const int C = h->C, R = h->ratio * C;
    const int64_t T = (int64_t)B * H * W;
    if (T * C > ((int64_t)1 << 40)) return SWIN_WATTN_EINVAL;
    const void *req[] = {x, out, p->ln1_gamma, p->ln1_beta, p->Wqkv, p->Wproj, p->ln2_gamma, p->ln2_beta, p->W1, p->W2};
    for (const void *q : req)
        if (!q || !aligned16(q)) return SWIN_WATTN_EINVAL;
    const void *opt[] = {p->bqkv, p->bproj, p->b1, p->b2, p->bias_table, p->logit_scale};
    for (const void *q : opt)
        if (q && !aligned16(q)) return SWIN_WATTN_EINVAL;
    {
        const char *xb = (const char *)x, *ob = (const char *)out;
        const int64_t bytes = T * C * 2;
        if (xb < ob + bytes && ob < xb + bytes) return SWIN_WATTN_EINVAL;
    }
    h->last_launches = 0;
    if (B == 0) return SWIN_WATTN_OK;
    const size_t need = (size_t)T * (3 * C + R) * 2;
    int wrc = ws_ensure(&h->ws, &h->ws_bytes, need);
    if (wrc) return wrc;
    cudaStream_t s = (cudaStream_t)stream;
    bf16 *z = (bf16 *)h->ws, *t1 = z + T * C, *t2 = t1 + T * C, *m1 = t2 + T * C;
    const bf16 *xx = (const bf16 *)x;
    bf16 *yy = (bf16 *)out;
    const Geom g = make_geom(B, H, W, C, h->M, h->shift);
    const DeviceStatus st{h->d_err, 2000000000ull};
    auto gemm = [&](const bf16 *A, int K, const void *Bw, const void *bias, bf16 *D, int N, int epi,
                    const bf16 *Rm) {
        GemmArgs a{};
        a.A = A;
        a.lda = K;
        a.Bw = (const bf16 *)Bw;
        a.bias = (const bf16 *)bias;
        a.D = D;
        a.ldd = N;
        a.rows = T;
        a.N = N;
        a.K = K;
        a.g = g;
        a.epi = epi;
        a.R = Rm;
        a.ldr = N;
        return launch_gemm(a, LOAD_PLAIN, STORE_PLAIN, st, s);
    };
    const bf16 *g1 = (const bf16 *)p->ln1_gamma, *be1 = (const bf16 *)p->ln1_beta;
    const bf16 *g2 = (const bf16 *)p->ln2_gamma, *be2 = (const bf16 *)p->ln2_beta;
    int rc;
    cudaError_t e;
    // Where the attention runs as the fused kernel, LayerNorm 1 and the first
    // residual go into it (V1: LN of its x tiles before the QKV MMAs, x added
    // to its output rows; V2: LN of its output rows, then x added), and z
    // comes straight out of it.
    const bool v1 = (h->mode & 0xf) == SWIN_WATTN_V1;
    // The MLP sub-layer on the residual stream z, out = z + MLP(LN2(z)) (V1) or
    // z + LN2(MLP(z)) (V2): one kernel (LayerNorm 2 folded in, the hidden
    // activation kept on chip) where the weights fit its shared memory, else
    // LayerNorm 2 (V1; unless ln2_done: t1 already holds it) and two GEMMs
    // (GELU and residual epilogues; V2 a LayerNorm + residual pass after them,
    // t1 as scratch).
    h->last_launches = 0;
    auto mlp = [&](bool ln2_done) -> cudaError_t {
        if (mlp_fused_supported(C, R)) {
            h->last_launches += 1;
            return launch_mlp_fused(z, (const bf16 *)p->W1, (const bf16 *)p->b1, (const bf16 *)p->W2,
                                    (const bf16 *)p->b2, g2, be2, !v1, yy, T, C, R, st, s, h->overlap);
        }
        cudaError_t e2;
        if (v1) {
            if (!ln2_done) {
                h->last_launches += 1;
                if ((e2 = launch_layernorm(z, nullptr, g2, be2, nullptr, t1, T, C, 0, s)) != cudaSuccess) return e2;
            }
            h->last_launches += 2;
            if ((e2 = gemm(t1, C, p->W1, p->b1, m1, R, EPI_GELU, nullptr)) != cudaSuccess) return e2;
            return gemm(m1, R, p->W2, p->b2, yy, C, EPI_RESID, z);
        }
        h->last_launches += 3;
        if ((e2 = gemm(z, C, p->W1, p->b1, m1, R, EPI_GELU, nullptr)) != cudaSuccess) return e2;
        if ((e2 = gemm(m1, R, p->W2, p->b2, t1, C, EPI_NONE, nullptr)) != cudaSuccess) return e2;
        return launch_layernorm(t1, z, g2, be2, nullptr, yy, T, C, 2, s);
    };
    rc = attn_forward_folded(h->attn, x, B, H, W, p->Wqkv, p->bqkv, p->bias_table, p->logit_scale, p->Wproj, p->bproj,
                             g1, be1, v1 ? 1 : 2, z, s);
    if (rc == SWIN_WATTN_OK) {
        h->last_launches = 1;   // the folded attention
        if ((e = mlp(false)) != cudaSuccess) return cuda_status(e);
        return ws_check(h->ws, s);
    }
    if (rc != SWIN_WATTN_EUNSUPPORTED) return rc;
    h->last_launches = 2;   // the two LayerNorm passes around the attention, plus its own and the MLP's
    if (v1) {
        if ((e = launch_layernorm(xx, nullptr, g1, be1, nullptr, t1, T, C, 0, s)) != cudaSuccess) return cuda_status(e);
        rc = swin_wattn_forward(h->attn, t1, B, H, W, p->Wqkv, p->bqkv, p->bias_table, p->logit_scale, p->Wproj,
                                p->bproj, t2, stream);
        if (rc != SWIN_WATTN_OK) return rc;
        h->last_launches += swin_wattn_last_launches(h->attn);
        if ((e = launch_layernorm(t2, xx, g2, be2, z, t1, T, C, 1, s)) != cudaSuccess) return cuda_status(e);
        if ((e = mlp(true)) != cudaSuccess) return cuda_status(e);
    } else {
        rc = swin_wattn_forward(h->attn, x, B, H, W, p->Wqkv, p->bqkv, p->bias_table, p->logit_scale, p->Wproj,
                                p->bproj, t2, stream);
        if (rc != SWIN_WATTN_OK) return rc;
        h->last_launches += swin_wattn_last_launches(h->attn);
        if ((e = launch_layernorm(t2, xx, g1, be1, nullptr, z, T, C, 2, s)) != cudaSuccess) return cuda_status(e);
        h->last_launches -= 1;   // (V2: one LayerNorm pass before the MLP)
        if ((e = mlp(true)) != cudaSuccess) return cuda_status(e);
    }
    return ws_check(h->ws, s);
}

int swin_block_test_layernorm(const void *a, const void *b, const void *gamma, const void *beta, void *out_sum,
                              void *out_ln, int rows, int C, int flags, swin_stream_t stream)
{
    if (!a || !gamma || !beta || !out_ln || rows < 0 || C <= 0 || C % 8 || C > 2048 || flags < 0 || flags > 2)
        return SWIN_WATTN_EINVAL;
    if (flags != 0 && !b) return SWIN_WATTN_EINVAL;
    const void *ps[] = {a, b, gamma, beta, out_sum, out_ln};
    for (const void *q : ps)
        if (q && !aligned16(q)) return SWIN_WATTN_EINVAL;
    if (rows == 0) return SWIN_WATTN_OK;
    return cuda_status(launch_layernorm((const bf16 *)a, (const bf16 *)b, (const bf16 *)gamma, (const bf16 *)beta,
                                        (bf16 *)out_sum, (bf16 *)out_ln, rows, C, flags, (cudaStream_t)stream));
}

int swin_stage_norm(const void *x, int rows, int C, const void *gamma, const void *beta, void *out, swin_stream_t stream)
{
    if (!x || !gamma || !beta || !out || rows < 0 || C <= 0 || C % 8 || C > 2048) return SWIN_WATTN_EINVAL;
    const void *ps[] = {x, gamma, beta, out};
    for (const void *q : ps)
        if (!aligned16(q)) return SWIN_WATTN_EINVAL;
    const char *xb = (const char *)x, *ob = (const char *)out;
    const int64_t bytes = (int64_t)rows * C * 2;
    if (xb != ob && xb < ob + bytes && ob < xb + bytes) return SWIN_WATTN_EINVAL;
    if (rows == 0) return SWIN_WATTN_OK;
    return cuda_status(launch_layernorm((const bf16 *)x, nullptr, (const bf16 *)gamma, (const bf16 *)beta, nullptr,
                                        (bf16 *)out, rows, C, 0, (cudaStream_t)stream));
}

// ---- merging step between stages ------------------------------------------------

} // extern "C"

struct swin_merge_s {
    int C;
    int *d_err;
    void *ws;   // the normalised 4C-channel rows, bf16
    size_t ws_bytes;
};

extern "C" {

int swin_merge_create(swin_merge_t *out, int C)
{
    if (!out) return SWIN_WATTN_EINVAL;
    *out = nullptr;
    if (C <= 0 || C % 8 || 4 * C > 2048) return SWIN_WATTN_EINVAL;
    swin_merge_s *h = new (std::nothrow) swin_merge_s{};
    if (!h) return SWIN_WATTN_ENOMEM;
    h->C = C;
    if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess || cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return SWIN_WATTN_ENOMEM;
    }
    *out = h;
    return SWIN_WATTN_OK;
}

int swin_merge_destroy(swin_merge_t h)
{
    if (!h) return SWIN_WATTN_OK;
    ws_free(&h->ws, &h->ws_bytes);
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return SWIN_WATTN_OK;
}

int swin_merge_forward(swin_merge_t h, const void *x, int B, int H, int W, const void *gamma, const void *beta,
                       const void *Wm, void *out, swin_stream_t stream)
{
    if (!h || !x || !gamma || !beta || !Wm || !out) return SWIN_WATTN_EINVAL;
    if (B < 0 || H <= 0 || W <= 0 || H % 2 || W % 2) return SWIN_WATTN_EINVAL;
    const void *ps[] = {x, gamma, beta, Wm, out};
    for (const void *q : ps)
        if (!aligned16(q)) return SWIN_WATTN_EINVAL;
    const int C = h->C;
    const int64_t rows = (int64_t)B * (H / 2) * (W / 2);
    if (rows * 4 * C > ((int64_t)1 << 40)) return SWIN_WATTN_EINVAL;
    {
        const char *xb = (const char *)x, *ob = (const char *)out;
        const int64_t xbytes = rows * 4 * C * 2, obytes = rows * 2 * C * 2;
        if (xb < ob + obytes && ob < xb + xbytes) return SWIN_WATTN_EINVAL;
    }
    if (B == 0) return SWIN_WATTN_OK;
    const size_t need = (size_t)rows * 4 * C * 2;
    int wrc = ws_ensure(&h->ws, &h->ws_bytes, need);
    if (wrc) return wrc;
    cudaStream_t s = (cudaStream_t)stream;
    bf16 *u = (bf16 *)h->ws;
    cudaError_t e = launch_layernorm((const bf16 *)x, nullptr, (const bf16 *)gamma, (const bf16 *)beta, nullptr, u,
                                     rows, 4 * C, 0, s, H, W);
    if (e != cudaSuccess) return cuda_status(e);
    GemmArgs a{};
    a.A = u;
    a.lda = 4 * C;
    a.Bw = (const bf16 *)Wm;
    a.D = (bf16 *)out;
    a.ldd = 2 * C;
    a.rows = rows;
    a.N = 2 * C;
    a.K = 4 * C;
    a.g = make_geom(1, 1, 1, 2 * C, 1, 0);
    const int rc = cuda_status(launch_gemm(a, LOAD_PLAIN, STORE_PLAIN, DeviceStatus{h->d_err, 2000000000ull}, s));
    return rc ? rc : ws_check(h->ws, s);
}

} // extern "C"
