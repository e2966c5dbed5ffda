// Backward pass of the shifted-window attention block, V1 ("Boosting Swin
// Transformer Speed", Training Optimization: the fused MHA kernel and the
// index-mapping kernels of window partition, shift and reverse, whose
// gradients training needs).  With the forward in window order
//   xs = gather(x), qkv = xs Wqkv^T + bqkv, S = q k^T / sqrt(d) + B[idx] (mask),
//   P = softmax(S), o = P v, y = o Wproj^T + bproj, out = scatter(y)
// and dy the gradient of out:
//   dy_w = gather(dy), dWproj = dy_w^T o, dbproj = sum dy_w, do = dy_w Wproj,
//   dP = do v^T, dS = P (dP - rowsum(P dP)), dq = dS k / sqrt(d),
//   dk = dS^T q / sqrt(d), dv = P^T do, dB[idx(i,j)] += dS_ij,
//   dWqkv = dqkv^T xs, dbqkv = sum dqkv, dx = scatter(dqkv Wqkv).
// This file holds the gathers, a weight transpose, column sums and the
// attention backward (which also yields o, so the forward attention is not
// run again); the GEMMs are launched by the caller.
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

// out[r, :] = in[token(r), :] for window-order rows r (16-byte chunks).
__global__ void gather_rows_kernel(const bf16 *in, bf16 *out, Geom g, int C)
{
    const int cpr = C / 8;
    const int64_t total = g.T * cpr;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = q / cpr;
        const int c = (int)(q - r * cpr);
        const int64_t tok = window_row_to_token(g, r);
        *reinterpret_cast<uint4 *>(out + r * C + c * 8) = *reinterpret_cast<const uint4 *>(in + tok * C + c * 8);
    }
}

// out [cols, rows] = in [rows, cols]^T (bf16), 32 x 32 tiles through shared memory.
__global__ void transpose_kernel(const bf16 *in, bf16 *out, int rows, int cols)
{
    __shared__ bf16 tile[32][34];
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = in[(int64_t)r * cols + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) out[(int64_t)c * rows + r] = tile[threadIdx.x][i];
    }
}

// out[n] += sum over rows of in[row, n] in fp32.  A thread owns one 16-byte
// chunk (8 columns) and a row offset, so that a CTA reads whole rows with
// coalesced 16-byte loads; the row offsets' partial sums meet in shared
// memory and leave with one atomic add per column and CTA.
__global__ void colsum_kernel(const bf16 *in, int64_t rows, int N, float *out)
{
    extern __shared__ float part[]; // [rows per iteration][N]
    const int cpr = N / 8, rpi = blockDim.x / cpr;
    const int c = threadIdx.x % cpr, rr = threadIdx.x / cpr;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    if (rr < rpi) {
        for (int64_t r = (int64_t)blockIdx.x * rpi + rr; r < rows; r += (int64_t)gridDim.x * rpi) {
            const uint4 u = *reinterpret_cast<const uint4 *>(in + r * N + c * 8);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = unpack_bf16x2(w[k]);
                acc[2 * k] += f.x;
                acc[2 * k + 1] += f.y;
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) part[rr * N + c * 8 + k] = acc[k];
    }
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        float s = 0.f;
        for (int q = 0; q < rpi; ++q) s += part[q * N + n];
        atomicAdd(&out[n], s);
    }
}

// ---- attention backward on the tensor cores ------------------------------------
//
// A unit is one head of two consecutive windows, stacked into 128 rows (window
// 2p in rows 0..63, window 2p+1 in rows 64..127, tokens past N zero).  With the
// head's q, k, v, do of both windows in shared memory ([128 rows][32 ch],
// 64-byte swizzle):
//   S = q k^T and dP = do v^T                  (M = 128, N = 128, K = 32)
// a thread per row turns its window's half of the two rows into P and
// dS = P (dP - rowsum(P dP)) (bf16, block-diagonal: the other window's half
// stays zero), then
//   o = P v,  dq = dS k,  dv = P^T do,  dk = dS^T q   (M = 128, N = 32, K = 128)
// where P^T and dS^T are the same shared-memory tiles read M-major.  Cross-
// window products vanish because the off-diagonal blocks are zero.
constexpr int TB_THREADS = 128;

struct TbLayout {
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t Q = 0, K = 8192, V = 16384, DO = 24576; // [128][64 B] tiles
    static constexpr uint32_t P = 32768, DS = 65536;                   // 4 panels of [128][32 keys]
    static constexpr uint32_t KOFS = 98304;                            // int [64]
    static constexpr uint32_t REG = KOFS + 256;                         // int [128]
    static constexpr uint32_t TAB = REG + 512;                          // float [heads * L^2] (padded to 4)
    __host__ __device__ static uint32_t hl(int heads, int M) { return ((uint32_t)heads * (2 * M - 1) * (2 * M - 1) + 3u) & ~3u; }
    __host__ __device__ static uint32_t dtab(int heads, int M) { return TAB + 4 * hl(heads, M); }
    __host__ __device__ static uint32_t bar(int heads, int M) { return dtab(heads, M) + 4 * hl(heads, M); }
    static size_t bytes(int heads, int M) { return (size_t)bar(heads, M) + 16 + 1024; }
};

__device__ __forceinline__ int bw_region(const Geom &g, int wi, int wj, int t)
{
    if (g.s == 0) return 0;
    const int ti = t / g.M, tj = t - (t / g.M) * g.M;
    return 3 * shift_band(wi * g.M + ti, g.H, g.M, g.s) + shift_band(wj * g.M + tj, g.W, g.M, g.s);
}

__device__ __forceinline__ void store_row8(uint32_t dst, const float *v, float mul)
{
    const uint32_t a = pack_bf16x2(v[0] * mul, v[1] * mul), b = pack_bf16x2(v[2] * mul, v[3] * mul);
    const uint32_t c = pack_bf16x2(v[4] * mul, v[5] * mul), d = pack_bf16x2(v[6] * mul, v[7] * mul);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void store_global32(bf16 *dst, const float (&v)[32], float mul)
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * q] * mul, v[8 * q + 1] * mul);
        u.y = pack_bf16x2(v[8 * q + 2] * mul, v[8 * q + 3] * mul);
        u.z = pack_bf16x2(v[8 * q + 4] * mul, v[8 * q + 5] * mul);
        u.w = pack_bf16x2(v[8 * q + 6] * mul, v[8 * q + 7] * mul);
        *reinterpret_cast<uint4 *>(dst + 8 * q) = u;
    }
}

__global__ void __launch_bounds__(TB_THREADS, 2)
attn_backward_tc_kernel(const bf16 *qkv, const bf16 *dO, const bf16 *table, int heads, Geom g, bf16 *attn,
                        bf16 *dqkv, float *dtable, DeviceStatus st)
{
    extern __shared__ uint8_t smraw[];
    using Ly = TbLayout;
    uint8_t *sm = smem_align(smraw, 1024);
    const uint32_t base = smem_u32(sm);
    const int N = g.N, M = g.M, C = g.C, L = 2 * M - 1, LL = L * L;
    int *kofs = reinterpret_cast<int *>(sm + Ly::KOFS);
    int *reg = reinterpret_cast<int *>(sm + Ly::REG);
    float *tab = reinterpret_cast<float *>(sm + Ly::TAB);
    float *dtab = reinterpret_cast<float *>(sm + Ly::dtab(heads, M));
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + Ly::bar(heads, M));
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int per = g.nh * g.nw;
    const int64_t npairs = (g.nwin + 1) / 2, nunits = npairs * heads;
    const float scale = 0.17677669529663687f; // 1 / sqrt(32)
    const float log2e = 1.4426950408889634f;

    // P and dS start (and their off-diagonal blocks stay) zero
    for (int e = tid; e < 65536 / 16; e += TB_THREADS)
        *reinterpret_cast<uint4 *>(sm + Ly::P + 16 * e) = make_uint4(0, 0, 0, 0);
    for (int j = tid; j < 64; j += TB_THREADS) kofs[j] = (j / M) * L + (j % M);
    for (int e = tid; e < heads * LL; e += TB_THREADS) {
        const int h = e / LL, idx = e - h * LL;
        tab[e] = __bfloat162float(table[(int64_t)idx * heads + h]);
        dtab[e] = 0.f;
    }
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), 256);
        tmem_relinquish();
    }

    // cp.async of unit u's q, k, v, do (zero rows past N or past the last
    // window) and the shift region of this thread's row
    auto load_unit = [&](int64_t u) {
        const int64_t pair = u / heads;
        const int head = (int)(u - pair * heads);
        for (int e = tid; e < 2048; e += TB_THREADS) {
            const int r = e & 127, ch = e >> 7, tsr = ch >> 2, c = ch & 3;
            const int i = r & 63;
            const int64_t win = 2 * pair + (r >> 6);
            const bool ok = i < N && win < g.nwin;
            const int64_t row = win * N + i;
            const bf16 *src = !ok ? qkv
                              : tsr < 3 ? qkv + row * 3 * C + tsr * C + head * 32 + c * 8
                                        : dO + row * C + head * 32 + c * 8;
            cp_async16(base + (uint32_t)tsr * 8192u + sw64_offset(r, c), src, ok ? 16u : 0u);
        }
        cp_async_commit();
        const int i = tid & 63;
        const int64_t win = 2 * pair + (tid >> 6);
        int rg = -1;
        if (i < N && win < g.nwin) {
            const int rem = (int)(win % per);
            rg = bw_region(g, rem / g.nw, rem % g.nw, i);
        }
        reg[tid] = rg;
    };

    uint32_t phase = 0;
    bool failed = false;
    if (blockIdx.x < nunits) load_unit(blockIdx.x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    const int r = tid, hf = r >> 6, i = r & 63;

    for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
        const int64_t pair = u / heads;
        const int head = (int)(u - pair * heads);
        const int64_t win = 2 * pair + hf;
        const bool rv = i < N && win < g.nwin;
        cp_async_wait<0>();
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id = idesc_bf16(128, 128);
#pragma unroll
            for (int ks = 0; ks < 2; ++ks) {
                mma_bf16(tmem, desc_kmajor_sw64(base + Ly::Q + 32 * ks), desc_kmajor_sw64(base + Ly::K + 32 * ks), id,
                         ks);
                mma_bf16(tmem + 128, desc_kmajor_sw64(base + Ly::DO + 32 * ks),
                         desc_kmajor_sw64(base + Ly::V + 32 * ks), id, ks);
            }
            mma_commit(smem_u32(bar));
        }
        bool ok = mbar_wait(smem_u32(bar), phase, st.wait_ns);
        phase ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();

        // ---- P and dS of this thread's row (its window's 64 keys) ----
        {
            float s0[32], s1[32], d0[32], d1[32];
            tmem_ld32(t_lane + 64 * hf, s0);
            tmem_ld32(t_lane + 64 * hf + 32, s1);
            tmem_ld32(t_lane + 128 + 64 * hf, d0);
            tmem_ld32(t_lane + 128 + 64 * hf + 32, d1);
            tmem_wait_ld();
            const int myreg = reg[r];
            const int bi = rv ? (i / M + M - 1) * L + (i % M) + M - 1 : 0;
            const float *tb = tab + head * LL;
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float &s = j < 32 ? s0[j] : s1[j - 32];
                const bool ok_j = rv && j < N && reg[64 * hf + j] == myreg;
                s = ok_j ? fmaf(s, scale, tb[bi - kofs[j]]) : -INFINITY;
                mx = fmaxf(mx, s);
            }
            float sum = 0.f;
            const float mxl = rv ? mx * log2e : 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float &s = j < 32 ? s0[j] : s1[j - 32];
                s = ex2_approx(fmaf(s, log2e, -mxl)); // -inf -> 0
                sum += s;
            }
            const float inv = rv ? 1.0f / sum : 0.f;
            float dd = 0.f;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                float &s = j < 32 ? s0[j] : s1[j - 32];
                const float dp = j < 32 ? d0[j] : d1[j - 32];
                s *= inv;
                dd = fmaf(s, dp, dd);
            }
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float p = j < 32 ? s0[j] : s1[j - 32];
                float &d = j < 32 ? d0[j] : d1[j - 32];
                d = p * (d - dd);
            }
            // bf16 rows into the P and dS panels (keys 64*hf .. 64*hf+63)
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t off = (uint32_t)(2 * hf + q) * 8192u + sw64_offset(r, c);
                    store_row8(base + Ly::P + off, (q == 0 ? s0 : s1) + 8 * c, 1.f);
                    store_row8(base + Ly::DS + off, (q == 0 ? d0 : d1) + 8 * c, 1.f);
                }
            if (rv) {
                float *dt = dtab + head * LL;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float d = j < 32 ? d0[j] : d1[j - 32];
                    if (j < N && d != 0.f) atomicAdd(&dt[bi - kofs[j]], d);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t id_k = idesc_bf16_bmn(128, 32), id_m = idesc_bf16_amn_bmn(128, 32);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t kpan = (uint32_t)(kk >> 1) * 8192u + 32u * (kk & 1);
                mma_bf16(tmem + 0, desc_kmajor_sw64(base + Ly::P + kpan), desc_mnmajor_sw64(base + Ly::V + 1024 * kk, 8192),
                         id_k, kk);
                mma_bf16(tmem + 32, desc_kmajor_sw64(base + Ly::DS + kpan),
                         desc_mnmajor_sw64(base + Ly::K + 1024 * kk, 8192), id_k, kk);
                mma_bf16(tmem + 64, desc_mnmajor_sw64(base + Ly::DS + 1024 * kk, 8192),
                         desc_mnmajor_sw64(base + Ly::Q + 1024 * kk, 8192), id_m, kk);
                mma_bf16(tmem + 96, desc_mnmajor_sw64(base + Ly::P + 1024 * kk, 8192),
                         desc_mnmajor_sw64(base + Ly::DO + 1024 * kk, 8192), id_m, kk);
            }
            mma_commit(smem_u32(bar));
        }
        ok = mbar_wait(smem_u32(bar), phase, st.wait_ns);
        phase ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
        // q, k, v, do are free: start the next unit's loads under the epilogue
        if (u + gridDim.x < nunits) load_unit(u + gridDim.x);

        // ---- o, dq, dk, dv rows out (row r: query or key token i of window win) ----
        {
            float a[32], b[32];
            const int64_t row = win * N + i;
            tmem_ld32(t_lane + 0, a);
            tmem_ld32(t_lane + 32, b);
            tmem_wait_ld();
            if (rv) {
                store_global32(attn + row * C + head * 32, a, 1.f);
                store_global32(dqkv + row * 3 * C + head * 32, b, scale);
            }
            tmem_ld32(t_lane + 64, a);
            tmem_ld32(t_lane + 96, b);
            tmem_wait_ld();
            if (rv) {
                store_global32(dqkv + row * 3 * C + C + head * 32, a, scale);
                store_global32(dqkv + row * 3 * C + 2 * C + head * 32, b, 1.f);
            }
        }
        tc_fence_before();
        __syncthreads();
    }
    if (failed) {
        if (tid == 0) atomicOr(st.err, ERR_TIMEOUT);
        cp_async_wait<0>();
    }
    __syncthreads();
    for (int e = tid; e < heads * LL; e += TB_THREADS) {
        const int h = e / LL, idx = e - h * LL;
        if (dtab[e] != 0.f) atomicAdd(&dtable[(int64_t)idx * heads + h], dtab[e]);
    }
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

} // namespace

cudaError_t launch_gather_rows(const bf16 *in, bf16 *out, const Geom &g, int C, cudaStream_t stream)
{
    const int64_t total = g.T * (C / 8);
    const int64_t want = (total + 255) / 256;
    const unsigned grid = (unsigned)(want < 152 * 16 ? want : 152 * 16);
    gather_rows_kernel<<<grid, 256, 0, stream>>>(in, out, g, C);
    return cudaGetLastError();
}

cudaError_t launch_transpose(const bf16 *in, bf16 *out, int rows, int cols, cudaStream_t stream)
{
    dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32)), block(32, 8);
    transpose_kernel<<<grid, block, 0, stream>>>(in, out, rows, cols);
    return cudaGetLastError();
}

cudaError_t launch_colsum(const bf16 *in, int64_t rows, int N, float *out, cudaStream_t stream)
{
    if (N <= 0 || N % 8 || N > 8 * 256) return cudaErrorInvalidValue;
    if (rows <= 0) return cudaSuccess;
    const int threads = 256, rpi = threads / (N / 8);
    const int64_t want = (rows + rpi - 1) / rpi;
    const unsigned grid = (unsigned)(want < 152 * 8 ? want : 152 * 8);
    colsum_kernel<<<grid, threads, (size_t)rpi * N * 4, stream>>>(in, rows, N, out);
    return cudaGetLastError();
}

bool attn_backward_supported(int M, int C, int heads)
{
    return M * M <= 64 && C == heads * 32 && TbLayout::bytes(heads, M) <= 227 * 1024;
}

cudaError_t launch_attn_backward(const bf16 *qkv, const bf16 *dO, const bf16 *table, int heads, const Geom &g,
                                 bf16 *attn, bf16 *dqkv, float *dtable, DeviceStatus st, cudaStream_t stream)
{
    if (!attn_backward_supported(g.M, g.C, heads)) return cudaErrorInvalidValue;
    const size_t smem = TbLayout::bytes(heads, g.M);
    cudaError_t e = cudaFuncSetAttribute(attn_backward_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    }
    const int per_sm = 2 * TbLayout::bytes(heads, g.M) + 2048 <= 228 * 1024 ? 2 : 1;
    const int64_t units = (g.nwin + 1) / 2 * heads;
    const int64_t cap = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    attn_backward_tc_kernel<<<grid, TB_THREADS, smem, stream>>>(qkv, dO, table, heads, g, attn, dqkv, dtable, st);
    return cudaGetLastError();
}

} // namespace swin
