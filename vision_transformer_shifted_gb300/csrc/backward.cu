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
// per-window attention backward; the GEMMs are launched by the caller.
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

// out[n] = sum over rows of in[row, n] in fp32: each CTA sums a strided set
// of rows into registers (a thread owns columns tid, tid + 256, ...), then
// adds its partial sums with one atomic per column.  out must be zeroed.
__global__ void colsum_kernel(const bf16 *in, int64_t rows, int N, float *out)
{
    constexpr int PER = 8; // N <= 8 * 256
    float acc[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) acc[u] = 0.f;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const bf16 *row = in + r * N;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int n = threadIdx.x + u * 256;
            if (n < N) acc[u] += __bfloat162float(row[n]);
        }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int n = threadIdx.x + u * 256;
        if (n < N) atomicAdd(&out[n], acc[u]);
    }
}

// ---- attention backward, one CTA per (window, head) ----------------------------

constexpr int BW_THREADS = 256;
constexpr int NP = 64;       // padded tokens per window (N <= 64)
constexpr int HD = 32;       // channels per head
constexpr int TS = NP + 4;   // row stride of the transposed dS (keeps float4 alignment)

struct BwLayout {
    // floats: qT, kT, vT, doT [HD][NP]; q, k, do [NP][HD]; P, dS [NP][NP];
    // dST [NP][TS]; tab, dtab [(2M-1)^2]; then region ids [NP] (int)
    static constexpr int qT = 0, kT = qT + HD * NP, vT = kT + HD * NP, doT = vT + HD * NP;
    static constexpr int q = doT + HD * NP, k = q + NP * HD, dO = k + NP * HD;
    static constexpr int P = dO + NP * HD, dS = P + NP * NP, dST = dS + NP * NP;
    static constexpr int tab = dST + NP * TS;
    static size_t bytes(int M)
    {
        const int L2 = (2 * M - 1) * (2 * M - 1);
        return (size_t)(tab + 2 * ((L2 + 3) & ~3)) * 4 + NP * 4;
    }
};

__device__ __forceinline__ int bw_region(const Geom &g, int wi, int wj, int t)
{
    if (g.s == 0) return 0;
    const int ti = t / g.M, tj = t - (t / g.M) * g.M;
    return 3 * shift_band(wi * g.M + ti, g.H, g.M, g.s) + shift_band(wj * g.M + tj, g.W, g.M, g.s);
}

__device__ __forceinline__ int rel_idx(int i, int j, int M)
{
    const int ri = i / M, ci = i - ri * M, rj = j / M, cj = j - rj * M;
    return (ri - rj + M - 1) * (2 * M - 1) + (ci - cj + M - 1);
}

// S and P are recomputed from q, k and the table (the forward keeps neither).
// Phase 1: a thread owns a 4 x 4 block of (S, dP) over its 32 channels.
// Phase 2: a warp per row: softmax, D_i = sum_j P_ij dP_ij, dS = P (dP - D),
// the table gradient (shared-memory atomics).  Phase 3: a thread owns 4 rows
// x 2 channels of dq, dk and dv.  fp32 throughout, bf16 out.
__global__ void __launch_bounds__(BW_THREADS, 2)
attn_backward_kernel(const bf16 *qkv, const bf16 *dO, const bf16 *table, int heads, Geom g, bf16 *dqkv, float *dtable)
{
    extern __shared__ __align__(16) float sm[];
    using Ly = BwLayout;
    const int N = g.N, M = g.M, C = g.C, L = 2 * M - 1, LL = L * L;
    const int LLp = (LL + 3) & ~3;
    float *tab = sm + Ly::tab, *dtab = tab + LLp;
    int *reg = reinterpret_cast<int *>(dtab + LLp);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t win = blockIdx.x;
    const int head = blockIdx.y;
    const int per = g.nh * g.nw;
    const int rem = (int)(win % per);
    const int wi = rem / g.nw, wj = rem - (rem / g.nw) * g.nw;
    const float scale = 0.17677669529663687f; // 1 / sqrt(32)

    // stage q, k, v, do of the head (zero rows past N) in both layouts
    for (int e = tid; e < NP * 16; e += BW_THREADS) {
        const int i = e & (NP - 1), chunk = e >> 6; // chunk: tensor (q, k, v, do) x 4 groups of 8 channels
        const int tsr = chunk >> 2, c0 = (chunk & 3) * 8;
        float f[8];
        if (i < N) {
            const int64_t row = win * N + i;
            const bf16 *src = tsr < 3 ? qkv + row * 3 * C + tsr * C + head * HD + c0 : dO + row * C + head * HD + c0;
            const uint4 u = *reinterpret_cast<const uint4 *>(src);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[t]));
                f[2 * t] = p.x;
                f[2 * t + 1] = p.y;
            }
        } else {
#pragma unroll
            for (int t = 0; t < 8; ++t) f[t] = 0.f;
        }
        float *tr = sm + (tsr == 0 ? Ly::qT : tsr == 1 ? Ly::kT : tsr == 2 ? Ly::vT : Ly::doT);
#pragma unroll
        for (int t = 0; t < 8; ++t) tr[(c0 + t) * NP + i] = f[t];
        if (tsr != 2) {
            float *rm = sm + (tsr == 0 ? Ly::q : tsr == 1 ? Ly::k : Ly::dO) + i * HD + c0;
            *reinterpret_cast<float4 *>(rm) = make_float4(f[0], f[1], f[2], f[3]);
            *reinterpret_cast<float4 *>(rm + 4) = make_float4(f[4], f[5], f[6], f[7]);
        }
    }
    for (int i = tid; i < NP; i += BW_THREADS) reg[i] = i < N ? bw_region(g, wi, wj, i) : -1;
    for (int i = tid; i < LL; i += BW_THREADS) {
        tab[i] = __bfloat162float(table[(int64_t)i * heads + head]);
        dtab[i] = 0.f;
    }
    __syncthreads();

    // phase 1: S = q k^T scale + B (masked), dP = do v^T
    {
        const int ti = tid >> 4, tj = tid & 15;
        float s[4][4], dp[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) s[a][b] = dp[a][b] = 0.f;
#pragma unroll 4
        for (int c = 0; c < HD; ++c) {
            const float4 qa = *reinterpret_cast<const float4 *>(sm + Ly::qT + c * NP + 4 * ti);
            const float4 kb = *reinterpret_cast<const float4 *>(sm + Ly::kT + c * NP + 4 * tj);
            const float4 da = *reinterpret_cast<const float4 *>(sm + Ly::doT + c * NP + 4 * ti);
            const float4 vb = *reinterpret_cast<const float4 *>(sm + Ly::vT + c * NP + 4 * tj);
            const float qv[4] = {qa.x, qa.y, qa.z, qa.w}, kv[4] = {kb.x, kb.y, kb.z, kb.w};
            const float dv[4] = {da.x, da.y, da.z, da.w}, vv[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    s[a][b] = fmaf(qv[a], kv[b], s[a][b]);
                    dp[a][b] = fmaf(dv[a], vv[b], dp[a][b]);
                }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = 4 * ti + a;
            float sv[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int j = 4 * tj + b;
                const bool ok = i < N && j < N && reg[i] == reg[j];
                sv[b] = ok ? fmaf(s[a][b], scale, tab[rel_idx(i, j, M)]) : -INFINITY;
            }
            *reinterpret_cast<float4 *>(sm + Ly::P + i * NP + 4 * tj) = make_float4(sv[0], sv[1], sv[2], sv[3]);
            *reinterpret_cast<float4 *>(sm + Ly::dS + i * NP + 4 * tj) =
                make_float4(dp[a][0], dp[a][1], dp[a][2], dp[a][3]);
        }
    }
    __syncthreads();

    // phase 2: a warp per row; lanes own columns lane and lane + 32
    for (int i = warp; i < NP; i += BW_THREADS / 32) {
        float *Pr = sm + Ly::P + i * NP, *dSr = sm + Ly::dS + i * NP;
        if (i >= N) {
            Pr[lane] = Pr[lane + 32] = 0.f;
            dSr[lane] = dSr[lane + 32] = 0.f;
            sm[Ly::dST + lane * TS + i] = 0.f;
            sm[Ly::dST + (lane + 32) * TS + i] = 0.f;
            continue;
        }
        const float s0 = Pr[lane], s1 = Pr[lane + 32];
        float mx = fmaxf(s0, s1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // the diagonal is never masked, so mx is finite
        const float e0 = __expf(s0 - mx), e1 = __expf(s1 - mx);
        float sum = e0 + e1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.0f / sum;
        const float p0 = e0 * inv, p1 = e1 * inv;
        const float g0 = dSr[lane], g1 = dSr[lane + 32];
        float dd = p0 * g0 + p1 * g1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
        const float ds0 = p0 * (g0 - dd), ds1 = p1 * (g1 - dd);
        Pr[lane] = p0;
        Pr[lane + 32] = p1;
        dSr[lane] = ds0;
        dSr[lane + 32] = ds1;
        sm[Ly::dST + lane * TS + i] = ds0;
        sm[Ly::dST + (lane + 32) * TS + i] = ds1;
        if (lane < N && ds0 != 0.f) atomicAdd(&dtab[rel_idx(i, lane, M)], ds0);
        if (lane + 32 < N && ds1 != 0.f) atomicAdd(&dtab[rel_idx(i, lane + 32, M)], ds1);
    }
    __syncthreads();

    // phase 3: dq = dS k scale, dk = dS^T q scale, dv = P^T do
    {
        const int rg = tid >> 4, c0 = (tid & 15) * 2;
        float aq[4][2], ak[4][2], av[4][2];
#pragma unroll
        for (int a = 0; a < 4; ++a) aq[a][0] = aq[a][1] = ak[a][0] = ak[a][1] = av[a][0] = av[a][1] = 0.f;
        for (int j = 0; j < N; ++j) {
            const float4 dsT = *reinterpret_cast<const float4 *>(sm + Ly::dST + j * TS + 4 * rg);
            const float4 dsR = *reinterpret_cast<const float4 *>(sm + Ly::dS + j * NP + 4 * rg);
            const float4 pR = *reinterpret_cast<const float4 *>(sm + Ly::P + j * NP + 4 * rg);
            const float2 kk = *reinterpret_cast<const float2 *>(sm + Ly::k + j * HD + c0);
            const float2 qq = *reinterpret_cast<const float2 *>(sm + Ly::q + j * HD + c0);
            const float2 oo = *reinterpret_cast<const float2 *>(sm + Ly::dO + j * HD + c0);
            const float t4[4] = {dsT.x, dsT.y, dsT.z, dsT.w};
            const float r4[4] = {dsR.x, dsR.y, dsR.z, dsR.w};
            const float p4[4] = {pR.x, pR.y, pR.z, pR.w};
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                aq[a][0] = fmaf(t4[a], kk.x, aq[a][0]);
                aq[a][1] = fmaf(t4[a], kk.y, aq[a][1]);
                ak[a][0] = fmaf(r4[a], qq.x, ak[a][0]);
                ak[a][1] = fmaf(r4[a], qq.y, ak[a][1]);
                av[a][0] = fmaf(p4[a], oo.x, av[a][0]);
                av[a][1] = fmaf(p4[a], oo.y, av[a][1]);
            }
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int i = 4 * rg + a;
            if (i >= N) continue;
            bf16 *row = dqkv + (win * N + i) * 3 * C + head * HD + c0;
            *reinterpret_cast<uint32_t *>(row) = pack_bf16x2(aq[a][0] * scale, aq[a][1] * scale);
            *reinterpret_cast<uint32_t *>(row + C) = pack_bf16x2(ak[a][0] * scale, ak[a][1] * scale);
            *reinterpret_cast<uint32_t *>(row + 2 * C) = pack_bf16x2(av[a][0], av[a][1]);
        }
    }
    for (int i = tid; i < LL; i += BW_THREADS)
        if (dtab[i] != 0.f) atomicAdd(&dtable[(int64_t)i * heads + head], dtab[i]);
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
    if (N <= 0 || N > 8 * 256) return cudaErrorInvalidValue;
    const unsigned grid = (unsigned)(rows < 152 * 8 ? (rows > 0 ? rows : 1) : 152 * 8);
    colsum_kernel<<<grid, 256, 0, stream>>>(in, rows, N, out);
    return cudaGetLastError();
}

bool attn_backward_supported(int M, int C, int heads) { return M * M <= NP && C == heads * HD; }

cudaError_t launch_attn_backward(const bf16 *qkv, const bf16 *dO, const bf16 *table, int heads, const Geom &g,
                                 bf16 *dqkv, float *dtable, cudaStream_t stream)
{
    if (!attn_backward_supported(g.M, g.C, heads)) return cudaErrorInvalidValue;
    const size_t smem = BwLayout::bytes(g.M);
    cudaError_t e = cudaFuncSetAttribute(attn_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)g.nwin, (unsigned)heads);
    attn_backward_kernel<<<grid, BW_THREADS, smem, stream>>>(qkv, dO, table, heads, g, dqkv, dtable);
    return cudaGetLastError();
}

} // namespace swin
