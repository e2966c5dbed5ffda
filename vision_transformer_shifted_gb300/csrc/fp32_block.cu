// fp32 block (CUDA-core FMA, no TF32), the V2 bias-table builder and the
// bounded-wait probe.
//
// The fp32 block serves the fp32 mode (small blocks checked to 1e-5): one CTA
// per window runs every step of the block -- gather through cyclic shift and
// partition, QKV projection with bias, V1/V2 logits with relative bias and
// shift mask, softmax, P.V, output projection with bias, scatter through
// window reverse and roll back (pages "Boosting Swin Transformer Speed",
// Introduction / Training Optimization; "Swin Transformer V2"
// (neura.market), How It Works).
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int FP32_THREADS = 256;

__global__ void __launch_bounds__(FP32_THREADS) fp32_block_kernel(Fp32Args a)
{
    extern __shared__ float fsm[];
    const Geom g = a.g;
    const int M = g.M, N = g.N, C = g.C, h = a.heads, d = C / h, L = 2 * M - 1;
    float *xw = fsm;                  // [N][C]
    float *qkv = xw + N * C;          // [N][3C]
    float *o = qkv + N * 3 * C;       // [N][C]
    float *logit = o + N * C;         // [warps][N] scratch rows
    const int64_t win = blockIdx.x;
    const int per = g.nh * g.nw;
    const int rem = (int)(win % per);
    const int wi = rem / g.nw, wj = rem % g.nw;
    const int tid = threadIdx.x;

    // gather: token t of the window comes from the original (i+s, j+s)
    for (int idx = tid; idx < N * C; idx += FP32_THREADS) {
        const int t = idx / C, c = idx % C;
        const int64_t tok = window_row_to_token(g, win * N + t);
        xw[idx] = a.x[tok * C + c];
    }
    __syncthreads();
    for (int idx = tid; idx < N * 3 * C; idx += FP32_THREADS) {
        const int t = idx / (3 * C), oc = idx % (3 * C);
        float acc = a.bqkv ? a.bqkv[oc] : 0.f;
        const float *w = a.Wqkv + (int64_t)oc * C;
        const float *xr = xw + t * C;
        for (int c = 0; c < C; ++c) acc = fmaf(xr[c], w[c], acc);
        qkv[idx] = acc;
    }
    __syncthreads();
    if (a.mode == 1) { // V2: unit-norm q and k rows per head
        for (int idx = tid; idx < N * 2 * h; idx += FP32_THREADS) {
            const int t = idx / (2 * h), ph = idx % (2 * h);
            float *v = qkv + t * 3 * C + (ph / h) * C + (ph % h) * d;
            float ss = 0.f;
            for (int e = 0; e < d; ++e) ss = fmaf(v[e], v[e], ss);
            const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
            for (int e = 0; e < d; ++e) v[e] *= inv;
        }
        __syncthreads();
    }
    // attention: one warp per (head, query) row
    const int warp = tid >> 5, lane = tid & 31;
    float *lrow = logit + warp * N;
    for (int rowid = warp; rowid < h * N; rowid += FP32_THREADS / 32) {
        const int hd = rowid / N, qi = rowid % N;
        const float scale = a.mode == 1 ? 1.0f / fmaxf(a.tau[hd], 0.01f) : 1.0f / sqrtf((float)d);
        const int ri = qi / M, ci = qi % M;
        int qreg = 0;
        if (g.s > 0) qreg = 3 * shift_band(wi * M + ri, g.H, M, g.s) + shift_band(wj * M + ci, g.W, M, g.s);
        const float *q = qkv + qi * 3 * C + hd * d;
        float mx = -INFINITY;
        for (int kj = lane; kj < N; kj += 32) {
            const int rj = kj / M, cj = kj % M;
            int kreg = 0;
            if (g.s > 0) kreg = 3 * shift_band(wi * M + rj, g.H, M, g.s) + shift_band(wj * M + cj, g.W, M, g.s);
            float v = -INFINITY;
            if (kreg == qreg) {
                const float *k = qkv + kj * 3 * C + C + hd * d;
                float dot = 0.f;
                for (int e = 0; e < d; ++e) dot = fmaf(q[e], k[e], dot);
                v = dot * scale + a.table[(int64_t)((ri - rj + M - 1) * L + (ci - cj + M - 1)) * h + hd];
            }
            lrow[kj] = v;
            mx = fmaxf(mx, v);
        }
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        float sum = 0.f;
        for (int kj = lane; kj < N; kj += 32) {
            const float p = expf(lrow[kj] - mx);
            lrow[kj] = p;
            sum += p;
        }
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        __syncwarp();
        const float inv = 1.0f / sum;
        for (int e = lane; e < d; e += 32) {
            float acc = 0.f;
            for (int kj = 0; kj < N; ++kj) acc = fmaf(lrow[kj], qkv[kj * 3 * C + 2 * C + hd * d + e], acc);
            o[qi * C + hd * d + e] = acc * inv;
        }
        __syncwarp();
    }
    __syncthreads();
    // projection, scatter back through window reverse and roll by +s
    for (int idx = tid; idx < N * C; idx += FP32_THREADS) {
        const int t = idx / C, oc = idx % C;
        float acc = a.bproj ? a.bproj[oc] : 0.f;
        const float *w = a.Wproj + (int64_t)oc * C;
        const float *orow = o + t * C;
        for (int c = 0; c < C; ++c) acc = fmaf(orow[c], w[c], acc);
        a.out[window_row_to_token(g, win * N + t) * C + oc] = acc;
    }
}

// One CTA per table row idx: hidden = relu(W1 u + b1) in shared memory, then
// one warp per head reduces W2[head] . hidden.
__global__ void cpb_table_kernel(const float *W1, const float *b1, const float *W2, int hidden, int M, int heads,
                                 int out_bf16, void *table)
{
    extern __shared__ float hid[];
    const int L = 2 * M - 1;
    const int idx = blockIdx.x;
    const int dr = idx / L - (M - 1), dc = idx % L - (M - 1);
    const float u0 = dr == 0 ? 0.f : copysignf(log1pf(fabsf((float)dr)), (float)dr);
    const float u1 = dc == 0 ? 0.f : copysignf(log1pf(fabsf((float)dc)), (float)dc);
    for (int k = threadIdx.x; k < hidden; k += blockDim.x) {
        const float v = fmaf(W1[2 * k], u0, fmaf(W1[2 * k + 1], u1, b1 ? b1[k] : 0.f));
        hid[k] = fmaxf(v, 0.f);
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int hd = warp; hd < heads; hd += nwarps) {
        float acc = 0.f;
        for (int k = lane; k < hidden; k += 32) acc = fmaf(W2[(int64_t)hd * hidden + k], hid[k], acc);
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            if (out_bf16) reinterpret_cast<bf16 *>(table)[(int64_t)idx * heads + hd] = __float2bfloat16_rn(acc);
            else reinterpret_cast<float *>(table)[(int64_t)idx * heads + hd] = acc;
        }
    }
}

// Gradient of G's weights from the gradient of its table (the chain rule
// through table[idx, h] = sum_k W2[h, k] relu(W1[k] . u(idx) + b1[k])): one
// thread per hidden unit k recomputes its pre-activation at every relative
// offset and accumulates dW2[:, k], dW1[k, :] and db1[k] in registers (no
// atomics).  dtable and the coordinates u come through shared memory.
constexpr int CPB_MAX_HEADS = 16;

__global__ void cpb_backward_kernel(const float *W1, const float *b1, const float *W2, const float *dtable, int hidden,
                                    int M, int heads, float *dW1, float *db1, float *dW2)
{
    extern __shared__ float cpb_sm[];
    const int L = 2 * M - 1, LL = L * L;
    float *sdt = cpb_sm, *su = cpb_sm + LL * heads;
    for (int e = threadIdx.x; e < LL * heads; e += blockDim.x) sdt[e] = dtable[e];
    for (int idx = threadIdx.x; idx < LL; idx += blockDim.x) {
        const int dr = idx / L - (M - 1), dc = idx % L - (M - 1);
        su[2 * idx] = dr == 0 ? 0.f : copysignf(log1pf(fabsf((float)dr)), (float)dr);
        su[2 * idx + 1] = dc == 0 ? 0.f : copysignf(log1pf(fabsf((float)dc)), (float)dc);
    }
    __syncthreads();
    const int k = blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= hidden) return;
    const float w0 = W1[2 * k], w1 = W1[2 * k + 1], bb = b1 ? b1[k] : 0.f;
    float w2[CPB_MAX_HEADS], acc[CPB_MAX_HEADS];
#pragma unroll
    for (int hd = 0; hd < CPB_MAX_HEADS; ++hd) {
        w2[hd] = hd < heads ? W2[(int64_t)hd * hidden + k] : 0.f;
        acc[hd] = 0.f;
    }
    float dw0 = 0.f, dw1 = 0.f, db = 0.f;
    for (int idx = 0; idx < LL; ++idx) {
        const float u0 = su[2 * idx], u1 = su[2 * idx + 1];
        const float pre = fmaf(w0, u0, fmaf(w1, u1, bb));
        if (pre <= 0.f) continue;
        float dh = 0.f;
#pragma unroll
        for (int hd = 0; hd < CPB_MAX_HEADS; ++hd) {
            if (hd < heads) {
                const float g = sdt[idx * heads + hd];
                dh = fmaf(g, w2[hd], dh);
                acc[hd] = fmaf(g, pre, acc[hd]);
            }
        }
        dw0 = fmaf(dh, u0, dw0);
        dw1 = fmaf(dh, u1, dw1);
        db += dh;
    }
    dW1[2 * k] = dw0;
    dW1[2 * k + 1] = dw1;
    if (db1) db1[k] = db;
#pragma unroll
    for (int hd = 0; hd < CPB_MAX_HEADS; ++hd)
        if (hd < heads) dW2[(int64_t)hd * hidden + k] = acc[hd];
}

// Waits on an mbarrier that nothing arrives on, with the caller's limit, and
// records the timeout: exercises the bounded-wait exit of the kernels.
__global__ void watchdog_kernel(DeviceStatus st)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool ok = mbar_wait(smem_u32(&bar), 0, st.wait_ns);
    if (!ok && threadIdx.x == 0) atomicOr(st.err, ERR_TIMEOUT);
}

} // namespace

size_t fp32_block_smem_bytes(int N, int C)
{
    return (size_t)(N * C + N * 3 * C + N * C + (FP32_THREADS / 32) * N) * sizeof(float);
}

cudaError_t launch_fp32_block(const Fp32Args &a, cudaStream_t stream)
{
    const size_t smem = fp32_block_smem_bytes(a.g.N, a.g.C);
    if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(fp32_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fp32_block_kernel<<<(unsigned)a.g.nwin, FP32_THREADS, smem, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_cpb_table(const float *W1, const float *b1, const float *W2, int hidden, int M, int heads,
                             bool out_bf16, void *table, cudaStream_t stream)
{
    const int L = 2 * M - 1;
    cpb_table_kernel<<<L * L, 256, hidden * sizeof(float), stream>>>(W1, b1, W2, hidden, M, heads, out_bf16 ? 1 : 0,
                                                                   table);
    return cudaGetLastError();
}

cudaError_t launch_cpb_backward(const float *W1, const float *b1, const float *W2, const float *dtable, int hidden,
                                int M, int heads, float *dW1, float *db1, float *dW2, cudaStream_t stream)
{
    if (heads > CPB_MAX_HEADS || hidden <= 0) return cudaErrorInvalidValue;
    const int L = 2 * M - 1;
    const size_t smem = ((size_t)L * L * heads + 2 * (size_t)L * L) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(cpb_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cpb_backward_kernel<<<(hidden + 127) / 128, 128, smem, stream>>>(W1, b1, W2, dtable, hidden, M, heads, dW1, db1,
                                                                     dW2);
    return cudaGetLastError();
}

cudaError_t launch_watchdog(DeviceStatus st, cudaStream_t stream)
{
    watchdog_kernel<<<1, 32, 0, stream>>>(st);
    return cudaGetLastError();
}

} // namespace swin
