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
// The weight and bias gradients are sums over tokens, so they do not depend
// on the order of the rows: the attention backward writes o and dqkv straight
// back in token order, dWproj = dy^T o and dWqkv = dqkv^T x then take dy and x
// as they are, dx = dqkv Wqkv needs no scatter, and only the two GEMMs that
// feed the attention backward (qkv and do, in window order) gather their rows.
// This file holds a weight transpose, column sums and the tcgen05 attention
// kernel in two modes: the backward (which also yields o, so the forward
// attention is not run again) and the forward attention step of the
// three-kernel path for windows of at most 64 tokens; the GEMMs are launched
// by the caller.
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

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

// ---- attention backward on the tensor cores ------------------------------------
//
// A unit is one head of two consecutive windows, stacked into 128 rows (window
// 2p in rows 0..63, window 2p+1 in rows 64..127; rows past N stay zero).  TMA
// brings the head's q, k, v, do of both windows into shared memory ([128 rows]
// [32 ch], 64-byte swizzle), then
//   S = q k^T and dP = do v^T                  (M = 128, N = 128, K = 32)
// two threads per row (one per 32 keys of the row's window) turn their halves
// into P and dS = P (dP - rowsum(P dP)), merging the row's maximum, sum and
// rowsum through shared memory, and store them as bf16 (block-diagonal: the
// other window's block stays zero); then
//   o = P v,  dq = dS k,  dv = P^T do,  dk = dS^T q   (M = 128, N = 32, K = 128)
// with P^T and dS^T the same shared-memory tiles read M-major (S and dP come
// from two issuing threads, the four outputs from four, so that the MMAs'
// issue costs overlap).  Cross-window
// products vanish because the off-diagonal blocks are zero.  Units run head
// by head (unit u: head u / pairs; a CTA takes a contiguous range of units),
// so a CTA keeps one head's bias matrix in
// shared memory and the table gradient of each (query, key) position in
// registers, folding it into the table only when the head changes.
constexpr int TB_THREADS = 256;
constexpr int BIAS_STRIDE = 144; // bytes per bias row: 64 bf16 + 16 pad (conflict-free 16-byte loads)

template <bool BW>
struct TbLayout {
    // byte offsets from the 1024-aligned base; the forward mode has no do tile,
    // no dS panels and no table gradient, so three CTAs share an SM
    static constexpr uint32_t Q = 0, K = 8192, V = 16384, DO = 24576;  // [128][64 B] tiles
    static constexpr uint32_t P = BW ? 32768 : 24576;                   // 4 panels of [128][32 keys]
    static constexpr uint32_t DS = P + 32768;                          // (backward only)
    static constexpr uint32_t BIAS = BW ? 98304 : 57344;               // bf16 [64][72]
    static constexpr uint32_t MASK = BIAS + 64 * BIAS_STRIDE;          // uint64 [4 classes][64 rows]
    static constexpr uint32_t RED = MASK + 4 * 64 * 8;                 // float [2][128][4]
    static constexpr uint32_t DTAB = RED + 2 * 128 * 16;               // float [(2M-1)^2 <= 225], padded
    static constexpr uint32_t BAR = DTAB + (BW ? 228 * 4 : 0);         // 3 mbarriers + TMEM slot
    static constexpr size_t bytes() { return (size_t)BAR + 32 + 1024; }
    // TMEM: S and dP (backward); S, then o over S's first 32 columns (forward)
    static constexpr uint32_t TCOLS = BW ? 256 : 128;
    static constexpr int CTAS_PER_SM = BW ? 2 : 3;
};

__device__ __forceinline__ int band_in_window(int t, int M, int s) { return t < M - s ? 1 : 2; }

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

// With u = v / n (unit length) and du the gradient of u: dv = (du - u (u . du))
// / n.  du (32 channels of one row) is scaled by f = scale / n, u is the row's
// bf16 copy in the 64-byte-swizzled tile at `tile`.
__device__ __forceinline__ void unit_scale_backward(float (&du)[32], uint32_t tile, int row, float f)
{
    // two passes over the row in shared memory (u . du, then the update), so
    // that u never needs 32 registers of its own
    float dot = 0.f;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(tile + sw64_offset(row, c)));
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 p = unpack_bf16x2(w[t]);
                const int e = 8 * c + 2 * t;
                if (pass == 0) {
                    dot = fmaf(p.x, du[e], fmaf(p.y, du[e + 1], dot));
                } else {
                    du[e] = (du[e] - p.x * dot) * f;
                    du[e + 1] = (du[e + 1] - p.y * dot) * f;
                }
            }
        }
    }
}

// BW = false: the forward attention alone (S, P, o = P v; V1 scale 1/sqrt(32)
// or V2 1/max(tau, 0.01) per head), o written in window order.
// BW = true: the backward of the V1 block as described above.
template <bool BW>
__global__ void __launch_bounds__(TB_THREADS, TbLayout<BW>::CTAS_PER_SM)
attn_tc_kernel(const bf16 *table, const float *tau, int heads, int v2, Geom g, bf16 *attn, bf16 *dqkv, float *dtable,
               const float *norms, float *dtau, DeviceStatus st, const __grid_constant__ CUtensorMap tm_qkv,
               const __grid_constant__ CUtensorMap tm_do)
{
    extern __shared__ uint8_t smraw[];
    using Ly = TbLayout<BW>;
    uint8_t *sm = smem_align(smraw, 1024);
    const uint32_t base = smem_u32(sm);
    const int N = g.N, M = g.M, C = g.C, L = 2 * M - 1, LL = L * L;
    const uint64_t *mask = reinterpret_cast<const uint64_t *>(sm + Ly::MASK);
    float *red = reinterpret_cast<float *>(sm + Ly::RED);
    float *dtab = reinterpret_cast<float *>(sm + Ly::DTAB);
    const uint32_t bar_ld = base + Ly::BAR, bar_s = bar_ld + 8, bar_o = bar_ld + 16;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Ly::BAR + 24);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, h2 = warp >> 2;     // TMEM lane quadrant; which 32 keys of the row
    const int r = quad * 32 + lane, hf = r >> 6, i = r & 63;
    const int64_t npairs = (g.nwin + 1) / 2, nunits = npairs * heads;
    float scale = 0.17677669529663687f;          // logit scale of the current head (V1: 1 / sqrt(32))
    float tau_acc = 0.f;                         // V2 backward: sum of dS * cos over this CTA's rows of the head
    const float log2e = 1.4426950408889634f;

    // zero the operand tiles (rows past N are never loaded) and P, dS (their
    // off-diagonal blocks are never written)
    for (int e = tid; e < Ly::BIAS / 16; e += TB_THREADS)
        *reinterpret_cast<uint4 *>(sm + 16 * e) = make_uint4(0, 0, 0, 0);
    // visibility masks: bit j of mask[cls][i] = key j visible to query i, for
    // the four window classes (cls bit 0: last window row, bit 1: last window
    // column, where the shifted frame's bands split the window at M - s)
    {
        const int cls = tid >> 6, ii = tid & 63;
        uint64_t m = 0;
        if (ii < N) {
            const int s = g.s;
            auto region = [&](int t) {
                if (s == 0) return 0;
                return 3 * ((cls & 1) ? band_in_window(t / M, M, s) : 0) + ((cls & 2) ? band_in_window(t % M, M, s) : 0);
            };
            const int ri = region(ii);
            for (int j = 0; j < N; ++j)
                if (region(j) == ri) m |= 1ull << j;
        }
        reinterpret_cast<uint64_t *>(sm + Ly::MASK)[tid] = m;
    }
    if (BW)
        for (int e = tid; e < 228; e += TB_THREADS) dtab[e] = 0.f;
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_s, BW ? 2 : 1);
        mbar_init(bar_o, BW ? 4 : 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), Ly::TCOLS);
        tmem_relinquish();
    }
    fence_proxy_async_smem(); // the zeroed tiles, before any TMA or MMA touches them

    // TMA of unit u's q, k, v (and do) (one box of N rows x 32 channels per window and tensor)
    auto load_unit = [&](int64_t u) {
        const int head = (int)(u / npairs);
        const int64_t pair = u - (int64_t)head * npairs;
        const int nw = 2 * pair + 1 < g.nwin ? 2 : 1;
        mbar_arrive_expect_tx(bar_ld, (uint32_t)(nw * (BW ? 4 : 3) * N * 64));
        for (int w = 0; w < nw; ++w) {
            const int y = (int)((2 * pair + w) * N);
            const uint32_t dst = base + (uint32_t)w * 4096u;
            tma_load_2d(dst + Ly::Q, &tm_qkv, head * 32, y, bar_ld);
            tma_load_2d(dst + Ly::K, &tm_qkv, C + head * 32, y, bar_ld);
            tma_load_2d(dst + Ly::V, &tm_qkv, 2 * C + head * 32, y, bar_ld);
            if (BW) tma_load_2d(dst + Ly::DO, &tm_do, head * 32, y, bar_ld);
        }
    };

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // (every read of q, k, v, dO comes after: a no-op unless launched to
    // overlap the kernels before it)
    griddep_launch_dependents();
    griddep_wait();
    // a contiguous range of units per CTA (head changes at most a few times)
    const int64_t u_begin = nunits * blockIdx.x / gridDim.x, u_end = nunits * (blockIdx.x + 1) / gridDim.x;
    if (tid == 0 && u_begin < u_end) load_unit(u_begin);
    const uint32_t tmem = *tslot;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);

    uint32_t phase = 0;
    bool failed = false;
    int cur_head = -1;
    float acc[32]; // table gradient of (query i, key 32*h2 + j) over this CTA's units of cur_head
#pragma unroll
    for (int j = 0; j < 32; ++j) acc[j] = 0.f;

    // adds acc into the head's table gradient (shared, then global)
    auto flush_head = [&]() {
        if (i < N) {
            const int ri = i / M, ci = i % M;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = 32 * h2 + j;
                if (key < N && acc[j] != 0.f)
                    atomicAdd(&dtab[(ri - key / M + M - 1) * L + (ci - key % M + M - 1)], acc[j]);
                acc[j] = 0.f;
            }
        }
        if (v2) {
            // dtau = -sum(dS cos) / tau^2 above the 0.01 clip, 0 below it
            float t = tau_acc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            const float tv = tau[cur_head];
            if (lane == 0 && tv > 0.01f && t != 0.f) atomicAdd(&dtau[cur_head], -t / (tv * tv));
            tau_acc = 0.f;
        }
        __syncthreads();
        for (int e = tid; e < LL; e += TB_THREADS) {
            if (dtab[e] != 0.f) atomicAdd(&dtable[(int64_t)e * heads + cur_head], dtab[e]);
            dtab[e] = 0.f;
        }
    };

    for (int64_t u = u_begin; u < u_end; ++u) {
        const int head = (int)(u / npairs);
        const int64_t pair = u - (int64_t)head * npairs;
        const int64_t win = 2 * pair + hf;
        const bool rv = i < N && win < g.nwin;
        if (head != cur_head) {
            if (BW && cur_head >= 0) flush_head();
            if (v2) scale = 1.0f / fmaxf(tau[head], 0.01f);
            // the head's bias matrix B[i][j] = table[idx(i, j), head] (zero outside N x N)
            for (int e = tid; e < 64 * 64; e += TB_THREADS) {
                const int a = e >> 6, b = e & 63;
                bf16 v = __float2bfloat16(0.f);
                if (a < N && b < N)
                    v = table[(int64_t)((a / M - b / M + M - 1) * L + (a % M - b % M + M - 1)) * heads + head];
                *reinterpret_cast<bf16 *>(sm + Ly::BIAS + a * BIAS_STRIDE + 2 * b) = v;
            }
            cur_head = head;
            __syncthreads();
        }
        int cls = 0;
        if (g.s > 0 && rv) {
            const int rem = (int)(win % (g.nh * g.nw));
            cls = (rem / g.nw == g.nh - 1 ? 1 : 0) | (rem % g.nw == g.nw - 1 ? 2 : 0);
        }
        if (tid == 0 || (BW && tid == 128)) {
            // S by thread 0, dP by thread 128 (their issue costs overlap)
            const bool okl = mbar_wait(bar_ld, phase, st.wait_ns);
            if (okl) {
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 128);
                const uint32_t a = tid == 0 ? Ly::Q : Ly::DO, b = tid == 0 ? Ly::K : Ly::V;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16(tmem + (tid == 0 ? 0 : 128), desc_kmajor_sw64(base + a + 32 * ks),
                             desc_kmajor_sw64(base + b + 32 * ks), id, ks);
                mma_commit(bar_s);
            }
        }
        bool ok = mbar_wait(bar_s, phase, st.wait_ns);
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();

        // ---- P (and dS): this thread's 32 keys of its row ----
        float s[32], d[32];
        tmem_ld32(t_lane + 64 * hf + 32 * h2, s);
        if (BW) tmem_ld32(t_lane + 128 + 64 * hf + 32 * h2, d);
        const uint32_t mb = rv ? (uint32_t)(mask[cls * 64 + i] >> (32 * h2)) : 0u;
        {
            const uint4 *brow = reinterpret_cast<const uint4 *>(sm + Ly::BIAS + i * BIAS_STRIDE + 64 * h2);
            uint4 bq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) bq[q] = brow[q];
            tmem_wait_ld();
            float mx = -INFINITY;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t w4[4] = {bq[q].x, bq[q].y, bq[q].z, bq[q].w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 b2 = unpack_bf16x2(w4[t]);
                    const int j = 8 * q + 2 * t;
                    s[j] = (mb >> j) & 1u ? fmaf(s[j], scale, b2.x) : -INFINITY;
                    s[j + 1] = (mb >> (j + 1)) & 1u ? fmaf(s[j + 1], scale, b2.y) : -INFINITY;
                    mx = fmaxf(mx, fmaxf(s[j], s[j + 1]));
                }
            }
            const float mxl = mb ? mx * log2e : 0.f;
            float sum = 0.f, dsum = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] = ex2_approx(fmaf(s[j], log2e, -mxl)); // masked: -inf -> 0
                sum += s[j];
                if (BW) dsum = fmaf(s[j], d[j], dsum);
            }
            float *mine = red + (h2 * 128 + r) * 4;
            mine[0] = mb ? mx : -INFINITY;
            mine[1] = sum;
            mine[2] = dsum;
            __syncthreads();
            const float *other = red + ((1 - h2) * 128 + r) * 4;
            const float mo = other[0], so = other[1], dso = other[2];
            const float mt = mb ? mx : -INFINITY;
            const float m = fmaxf(mt, mo);
            float p_scale = 0.f, D = 0.f;
            if (rv && m > -INFINITY) {
                const float ft = ex2_approx((mt - m) * log2e), fo = ex2_approx((mo - m) * log2e);
                const float inv = 1.0f / (sum * ft + so * fo);
                p_scale = ft * inv;
                D = (dsum * ft + dso * fo) * inv;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                s[j] *= p_scale;
                if (BW) {
                    d[j] = s[j] * (d[j] - D);
                    acc[j] += d[j];
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t off = (uint32_t)(2 * hf + h2) * 8192u + sw64_offset(r, c);
                store_row8(base + Ly::P + off, s + 8 * c, 1.f);
                if (BW) store_row8(base + Ly::DS + off, d + 8 * c, 1.f);
            }
            if (BW && v2) {
                // V2: d logit / d(1/tau) = cos = the raw S (still in TMEM), read
                // back 16 columns at a time
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float c16[16];
                    tmem_ld16(t_lane + 64 * hf + 32 * h2 + 16 * hh, c16);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) tau_acc = fmaf(d[16 * hh + j], c16[j], tau_acc);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (lane == 0 && (warp & 2) == 0 && (BW || warp == 0)) {
            // one issuer per output (warps 0, 1, 4, 5): o, dq, dk, dv (forward: o only)
            tc_fence_after();
            const int which = (warp & 1) | ((warp >> 2) << 1); // 0 o, 1 dq, 2 dk, 3 dv
            if (which < 2) {
                const uint32_t a = which == 0 ? Ly::P : Ly::DS, b = which == 0 ? Ly::V : Ly::K;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t kpan = (uint32_t)(kk >> 1) * 8192u + 32u * (kk & 1);
                    mma_bf16(tmem + 32 * which, desc_kmajor_sw64(base + a + kpan),
                             desc_mnmajor_sw64(base + b + 1024 * kk, 8192), idesc_bf16_bmn(128, 32), kk);
                }
            } else {
                const uint32_t a = which == 2 ? Ly::DS : Ly::P, b = which == 2 ? Ly::Q : Ly::DO;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16(tmem + 32 * which, desc_mnmajor_sw64(base + a + 1024 * kk, 8192),
                             desc_mnmajor_sw64(base + b + 1024 * kk, 8192), idesc_bf16_amn_bmn(128, 32), kk);
            }
            mma_commit(bar_o);
        }
        ok = mbar_wait(bar_o, phase, st.wait_ns);
        phase ^= 1;
        if (__syncthreads_or(!ok)) { failed = true; break; }
        tc_fence_after();
        // q, k, v, do are free: the next unit's loads run under the epilogue
        // (V2 backward: after it, which still reads the q and k rows)
        if (!(BW && v2) && tid == 0 && u + 1 < u_end) load_unit(u + 1);

        // ---- outputs of row r ----
        if (BW) {
            // o and dq (first four warps), dk and dv (last four), one after the
            // other; rows go back to their tokens' places (window reverse and
            // roll by +s).  V2: dq and dk through the unit-length scaling of q
            // and k (dS k and dS^T q are the gradients of the unit vectors).
            const int64_t tok = rv ? window_row_to_token(g, win * N + i) : 0;
            const float nrm = v2 && rv ? norms[(win * N + i) * (2 * heads) + h2 * heads + head] : 1.f;
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                float a[32];
                tmem_ld32(t_lane + 64 * h2 + 32 * part, a);
                tmem_wait_ld();
                // part 0: o (h2 0) or dS^T q (h2 1); part 1: dS k (h2 0) or dv (h2 1)
                const bool qk = (h2 == 0) == (part == 1);
                if (qk && v2) unit_scale_backward(a, base + (h2 == 0 ? Ly::Q : Ly::K), r, scale / nrm);
                if (rv) {
                    const int col = h2 == 0 ? (part == 0 ? 0 : 0) : (part == 0 ? C : 2 * C);
                    bf16 *dst = h2 == 0 && part == 0 ? attn + tok * C + head * 32
                                                     : dqkv + tok * 3 * C + col + head * 32;
                    store_global32(dst, a, qk && !v2 ? scale : 1.f);
                }
            }
        } else {
            // o in window order, 16 channels per thread
            float a[16];
            tmem_ld16(t_lane + 16 * h2, a);
            tmem_wait_ld();
            if (rv) {
                uint4 *dst = reinterpret_cast<uint4 *>(attn + (win * N + i) * C + head * 32 + 16 * h2);
#pragma unroll
                for (int q = 0; q < 2; ++q)
                    dst[q] = make_uint4(pack_bf16x2(a[8 * q], a[8 * q + 1]), pack_bf16x2(a[8 * q + 2], a[8 * q + 3]),
                                        pack_bf16x2(a[8 * q + 4], a[8 * q + 5]), pack_bf16x2(a[8 * q + 6], a[8 * q + 7]));
            }
        }
        tc_fence_before();
        __syncthreads();
        if (BW && v2 && tid == 0 && u + 1 < u_end) load_unit(u + 1);
    }
    if (failed) {
        if (tid == 0) atomicOr(st.err, ERR_TIMEOUT);
        // a load may still be in flight: wait for it (bounded) before leaving
        if (tid == 0) mbar_wait(bar_ld, phase, st.wait_ns);
    } else if (BW && cur_head >= 0) {
        flush_head();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, Ly::TCOLS);
}

} // namespace

cudaError_t launch_transpose(const bf16 *in, bf16 *out, int rows, int cols, cudaStream_t stream)
{
    dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows + 31) / 32)), block(32, 8);
    transpose_kernel<<<grid, block, 0, stream>>>(in, out, rows, cols);
    return cudaGetLastError();
}

bool attn_backward_supported(int M, int C, int heads) { return M * M <= 64 && C == heads * 32; }

namespace {

template <bool BW>
cudaError_t launch_attn_tc(const bf16 *qkv, const bf16 *dO, const bf16 *table, const float *tau, int heads, int v2,
                           const Geom &g, bf16 *attn, bf16 *dqkv, float *dtable, const float *norms, float *dtau,
                           DeviceStatus st, cudaStream_t stream, int overlap = 0)
{
    if (!attn_backward_supported(g.M, g.C, heads)) return cudaErrorInvalidValue;
    CUtensorMap tm_qkv, tm_do;
    // units run head by head: the other heads' 64-byte slices of a row are
    // read much later, so no 128-byte L2 promotion
    cudaError_t e = make_tensor_map_sw64(&tm_qkv, qkv, g.T, 3 * g.C, g.N, false);
    if (e == cudaSuccess) e = BW ? make_tensor_map_sw64(&tm_do, dO, g.T, g.C, g.N, false) : cudaSuccess;
    if (!BW) tm_do = tm_qkv; // unused
    if (e != cudaSuccess) return e;
    const size_t smem = TbLayout<BW>::bytes();
    e = cudaFuncSetAttribute(attn_tc_kernel<BW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    }
    const int64_t units = (g.nwin + 1) / 2 * heads;
    const int64_t cap = (int64_t)sms * TbLayout<BW>::CTAS_PER_SM;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    e = launch_maybe_overlapped(attn_tc_kernel<BW>, dim3(grid), dim3(TB_THREADS), smem, stream, overlap, table, tau,
                                heads, v2, g, attn, dqkv, dtable, norms, dtau, st, tm_qkv, tm_do);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_attn_backward(const bf16 *qkv, const bf16 *dO, const bf16 *table, const float *tau, int heads,
                                 int v2, const Geom &g, bf16 *attn, bf16 *dqkv, float *dtable, const float *norms,
                                 float *dtau, DeviceStatus st, cudaStream_t stream, int overlap)
{
    return launch_attn_tc<true>(qkv, dO, table, tau, heads, v2, g, attn, dqkv, dtable, norms, dtau, st, stream,
                                overlap);
}

cudaError_t launch_attn_forward_tc(const bf16 *qkv, const bf16 *table, const float *tau, int heads, int v2,
                                   const Geom &g, bf16 *attn, DeviceStatus st, cudaStream_t stream, int overlap)
{
    return launch_attn_tc<false>(qkv, nullptr, table, tau, heads, v2, g, attn, nullptr, nullptr, nullptr, nullptr, st,
                                 stream, overlap);
}

} // namespace swin
