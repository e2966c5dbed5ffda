// Backward of the shifted-window attention for windows of more than 64
// tokens (SwinV2 at window 24: 576 tokens), on tcgen05 tensor cores.
//
// Same gradients as the short-window kernel (csrc/backward.cu): with the
// row-wise softmax normaliser of the forward (its log2, lse, kept by the
// large-window forward kernel) P = exp2(logit2 - lse) needs no row reduction,
// so a CTA can own a tile of 128 KEYS of one window and head and walk over
// the window's query tiles (the FlashAttention backward order):
//   S^T  = k q^T and dP^T = v do^T            (M = 128 keys, N = 128 queries, K = 32)
//   P^T, dS^T = P^T (dP^T - D), D_i = do_i . o_i (computed beforehand)
//   dv  += P^T do,  dk += dS^T q             (kept in registers across query tiles)
//   dq_i += dS k                             (M = 128 queries: dS^T read M-major;
//                                             added to an fp32 buffer by atomics, since
//                                             every key tile of the window contributes)
// and the table gradient of each relative offset summed in shared memory per
// head (units run head by head, a contiguous range per CTA).  A last kernel
// turns the fp32 dq into bf16 (scale, and for V2 the unit-length backward).
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int FB_THREADS = 256;

struct FbLayout {
    // byte offsets from the 1024-aligned base
    static constexpr uint32_t K = 0, V = 8192, Q = 16384, DO = 24576; // [128 rows][64 B] tiles
    static constexpr uint32_t P = 32768, DS = 65536;                   // 4 panels [128 keys][32 queries]
    static constexpr uint32_t QB = 98304;                              // int [128]: relative-index base of each query (-1: none)
    static constexpr uint32_t QR = QB + 512;                           // int [128]: shift region of each query
    static constexpr uint32_t LSE = QR + 512;                          // float [128]
    static constexpr uint32_t DD = LSE + 512;                          // float [128]
    static constexpr uint32_t BIAS = DD + 512;                         // bf16 [(2M-1)^2] of the current head
    __host__ __device__ static uint32_t ll_pad(int M) { return ((uint32_t)(2 * M - 1) * (2 * M - 1) + 7u) & ~7u; }
    __host__ __device__ static uint32_t dtab(int M) { return BIAS + 2 * ll_pad(M); }
    __host__ __device__ static uint32_t bar(int M) { return dtab(M) + 4 * ll_pad(M); }
    // four mbarriers, then the TMEM address slot
    static size_t bytes(int M) { return (size_t)bar(M) + 48 + 1024; }
};

__device__ __forceinline__ int fb_band(int p, int n, int M, int s) { return p < n - M ? 0 : (p < n - s ? 1 : 2); }

// shift region of token t of window (wi, wj) (0 everywhere without a shift)
__device__ __forceinline__ int fb_region(const Geom &g, int wi, int wj, int t)
{
    if (g.s == 0) return 0;
    const int ti = t / g.M, tj = t - (t / g.M) * g.M;
    return 3 * fb_band(wi * g.M + ti, g.H, g.M, g.s) + fb_band(wj * g.M + tj, g.W, g.M, g.s);
}

__device__ __forceinline__ void fb_store8(uint32_t dst, const float *v)
{
    const uint32_t a = pack_bf16x2(v[0], v[1]), b = pack_bf16x2(v[2], v[3]);
    const uint32_t c = pack_bf16x2(v[4], v[5]), d = pack_bf16x2(v[6], v[7]);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// With u = v / n and du the gradient of u: dv = (du - u (u . du)) * f, f = scale / n
// (two passes over the row u in the 64-byte-swizzled tile).
__device__ __forceinline__ void fb_unit_backward(float (&du)[32], uint32_t tile, int row, float f, bool unit)
{
    float dot = 0.f;
    if (unit) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[4];
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(tile + sw64_offset(row, c)));
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 p = unpack_bf16x2(w[t]);
                dot = fmaf(p.x, du[8 * c + 2 * t], fmaf(p.y, du[8 * c + 2 * t + 1], dot));
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w[4] = {0, 0, 0, 0};
        if (unit)
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(tile + sw64_offset(row, c)));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 p = unpack_bf16x2(w[t]);
            du[8 * c + 2 * t] = (du[8 * c + 2 * t] - p.x * dot) * f;
            du[8 * c + 2 * t + 1] = (du[8 * c + 2 * t + 1] - p.y * dot) * f;
        }
    }
}

__global__ void __launch_bounds__(FB_THREADS, 2)
attn_flash_backward_kernel(const bf16 *table, const float *tau, int heads, int v2, Geom g, const float *lse,
                           const float *Dr, const float *norms, bf16 *dqkv, float *dq_acc, float *dtable, float *dtau,
                           DeviceStatus st, const __grid_constant__ CUtensorMap tm_qkv,
                           const __grid_constant__ CUtensorMap tm_do)
{
    extern __shared__ uint8_t smraw[];
    using Ly = FbLayout;
    uint8_t *sm = smem_align(smraw, 1024);
    const uint32_t base = smem_u32(sm);
    const int N = g.N, M = g.M, C = g.C, L = 2 * M - 1, LL = L * L;
    const int KT = (N + 127) / 128;                 // key tiles and query tiles per window
    int *qbase = reinterpret_cast<int *>(sm + Ly::QB);
    int *qreg = reinterpret_cast<int *>(sm + Ly::QR);
    float *slse = reinterpret_cast<float *>(sm + Ly::LSE);
    float *sdd = reinterpret_cast<float *>(sm + Ly::DD);
    const bf16 *sbias = reinterpret_cast<const bf16 *>(sm + Ly::BIAS);
    float *dtab = reinterpret_cast<float *>(sm + Ly::dtab(M));
    const uint32_t bar_kv = base + Ly::bar(M), bar_q = bar_kv + 8, bar_s = bar_kv + 16, bar_o = bar_kv + 24;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Ly::bar(M) + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, h2 = warp >> 2;
    const int r = quad * 32 + lane;                  // TMEM lane: key row (S^T), or query row (dq)
    const int per = g.nh * g.nw;
    const int64_t nunits = (int64_t)heads * g.nwin * KT;
    const float LOG2E = 1.4426950408889634f;

    for (int e = tid; e < (int)Ly::ll_pad(M); e += FB_THREADS) dtab[e] = 0.f;
    if (tid == 0) {
        mbar_init(bar_kv, 1);
        mbar_init(bar_q, 1);
        mbar_init(bar_s, 2);
        mbar_init(bar_o, 3);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);

    const int64_t u_begin = nunits * blockIdx.x / gridDim.x, u_end = nunits * (blockIdx.x + 1) / gridDim.x;
    auto decode = [&](int64_t u, int &head, int64_t &win, int &kt) {
        head = (int)(u / ((int64_t)g.nwin * KT));
        const int64_t rem = u - (int64_t)head * g.nwin * KT;
        win = rem / KT;
        kt = (int)(rem - win * KT);
    };
    auto load_kv = [&](int64_t u) {
        int head, kt;
        int64_t win;
        decode(u, head, win, kt);
        const int y = (int)(win * N + kt * 128);
        mbar_arrive_expect_tx(bar_kv, 2 * 128 * 64);
        tma_load_2d(base + Ly::K, &tm_qkv, C + head * 32, y, bar_kv);
        tma_load_2d(base + Ly::V, &tm_qkv, 2 * C + head * 32, y, bar_kv);
    };
    auto load_q = [&](int head, int64_t win, int qt) {
        const int y = (int)(win * N + qt * 128);
        mbar_arrive_expect_tx(bar_q, 2 * 128 * 64);
        tma_load_2d(base + Ly::Q, &tm_qkv, head * 32, y, bar_q);
        tma_load_2d(base + Ly::DO, &tm_do, head * 32, y, bar_q);
    };

    uint32_t ph_kv = 0, ph_q = 0, ph_mma = 0;
    // loads and MMAs issued but not yet waited for (the same in every thread)
    bool kv_pend = false, q_pend = false, s_pend = false, o_pend = false;
    bool failed = false;
    int cur_head = -1;
    float scale = 0.17677669529663687f; // logit scale of the current head (V1: 1 / sqrt(32))
    float tau_acc = 0.f;

    auto flush_head = [&]() {
        if (v2) {
            float t = tau_acc;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            const float tv = tau[cur_head];
            if (lane == 0 && tv > 0.01f && t != 0.f) atomicAdd(&dtau[cur_head], -t / (tv * tv));
            tau_acc = 0.f;
        }
        __syncthreads();
        for (int e = tid; e < LL; e += FB_THREADS) {
            if (dtab[e] != 0.f) atomicAdd(&dtable[(int64_t)e * heads + cur_head], dtab[e]);
            dtab[e] = 0.f;
        }
    };

    if (u_begin < u_end) {
        int h0, k0;
        int64_t w0;
        decode(u_begin, h0, w0, k0);
        if (tid == 0) {
            load_kv(u_begin);
            load_q(h0, w0, 0);
        }
        kv_pend = q_pend = true;
    }
    for (int64_t u = u_begin; u < u_end && !failed; ++u) {
        int head, kt;
        int64_t win;
        decode(u, head, win, kt);
        const int rem = (int)(win % per);
        const int wi = rem / g.nw, wj = rem - (rem / g.nw) * g.nw;
        if (head != cur_head) {
            if (cur_head >= 0) flush_head();
            for (int e = tid; e < LL; e += FB_THREADS)
                reinterpret_cast<bf16 *>(sm + Ly::BIAS)[e] = table[(int64_t)e * heads + head];
            if (v2) scale = 1.0f / fmaxf(tau[head], 0.01f);
            cur_head = head;
            __syncthreads();
        }
        const float sc2 = scale * LOG2E;
        // this thread's key (S^T row r)
        const int j = kt * 128 + r;
        const bool kvalid = j < N;
        const int kofs = kvalid ? (j / M) * L + (j % M) : 0;
        const int kreg = kvalid ? fb_region(g, wi, wj, j) : -2;
        float acc[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[c] = 0.f;

        for (int qt = 0; qt < KT; ++qt) {
            // the query tile's metadata
            if (tid < 128) {
                const int q = qt * 128 + tid;
                int qb = -1, qr = -1;
                float lv = 0.f, dv = 0.f;
                if (q < N) {
                    const int qi = q / M, qj = q - (q / M) * M;
                    qb = (qi + M - 1) * L + (qj + M - 1);
                    qr = fb_region(g, wi, wj, q);
                    lv = lse[(win * N + q) * heads + head];
                    dv = Dr[(win * N + q) * heads + head];
                }
                qbase[tid] = qb;
                qreg[tid] = qr;
                slse[tid] = lv;
                sdd[tid] = dv;
            }
            bool ok = true;
            if (qt == 0) ok = mbar_wait(bar_kv, ph_kv, st.wait_ns);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            if (qt == 0) { ph_kv ^= 1; kv_pend = false; }
            ok = mbar_wait(bar_q, ph_q, st.wait_ns);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            ph_q ^= 1;
            q_pend = false;
            if (tid == 0 || tid == 128) {
                // S^T by thread 0, dP^T by thread 128
                tc_fence_after();
                const uint32_t id = idesc_bf16(128, 128);
                const uint32_t a = tid == 0 ? Ly::K : Ly::V, b = tid == 0 ? Ly::Q : Ly::DO;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16(tmem + (tid == 0 ? 0 : 128), desc_kmajor_sw64(base + a + 32 * ks),
                             desc_kmajor_sw64(base + b + 32 * ks), id, ks);
                mma_commit(bar_s);
            }
            s_pend = true;
            ok = mbar_wait(bar_s, ph_mma, st.wait_ns);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            s_pend = false;
            tc_fence_after();

            // ---- P^T and dS^T of key row r, queries 64*h2 .. +63, 16 at a time ----
#pragma unroll 1
            for (int hh = 0; hh < 4; ++hh) {
                const int i0 = 64 * h2 + 16 * hh;
                float s[16], d[16];
                tmem_ld16(t_lane + i0, s);
                tmem_ld16(t_lane + 128 + i0, d);
                tmem_wait_ld();
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int i = i0 + jj;
                    const int qb = qbase[i];
                    const bool valid = kvalid && qb >= 0 && qreg[i] == kreg;
                    const int idx = valid ? qb - kofs : 0;
                    const float b = __bfloat162float(sbias[idx]);
                    const float p = valid ? ex2_approx(fmaf(s[jj], sc2, fmaf(b, LOG2E, -slse[i]))) : 0.f;
                    const float ds = p * (d[jj] - sdd[i]);
                    if (v2) tau_acc = fmaf(ds, s[jj], tau_acc);
                    if (ds != 0.f) atomicAdd(&dtab[idx], ds);
                    s[jj] = p;
                    d[jj] = ds;
                }
                // queries i0 .. i0+15: panel i0 / 32, 16-byte chunks 2 (i0 / 16 mod 2) ..
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const uint32_t off = (uint32_t)(i0 >> 5) * 8192u + sw64_offset(r, 2 * (hh & 1) + c);
                    fb_store8(base + Ly::P + off, s + 8 * c);
                    fb_store8(base + Ly::DS + off, d + 8 * c);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            if (lane == 0 && (warp == 0 || warp == 1 || warp == 4)) {
                // dv (warp 0), dk (warp 1), dq (warp 4)
                tc_fence_after();
                const int which = warp == 0 ? 0 : (warp == 1 ? 1 : 2);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t kpan = (uint32_t)(kk >> 1) * 8192u + 32u * (kk & 1);
                    if (which == 0)
                        mma_bf16(tmem + 0, desc_kmajor_sw64(base + Ly::P + kpan),
                                 desc_mnmajor_sw64(base + Ly::DO + 1024 * kk, 8192), idesc_bf16_bmn(128, 32), kk);
                    else if (which == 1)
                        mma_bf16(tmem + 32, desc_kmajor_sw64(base + Ly::DS + kpan),
                                 desc_mnmajor_sw64(base + Ly::Q + 1024 * kk, 8192), idesc_bf16_bmn(128, 32), kk);
                    else
                        mma_bf16(tmem + 64, desc_mnmajor_sw64(base + Ly::DS + 1024 * kk, 8192),
                                 desc_mnmajor_sw64(base + Ly::K + 1024 * kk, 8192), idesc_bf16_amn_bmn(128, 32), kk);
                }
                mma_commit(bar_o);
            }
            o_pend = true;
            ok = mbar_wait(bar_o, ph_mma, st.wait_ns);
            if (__syncthreads_or(!ok)) { failed = true; break; }
            ph_mma ^= 1;
            o_pend = false;
            tc_fence_after();
            // q and do are free: the next query tile's (or the next unit's first)
            // loads run under the epilogue
            if (qt + 1 < KT) {
                if (tid == 0) load_q(head, win, qt + 1);
                q_pend = true;
            } else if (u + 1 < u_end) {
                int h1, k1;
                int64_t w1;
                decode(u + 1, h1, w1, k1);
                if (tid == 0) load_q(h1, w1, 0);
                q_pend = true;
            }

            // ---- dv / dk of key row r into registers; dq of query row r to the fp32 buffer ----
            {
                float a[32];
                tmem_ld32(t_lane + 32 * h2, a);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] += a[c];
                float dq[16];
                tmem_ld16(t_lane + 64 + 16 * h2, dq);
                tmem_wait_ld();
                const int q = qt * 128 + r;
                if (q < N) {
                    float4 *dst = reinterpret_cast<float4 *>(dq_acc + (win * N + q) * C + head * 32 + 16 * h2);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        atomicAdd(dst + c, make_float4(dq[4 * c], dq[4 * c + 1], dq[4 * c + 2], dq[4 * c + 3]));
                }
            }
            tc_fence_before();
            __syncthreads();
        }
        if (failed) break;
        // the next unit's k and v (this unit's MMAs are done; V2 reads the k
        // rows below, so its load waits for the barrier at the end)
        if (!v2 && u + 1 < u_end) {
            if (tid == 0) load_kv(u + 1);
            kv_pend = true;
        }
        // dv (first four warps) and dk (last four) of key row r, back to the token's place
        if (kvalid) {
            const int64_t tok = window_row_to_token(g, win * N + j);
            if (h2 == 1) {
                // dk = scale dS^T q (V2: then through k's unit-length scaling)
                const float nrm = v2 ? norms[(win * N + j) * (2 * heads) + heads + head] : 1.f;
                fb_unit_backward(acc, base + Ly::K, r, scale / nrm, v2 != 0);
            }
            bf16 *dst = dqkv + tok * 3 * C + (h2 == 0 ? 2 * C : C) + head * 32;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 w;
                w.x = pack_bf16x2(acc[8 * q4], acc[8 * q4 + 1]);
                w.y = pack_bf16x2(acc[8 * q4 + 2], acc[8 * q4 + 3]);
                w.z = pack_bf16x2(acc[8 * q4 + 4], acc[8 * q4 + 5]);
                w.w = pack_bf16x2(acc[8 * q4 + 6], acc[8 * q4 + 7]);
                *reinterpret_cast<uint4 *>(dst + 8 * q4) = w;
            }
        }
        __syncthreads();
        if (v2 && u + 1 < u_end) {
            if (tid == 0) load_kv(u + 1);
            kv_pend = true;
        }
    }
    if (failed) {
        // copies and MMAs still in flight finish (bounded waits) before the
        // shared memory and TMEM are given up
        if (tid == 0) {
            atomicOr(st.err, ERR_TIMEOUT);
            if (kv_pend) mbar_wait(bar_kv, ph_kv, st.wait_ns);
            if (q_pend) mbar_wait(bar_q, ph_q, st.wait_ns);
            if (s_pend) mbar_wait(bar_s, ph_mma, st.wait_ns);
            if (o_pend) mbar_wait(bar_o, ph_mma, st.wait_ns);
        }
    } else if (cur_head >= 0) {
        flush_head();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// D_i = do_i . o_i per (row, head): do in window order, o in token order.
__global__ void rowdot_kernel(const bf16 *dO, const bf16 *o, Geom g, int heads, float *D)
{
    const int64_t total = g.T * heads;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / heads;
        const int hd = (int)(e - row * heads);
        const int64_t tok = window_row_to_token(g, row);
        const uint4 *a = reinterpret_cast<const uint4 *>(dO + row * g.C + hd * 32);
        const uint4 *b = reinterpret_cast<const uint4 *>(o + tok * g.C + hd * 32);
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 ua = a[q], ub = b[q];
            const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 x = unpack_bf16x2(wa[t]), y = unpack_bf16x2(wb[t]);
                s = fmaf(x.x, y.x, fmaf(x.y, y.y, s));
            }
        }
        D[e] = s;
    }
}

// dq of each (row, head) from the fp32 sums: scale (V2: 1/max(tau, 0.01), then
// through q's unit-length scaling, q^ from qkv and its norm), bf16 into dqkv
// at the row's token.
__global__ void dq_finalize_kernel(const float *dq_acc, const bf16 *qkv, const float *norms, const float *tau,
                                   int v2, Geom g, int heads, bf16 *dqkv)
{
    const int64_t total = g.T * heads;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / heads;
        const int hd = (int)(e - row * heads);
        const int C = g.C;
        float du[32];
        const float4 *src = reinterpret_cast<const float4 *>(dq_acc + row * C + hd * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 f = src[q];
            du[4 * q] = f.x;
            du[4 * q + 1] = f.y;
            du[4 * q + 2] = f.z;
            du[4 * q + 3] = f.w;
        }
        float f = 0.17677669529663687f;
        if (v2) {
            const float sc = 1.0f / fmaxf(tau[hd], 0.01f);
            const float nrm = norms[row * (2 * heads) + hd];
            const uint4 *u4 = reinterpret_cast<const uint4 *>(qkv + row * 3 * C + hd * 32);
            float u[32];
            float dot = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 w = u4[q];
                const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const float2 p = unpack_bf16x2(w4[t]);
                    u[8 * q + 2 * t] = p.x;
                    u[8 * q + 2 * t + 1] = p.y;
                }
            }
#pragma unroll
            for (int c = 0; c < 32; ++c) dot = fmaf(u[c], du[c], dot);
#pragma unroll
            for (int c = 0; c < 32; ++c) du[c] -= u[c] * dot;
            f = sc / nrm;
        }
        const int64_t tok = window_row_to_token(g, row);
        uint4 *dst = reinterpret_cast<uint4 *>(dqkv + tok * 3 * C + hd * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(du[8 * q] * f, du[8 * q + 1] * f), pack_bf16x2(du[8 * q + 2] * f, du[8 * q + 3] * f),
                                pack_bf16x2(du[8 * q + 4] * f, du[8 * q + 5] * f), pack_bf16x2(du[8 * q + 6] * f, du[8 * q + 7] * f));
    }
}

unsigned grid_for(int64_t n)
{
    const int64_t want = (n + 255) / 256;
    return (unsigned)(want < 152 * 16 ? (want > 0 ? want : 1) : 152 * 16);
}

} // namespace

bool attn_flash_backward_supported(int M, int C, int heads)
{
    return M * M > 64 && C == heads * 32 && FbLayout::bytes(M) <= 113 * 1024;
}

cudaError_t launch_attn_flash_backward(const bf16 *qkv, const bf16 *dO, const bf16 *attn, const bf16 *table,
                                       const float *tau, int heads, int v2, const Geom &g, const float *lse, float *D,
                                       const float *norms, bf16 *dqkv, float *dq_acc, float *dtable, float *dtau,
                                       DeviceStatus st, cudaStream_t stream)
{
    if (!attn_flash_backward_supported(g.M, g.C, heads)) return cudaErrorInvalidValue;
    cudaError_t e;
    rowdot_kernel<<<grid_for(g.T * heads), 256, 0, stream>>>(dO, attn, g, heads, D);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    CUtensorMap tm_qkv, tm_do;
    e = make_tensor_map_sw64(&tm_qkv, qkv, g.T, 3 * g.C, 128, false);
    if (e == cudaSuccess) e = make_tensor_map_sw64(&tm_do, dO, g.T, g.C, 128, false);
    if (e != cudaSuccess) return e;
    const size_t smem = FbLayout::bytes(g.M);
    e = cudaFuncSetAttribute(attn_flash_backward_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    }
    const int64_t units = (int64_t)heads * g.nwin * ((g.N + 127) / 128);
    const int64_t cap = (int64_t)sms * 2;
    const unsigned grid = (unsigned)(units < cap ? units : cap);
    attn_flash_backward_kernel<<<grid, FB_THREADS, smem, stream>>>(table, tau, heads, v2, g, lse, D, norms, dqkv, dq_acc,
                                                                   dtable, dtau, st, tm_qkv, tm_do);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    dq_finalize_kernel<<<grid_for(g.T * heads), 256, 0, stream>>>(dq_acc, qkv, norms, tau, v2, g, heads, dqkv);
    return cudaGetLastError();
}

} // namespace swin
