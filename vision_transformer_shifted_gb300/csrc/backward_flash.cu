// Backward of the shifted-window attention for windows of more than 64
// tokens (SwinV2 at window 24: 576 tokens), on tcgen05 tensor cores.
//
// Same gradients as the short-window kernel (csrc/backward.cu): with the
// row-wise softmax normaliser of the forward (its log2, lse, kept by the
// large-window forward kernel) P = exp2(logit2 - lse) needs no row reduction,
// so a CTA can own a tile of 128 KEYS of one window and head and walk over
// the window's query tiles (key-stationary order):
//   S^T  = k q^T and dP^T = v do^T            (M = 128 keys, N = 128 queries, K = 32)
//   P^T, dS^T = P^T (dP^T - D), D_i = do_i . o_i (computed beforehand)
//   dv  += P^T do,  dk += dS^T q             (P^T from TMEM; both kept in registers
//                                             across query tiles)
//   dq_i += dS k                             (M = 128 queries: dS^T read M-major;
//                                             added to an fp32 buffer by atomics, since
//                                             every key tile of the window contributes)
// and the table gradient of each relative offset summed in shared memory per
// head as fixed-point integers (units run head by head, a contiguous range per
// CTA).  A last kernel turns the fp32 dq into bf16 (scale, and for V2 the
// unit-length backward).
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int FB_THREADS = 256;
constexpr int FB_MAX_TILES = 5;   // windows of up to 640 tokens

// Table-gradient terms are summed in shared memory as fixed-point integers
// (shared-memory integer atomics are far cheaper than floating-point ones):
// a term x with |x| < FIX_MAX becomes round(x * 2^19).  One table entry gets at
// most one term per key of a (key tile, query tile) pair, so a unit (at most
// FB_MAX_TILES query tiles of 128 keys) adds at most 640 terms, each below
// 2^21 in size: the 32-bit sum cannot overflow, and it is moved into the fp32
// table after every unit.  Larger terms go to the fp32 table directly.
constexpr float FIX_SCALE = 524288.0f, FIX_INV = 1.0f / 524288.0f, FIX_MAX = 4.0f;
static_assert(FB_MAX_TILES * 128 * 4.0 * 524288.0 < 2147483647.0, "fixed-point table sums may overflow");
// round(y) for |y| < 2^22 through the float adder: y + 1.5 * 2^23 lies in
// [2^23, 2^24), where floats are spaced by exactly 1, so the addition rounds y
// to the nearest integer and the low mantissa bits hold it (offset by the
// bits of 1.5 * 2^23).
__device__ __forceinline__ int fb_round_fix(float x)
{
    return __float_as_int(fmaf(x, FIX_SCALE, 12582912.0f)) - 0x4B400000;
}

struct FbLayout {
    // byte offsets from the 512-aligned base
    static constexpr uint32_t K = 0, V = 8192, Q = 16384, DO = 24576; // [128 rows][64 B] tiles
    static constexpr uint32_t DS = 32768;                              // 4 panels [128 keys][32 queries]
    // per query of the tile: its relative-index bases in the bias table and in
    // the padded gradient table, and its shift region (-1: no query)
    static constexpr uint32_t QC = 65536;                              // int [128]
    static constexpr uint32_t LSE = QC + 512;                          // float [128]
    static constexpr uint32_t DD = LSE + 512;                          // float [128]
    static constexpr uint32_t BIAS = DD + 512;                         // bf16 [(2M-1)^2] of the current head
    __host__ __device__ static uint32_t ll_pad(int M) { return ((uint32_t)(2 * M - 1) * (2 * M - 1) + 7u) & ~7u; }
    // Row stride of the shared table gradient (>= 2M-1, = M mod 32): for one
    // query, a warp's 32 consecutive keys address consecutive words within a
    // window row, and the step to the next row (-(stride - M + 1)) is then
    // also -1 modulo 32, so the 32 lanes of one atomic add fall in 32 banks.
    __host__ __device__ static int lp(int M) { return M + 32 * ((M - 1 + 31) / 32); }
    __host__ __device__ static uint32_t dt_pad(int M) { return ((uint32_t)(2 * M - 1) * lp(M) + 3u) & ~3u; }
    // the table gradient: fp32, and the fixed-point sums of the current unit
    __host__ __device__ static uint32_t dtab(int M) { return BIAS + 2 * ll_pad(M); }
    __host__ __device__ static uint32_t dti(int M) { return dtab(M) + 4 * dt_pad(M); }
    __host__ __device__ static uint32_t bar(int M) { return dti(M) + 4 * dt_pad(M); }
    // four mbarriers, then the TMEM address slot
    // (64-byte swizzle atoms repeat every 512 bytes: the base is 512-aligned)
    static size_t bytes(int M) { return (size_t)bar(M) + 48 + 512; }
};

template <bool B>
struct FbTag {
    static constexpr bool value = B;
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
    uint8_t *sm = smem_align(smraw, 512);
    const uint32_t base = smem_u32(sm);
    const int N = g.N, M = g.M, C = g.C, L = 2 * M - 1, LL = L * L, LP = Ly::lp(M);
    const int KT = (N + 127) / 128;                 // key tiles and query tiles per window
    int *qcode = reinterpret_cast<int *>(sm + Ly::QC);
    float *slse = reinterpret_cast<float *>(sm + Ly::LSE);
    float *sdd = reinterpret_cast<float *>(sm + Ly::DD);
    const bf16 *sbias = reinterpret_cast<const bf16 *>(sm + Ly::BIAS);
    float *dtab = reinterpret_cast<float *>(sm + Ly::dtab(M));
    int *dti = reinterpret_cast<int *>(sm + Ly::dti(M));
    const uint32_t bar_kv = base + Ly::bar(M), bar_q = bar_kv + 8, bar_s = bar_kv + 16, bar_o = bar_kv + 24;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Ly::bar(M) + 32);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, h2 = warp >> 2;
    const int r = quad * 32 + lane;                  // TMEM lane: key row (S^T), or query row (dq)
    const int per = g.nh * g.nw;
    const int64_t nunits = (int64_t)heads * g.nwin * KT;
    const float LOG2E = 1.4426950408889634f;

    for (int e = tid; e < (int)Ly::dt_pad(M); e += FB_THREADS) {
        dtab[e] = 0.f;
        dti[e] = 0;
    }
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
    // threads 0..127: lse and D of query `tid` of the next query tile, fetched
    // one tile ahead so that their latency hides under the previous epilogue
    float nl = 0.f, nd = 0.f;
    auto fetch_rows = [&](int hd, int64_t w, int qt_) {
        if (tid < 128) {
            const int q = qt_ * 128 + tid;
            nl = nd = 0.f;
            if (q < N) {
                nl = lse[(w * N + q) * heads + hd];
                nd = Dr[(w * N + q) * heads + hd];
            }
        }
    };

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
            float *t = dtab + (e / L) * LP + (e - (e / L) * L);
            if (*t != 0.f) atomicAdd(&dtable[(int64_t)e * heads + cur_head], *t);
            *t = 0.f;
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
        fetch_rows(h0, w0, 0);
    }
    int step = 0;   // query-tile steps of this CTA (phase trace only)
    (void)step;
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
            // (the barrier before the first MMA below orders these writes)
        }
        const float sc2 = scale * LOG2E;
        // this thread's key (S^T row r); keys past the window match no query
        const int j = kt * 128 + r;
        const bool kvalid = j < N;
        const int kofs = kvalid ? (j / M) * L + (j % M) : 0;
        const int kofsp = kvalid ? (j / M) * LP + (j % M) : 0;
        const int kreg = kvalid ? fb_region(g, wi, wj, j) : 0x7FFF;
        float acc[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) acc[c] = 0.f;

        for (int qt = 0; qt < KT; ++qt, ++step) {
            // the query tile's metadata (its previous readers passed the P
            // store barrier of the last tile)
            if (tid < 128) {
                const int q = qt * 128 + tid;
                int code = -1;
                if (q < N) {
                    const int qi = q / M, qj = q - (q / M) * M;
                    code = ((qi + M - 1) * L + (qj + M - 1)) | (((qi + M - 1) * LP + (qj + M - 1)) << 12) |
                           (fb_region(g, wi, wj, q) << 24);
                }
                qcode[tid] = code;
                slse[tid] = nl;
                sdd[tid] = nd;
            }
            bool ok = true;
            if (qt == 0) ok = mbar_wait(bar_kv, ph_kv, st.wait_ns);
            ok = ok && mbar_wait(bar_q, ph_q, st.wait_ns);
            // A: tiles landed, metadata visible, the last TMEM reads done
            tc_fence_before();
            if (__syncthreads_or(!ok || failed)) { failed = true; break; }
            tc_fence_after();
            if (qt == 0) { ph_kv ^= 1; kv_pend = false; }
            ph_q ^= 1;
            q_pend = false;
            if (tid == 0 || tid == 128) {
                // S^T by thread 0, dP^T by thread 128
                const uint32_t id = idesc_bf16(128, 128);
                const uint32_t a = tid == 0 ? Ly::K : Ly::V, b = tid == 0 ? Ly::Q : Ly::DO;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16(tmem + (tid == 0 ? 0 : 128), desc_kmajor_sw64(base + a + 32 * ks),
                             desc_kmajor_sw64(base + b + 32 * ks), id, ks);
                mma_commit(bar_s);
            }
            s_pend = true;
            if (mbar_wait(bar_s, ph_mma, st.wait_ns)) s_pend = false;
            else failed = true;     // (uniform at the next barrier)
            tc_fence_after();

            // ---- P^T and dS^T of key row r, queries 64*h2 .. +63, 8 at a time ----
            // (FULL: every pair of the pass is valid -- an unmasked window, a real
            // key, eight real queries -- so no pair needs a check)
            auto pass = [&](auto full_tag, int hh) {
                constexpr bool FULL = decltype(full_tag)::value;
                const int i0 = 64 * h2 + 8 * hh;
                float s[8], d[8];
                tmem_ld8(t_lane + i0, s);
                tmem_ld8(t_lane + 128 + i0, d);
                int idx[8], idxp[8];   // bias and gradient table entries (-1: masked pair)
                {
                    const int4 *c4 = reinterpret_cast<const int4 *>(qcode + i0);
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const int4 c = c4[v];
                        const int cc[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const bool valid = FULL || (cc[t] >> 24) == kreg;
                            idx[4 * v + t] = valid ? (cc[t] & 0xFFF) - kofs : -1;
                            idxp[4 * v + t] = ((cc[t] >> 12) & 0xFFF) - kofsp;
                        }
                    }
                }
                // every bias load ahead of the table-gradient atomics below
                float bv[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    bv[jj] = __bfloat162float(sbias[FULL || idx[jj] >= 0 ? idx[jj] : 0]);
                tmem_wait_ld();
                float amax = 0.f;
                {
                    const float4 *l4 = reinterpret_cast<const float4 *>(slse + i0);
                    const float4 *d4 = reinterpret_cast<const float4 *>(sdd + i0);
#pragma unroll
                    for (int v = 0; v < 2; ++v) {
                        const float4 lv = l4[v], dv = d4[v];
                        const float ll[4] = {lv.x, lv.y, lv.z, lv.w}, dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int jj = 4 * v + t;
                            const float e = ex2_approx(fmaf(s[jj], sc2, fmaf(bv[jj], LOG2E, -ll[t])));
                            const float p = FULL || idx[jj] >= 0 ? e : 0.f;
                            const float ds = p * (d[jj] - dd[t]);
                            if (v2) tau_acc = fmaf(ds, s[jj], tau_acc);
                            s[jj] = p;
                            d[jj] = ds;
                            amax = fmaxf(amax, fabsf(ds));
                        }
                    }
                }
                // P^T of queries i0 .. i0+7 as bf16 pairs over TMEM columns
                // 64 h2 + 4 hh .. +3 (S^T columns this thread has read already);
                // dS^T to shared panel i0 / 32, 16-byte chunk i0 / 8 mod 4
                tmem_st4(t_lane + 64 * h2 + 4 * hh, pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]),
                         pack_bf16x2(s[4], s[5]), pack_bf16x2(s[6], s[7]));
                fb_store8(base + Ly::DS + (uint32_t)(i0 >> 5) * 8192u + sw64_offset(r, hh & 3), d);
                if (__all_sync(0xffffffffu, amax < FIX_MAX)) {
                    // the common case: every term of the warp on the fixed-point grid
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        if (FULL || idx[jj] >= 0) atomicAdd(&dti[idxp[jj]], fb_round_fix(d[jj]));
                } else {
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        if (!FULL && idx[jj] < 0) continue;
                        if (fabsf(d[jj]) < FIX_MAX) atomicAdd(&dti[idxp[jj]], fb_round_fix(d[jj]));
                        else atomicAdd(&dtab[idxp[jj]], d[jj]);
                    }
                }
            };
            const bool unmasked = g.s == 0 || (wi != g.nh - 1 && wj != g.nw - 1);
#pragma unroll 1
            for (int hh = 0; hh < 8; ++hh) {
                // the choice is made for the whole warp (a window's last key tile
                // can end inside a warp): both passes hold warp-collective TMEM
                // accesses and a vote, which every lane must reach together
                if (__all_sync(0xffffffffu, unmasked && kvalid && qt * 128 + 64 * h2 + 8 * hh + 8 <= N))
                    pass(FbTag<true>(), hh);
                else
                    pass(FbTag<false>(), hh);
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            // B: P^T and dS^T panels complete
            if (__syncthreads_or(failed)) { failed = true; break; }
            if (lane == 0 && (warp == 0 || warp == 1 || warp == 4)) {
                // TMEM columns: P^T over 0..31 and 64..95; dv (warp 0) into
                // 32..63, dk (warp 1) into 96..127, dq (warp 4) into 160..191
                tc_fence_after();
                const int which = warp == 0 ? 0 : (warp == 1 ? 1 : 2);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t kpan = (uint32_t)(kk >> 1) * 8192u + 32u * (kk & 1);
                    if (which == 0)
                        mma_bf16_ts(tmem + 32, tmem + 64 * (kk >> 2) + 8 * (kk & 3),
                                    desc_mnmajor_sw64(base + Ly::DO + 1024 * kk, 8192), idesc_bf16_bmn(128, 32), kk);
                    else if (which == 1)
                        mma_bf16(tmem + 96, desc_kmajor_sw64(base + Ly::DS + kpan),
                                 desc_mnmajor_sw64(base + Ly::Q + 1024 * kk, 8192), idesc_bf16_bmn(128, 32), kk);
                    else
                        mma_bf16(tmem + 160, desc_mnmajor_sw64(base + Ly::DS + 1024 * kk, 8192),
                                 desc_mnmajor_sw64(base + Ly::K + 1024 * kk, 8192), idesc_bf16_amn_bmn(128, 32), kk);
                }
                mma_commit(bar_o);
            }
            o_pend = true;
            if (mbar_wait(bar_o, ph_mma, st.wait_ns)) o_pend = false;
            else failed = true;     // (uniform at the next barrier)
            ph_mma ^= 1;
            tc_fence_after();
            // q and do are free (every MMA reading them has completed): the
            // next query tile's (or the next unit's first) loads and row data
            // come in under the epilogue
            if (qt + 1 < KT) {
                if (tid == 0 && !failed) load_q(head, win, qt + 1);
                q_pend = true;
                fetch_rows(head, win, qt + 1);
            } else if (u + 1 < u_end) {
                int h1, k1;
                int64_t w1;
                decode(u + 1, h1, w1, k1);
                if (tid == 0 && !failed) load_q(h1, w1, 0);
                q_pend = true;
                fetch_rows(h1, w1, 0);
            }

            // ---- dv / dk of key row r into registers; dq of query row r to the fp32 buffer ----
            {
                float a[32];
                tmem_ld32(t_lane + 32 + 64 * h2, a);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) acc[c] += a[c];
                float dq[16];
                tmem_ld16(t_lane + 160 + 16 * h2, dq);
                tmem_wait_ld();
                const int q = qt * 128 + r;
                if (q < N) {
                    float4 *dst = reinterpret_cast<float4 *>(dq_acc + (win * N + q) * C + head * 32 + 16 * h2);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        atomicAdd(dst + c, make_float4(dq[4 * c], dq[4 * c + 1], dq[4 * c + 2], dq[4 * c + 3]));
                }
            }
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
        // the k tile and the bias matrix are read by now; TMEM reads done
        tc_fence_before();
        __syncthreads();
        // this unit's fixed-point table sums into the fp32 table (the next
        // unit's first barrier orders this before its atomics)
        for (int e = tid; e < (int)Ly::dt_pad(M); e += FB_THREADS) {
            const int v = dti[e];
            if (v != 0) {
                dtab[e] = fmaf((float)v, FIX_INV, dtab[e]);
                dti[e] = 0;
            }
        }
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
    // (the table bases of a query are packed in 12 bits each)
    return M * M > 64 && (M * M + 127) / 128 <= FB_MAX_TILES && C == heads * 32 &&
           (2 * M - 2) * (FbLayout::lp(M) + 1) < 4096 &&
           FbLayout::bytes(M) <= 113 * 1024;
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
