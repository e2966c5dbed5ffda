// The whole shifted-window attention block in one persistent kernel
// (sm_103a, tcgen05 + TMEM), for windows of at most 64 tokens (M = 7, 8) and
// C = 64 or 96 channels (2 or 3 heads of 32).
//
// Steps, per tile of two windows (pages "Boosting Swin Transformer Speed",
// Introduction / Training Optimization / Inference Optimization; "Swin
// Transformer V2" (neura.market), How It Works):
//   S1  the tile's 2 x N tokens are gathered from x through the cyclic shift
//       by -s and the window partition (cp.async, one 16-byte chunk each);
//       window A fills rows 0..63 of a 128-row tile, window B rows 64..127
//   S2  [q|k] = X Wqk^T (128 x 2C) and v^T = Wv X^T (C x 128), both on
//       tcgen05 into TMEM; bias added when draining to shared memory; V2
//       normalises q and k to unit length in fp32 while draining
//   S3-S5 per head: S = q k^T (128 x 128 x 32) into TMEM; softmax of each
//       row over its own window's keys with the relative bias and the shift
//       mask computed from coordinates (fp32, exp2); P (bf16) back into TMEM
//       over the S columns
//   S6  o_h = P v_h (128 x 32 x 128) into TMEM, with P read from TMEM as the
//       A operand (so P never touches shared memory)
//   S7  y = (o / rowsum) Wproj^T on tcgen05, o staged as bf16 in the freed X
//       buffer
//   S8  y + bproj written straight from registers through the window
//       reverse + roll(+s) map into out[B, H, W, C]
// Nothing but x, the weights and out touches HBM.  The next tile's x is
// fetched with cp.async while the current one is computed.
//
// Warp roles: warps 0..7 compute (warp w serves TMEM lane quarter w % 4 =
// tile rows 32(w%4)..+31 and column half w / 4; every drain and the softmax
// split their columns between the two halves); warp 8 issues every tcgen05
// MMA.  They hand over through mbarriers: the compute warps arrive on
// "ready" barriers (one arrival per warp) once operands are in shared memory,
// the MMA warp commits "done" barriers.  The MMA warp issues the next tile's
// QKV projection as soon as the current tile's last softmax has freed TMEM
// columns 0..2C+127, so it runs under the current tile's P.V, o drain,
// projection and store.
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int FTHREADS = 288;          // 8 compute warps + 1 MMA warp
constexpr int NCOMPUTE = 256;
constexpr int NCWARPS = NCOMPUTE / 32;
constexpr float FLOG2E = 1.4426950408889634f;

// Optional phase trace (builds with -DSWIN_PHASE_TRACE only): thread 0 of
// CTA 0 records clock64() at the phase boundaries of its first tiles.
#ifdef SWIN_PHASE_TRACE
constexpr int TRACE_TILES = 16, TRACE_POINTS = 32;
__device__ long long g_phase_trace[2 * TRACE_TILES * TRACE_POINTS];
__device__ long long g_cta_trace[1024 * 4];
#define PHASE(k, i)                                                                                  \
    do {                                                                                             \
        if (blockIdx.x == 0 && (tid == 0 || tid == 128) && (k) < TRACE_TILES)                       \
            g_phase_trace[((tid >> 7) * TRACE_TILES + (k)) * TRACE_POINTS + (i)] = clock64();        \
    } while (0)
#else
#define PHASE(k, i) \
    do {            \
    } while (0)
#endif

template <int M, int C>
struct FusedCfg {
    static constexpr int N = M * M;
    static constexpr int HEADS = C / 32;
    static constexpr int L = 2 * M - 1;
    static constexpr int KB = C / 32;         // 32-channel K blocks (64-byte swizzle)
    // shared memory (bytes); SW64 tiles are 512-aligned, SW128 tiles 1024-aligned
    static constexpr int WQK = 0;                       // [2C rows][C]   SW64
    static constexpr int WV = WQK + 2 * C * C * 2;      // [128 rows][C]  SW64 (rows >= C zero)
    static constexpr int WP = WV + 128 * C * 2;         // [C rows][C]    SW64
    // x tile (then o) buffers X0 and X1; each is followed by scratch that is
    // free when the tile's output is staged (Q and K after X0, V^T after X1),
    // so the output staging rows (stride SROW) of buffer b start at X(b)
    static constexpr int XSZ = 128 * C * 2;
    static constexpr int X0 = WP + C * C * 2;           // [128][C]       SW64 (x, then o)
    static constexpr int Q = X0 + XSZ;                  // [128][32]      SW64
    static constexpr int K = Q + 128 * 64;
    static constexpr int X1 = K + 128 * 64;
    static constexpr int VT = X1 + XSZ;                 // 2 x [C rows][64 keys] SW128
    static constexpr int VT_BLK = C * 128;
    static constexpr int SROW = 2 * C + 16;             // staging row stride (bank-conflict free)
    static_assert(128 * SROW <= XSZ + 2 * 128 * 64 && 128 * SROW <= XSZ + 2 * VT_BLK, "staging fits");
    static constexpr int P = VT + 2 * VT_BLK;           // 2 x [128 rows][64 keys] SW128
    static constexpr int SMALL = P + 2 * 128 * 128;
    static constexpr int BYTES = SMALL + HEADS * L * L * 4 + 3 * C * 4 + C * 4 + HEADS * 4 + 2 * 128 * 4 +
                                 HEADS * 2 * 128 * 4 + 3 * 128 * 4 + 2 * 64 * 4 + 16 * 8 + 16 + 16;
    // TMEM columns
    static constexpr int T_QK = 0;                      // 2C
    static constexpr int T_VT = 2 * C;                  // 128 (v^T), then S
    static constexpr int T_S = T_VT;
    static constexpr int T_O = T_VT + 128;              // C
    static constexpr int T_Y = T_O + C;                 // C
    static_assert(T_Y + C <= 512, "TMEM budget");
    static_assert(N <= 64, "two windows per 128-row tile");
};

struct FusedArgs {
    const bf16 *x, *Wqkv, *bqkv, *table, *Wproj, *bproj;
    const float *tau;
    bf16 *out;
    int mode;
    Geom g;
};

// Barrier among the 256 compute threads (named barrier 1); returns the OR of
// `v` over them, so that a failure seen by one thread is seen by all.
__device__ __forceinline__ bool compute_sync_or(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// Bounded wait that also gives up as soon as another thread has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}

// One arrival per warp on a ready barrier: every lane's prior shared-memory
// writes (made visible to the async proxy by the caller) and TMEM loads
// happen before it.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

template <int M, int C>
__global__ void __launch_bounds__(FTHREADS, 1) fused_block_kernel(FusedArgs a, DeviceStatus st)
{
    using F = FusedCfg<M, C>;
    constexpr int N = F::N, HEADS = F::HEADS, L = F::L, KB = F::KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    float *sbias = reinterpret_cast<float *>(sm + F::SMALL);        // [HEADS][L*L], times log2(e)
    float *sbqkv = sbias + HEADS * L * L;                             // [3C]
    float *sbproj = sbqkv + 3 * C;                                    // [C]
    float *sscale = sbproj + C;                                       // [HEADS]
    float *smax = sscale + HEADS;                                     // [2][128] partial row maxima
    float *spart = smax + 2 * 128;                                    // [HEADS][2][128] partial row sums
    // token of each tile row (-1 if none), three rotating copies: tile k uses
    // copy k % 3 and fills copy (k + 1) % 3 for the next tile while other warps
    // may still read copy (k - 1) % 3 for the previous tile's stores
    int *rowtok = reinterpret_cast<int *>(spart + HEADS * 2 * 128);   // [3][128]
    int *key_region = rowtok + 3 * 128;                               // [2][64]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_align(reinterpret_cast<uint8_t *>(key_region + 2 * 64), 8));
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 16);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    __shared__ int slot_masked[2];

    const Geom g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool is_mma = warp == NCWARPS;
    const int quarter = warp & 3, half = (warp >> 2) & 1;
    const int row = quarter * 32 + lane;       // tile row = TMEM lane
    const int slot = row >> 6, t = row & 63;   // window slot and token of the row
    const uint32_t base = smem_u32(sm);
    // done barriers (tcgen05.commit) and ready barriers (one arrival per compute warp)
    const uint32_t B_QKV = smem_u32(&bars[0]), B_S = smem_u32(&bars[1]), B_PV = smem_u32(&bars[2]),
                   B_Y = smem_u32(&bars[3]);
    const uint32_t R_QK = smem_u32(&bars[4]), R_P = smem_u32(&bars[5]), R_O = smem_u32(&bars[6]),
                   R_FREE = smem_u32(&bars[7]);
    const int64_t ntiles = (g.nwin + 1) / 2;
    auto xbuf = [&](int buf) { return buf ? F::X1 : F::X0; };

    // ---- once per CTA: weights, biases, tables, barriers, TMEM ---------------
    if (!is_mma) {
        for (int q = tid; q < (2 * C) * (C / 8); q += NCOMPUTE) {     // Wq, Wk rows
            const int r = q / (C / 8), c16 = q % (C / 8);
            cp_async16(base + F::WQK + (c16 >> 2) * (2 * C * 64) + sw64_offset(r, c16 & 3),
                       a.Wqkv + (int64_t)r * C + c16 * 8, 16);
        }
        for (int q = tid; q < 128 * (C / 8); q += NCOMPUTE) {         // Wv rows, zero past C
            const int r = q / (C / 8), c16 = q % (C / 8);
            const bool ok = r < C;
            cp_async16(base + F::WV + (c16 >> 2) * (128 * 64) + sw64_offset(r, c16 & 3),
                       ok ? a.Wqkv + (int64_t)(2 * C + r) * C + c16 * 8 : a.Wqkv, ok ? 16u : 0u);
        }
        for (int q = tid; q < C * (C / 8); q += NCOMPUTE) {           // Wproj
            const int r = q / (C / 8), c16 = q % (C / 8);
            cp_async16(base + F::WP + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3),
                       a.Wproj + (int64_t)r * C + c16 * 8, 16);
        }
        for (int i = tid; i < HEADS * L * L; i += NCOMPUTE) {
            const int hd = i / (L * L), e = i % (L * L);
            sbias[i] = __bfloat162float(a.table[(int64_t)e * HEADS + hd]) * FLOG2E;
        }
        for (int i = tid; i < 3 * C; i += NCOMPUTE) sbqkv[i] = a.bqkv ? __bfloat162float(a.bqkv[i]) : 0.f;
        for (int i = tid; i < C; i += NCOMPUTE) sbproj[i] = a.bproj ? __bfloat162float(a.bproj[i]) : 0.f;
        if (tid < HEADS)
            sscale[tid] = a.mode == 1 ? FLOG2E / fmaxf(a.tau[tid], 0.01f) : FLOG2E * rsqrtf(32.0f);
    }
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
        for (int i = 4; i < 8; ++i) mbar_init(smem_u32(&bars[i]), NCWARPS);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (is_mma) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }

    // token (b*H*W + i*W + j) of every row of tile `tile`, -1 for padding rows
    // and a missing second window; rows 0..127 by threads 0..127
    auto row_tokens = [&](int64_t tile, int *dst) {
        if (tid < 128) {
            const int sl = tid >> 6, tt = tid & 63;
            const int win = (int)(2 * tile) + sl;
            dst[tid] = (tile < ntiles && tt < N && win < g.nwin) ? window_row_to_token32(g, win * N + tt) : -1;
        }
    };
    // x rows of the tile whose row tokens are in `tok` into X buffer `buf`
    // (zeros where tok < 0); compute threads only
    auto load_x = [&](const int *tok, int buf) {
        const uint32_t xb = base + xbuf(buf);
#pragma unroll
        for (int i = 0; i < 128 * (C / 8) / NCOMPUTE; ++i) {
            const int q = tid + NCOMPUTE * i;
            const int r = q / (C / 8), c16 = q % (C / 8);
            const int tk = tok[r];
            const bf16 *src = tk >= 0 ? a.x + (int64_t)tk * C + c16 * 8 : a.x;
            cp_async16(xb + (c16 >> 2) * (128 * 64) + sw64_offset(r, c16 & 3), src, tk >= 0 ? 16u : 0u);
        }
        cp_async_commit();
    };
#ifdef SWIN_PHASE_TRACE
    if (tid == 0) g_cta_trace[blockIdx.x * 4 + 0] = (long long)global_timer_ns();
#endif
    row_tokens(blockIdx.x, rowtok);
    __syncthreads();
    if (!is_mma) {
        load_x(rowtok, 0);
        cp_async_wait<0>();
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();   // weights, tables, the first tile's x, barriers, TMEM address
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (is_mma) {
        // ===================== MMA warp (lane 0 issues) =====================
        if (lane == 0) {
            uint32_t ph_qk = 0, ph_p = 0, ph_o = 0, ph_free = 0, ph_pv_m = 0;
            const uint32_t id_qk = idesc_bf16(128, 2 * C), id_vt = idesc_bf16(128, 128);
            const uint32_t id_s = idesc_bf16(128, 128), id_pv = idesc_bf16(128, 32), id_y = idesc_bf16(128, C);
            auto issue_qkv = [&](int buf) {
                const uint32_t xb = base + xbuf(buf);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_QK, desc_kmajor_sw64(xb + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(base + F::WQK + kb * (2 * C * 64) + 32 * ks), id_qk, (kb | ks) != 0);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_VT, desc_kmajor_sw64(base + F::WV + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(xb + kb * (128 * 64) + 32 * ks), id_vt, (kb | ks) != 0);
                mma_commit(B_QKV);
            };
            int k = 0;
            if ((int64_t)blockIdx.x < ntiles) issue_qkv(0);
#pragma unroll 1
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
                const int buf = k & 1;
                bool ok = true;
#pragma unroll 1
                for (int hd = 0; hd < HEADS && ok; ++hd) {
                    ok = wait_or_abort(R_QK, ph_qk, st.wait_ns, abort_flag);
                    ph_qk ^= 1;
                    if (!ok) break;
                    tc_fence_after();
                    mma_bf16(tmem + F::T_S, desc_kmajor_sw64(base + F::Q), desc_kmajor_sw64(base + F::K), id_s, 0);
                    mma_bf16(tmem + F::T_S, desc_kmajor_sw64(base + F::Q + 32), desc_kmajor_sw64(base + F::K + 32),
                             id_s, 1);
                    mma_commit(B_S);
                    ok = wait_or_abort(R_P, ph_p, st.wait_ns, abort_flag);
                    ph_p ^= 1;
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int kb = kk >> 2, ks = kk & 3;
                        mma_bf16_ts(tmem + F::T_O + 32 * hd, tmem + F::T_S + 8 * kk,
                                    desc_kmajor_sw128(base + F::VT + kb * F::VT_BLK + (hd * 32 / 8) * 1024 + 32 * ks),
                                    id_pv, kk != 0);
                    }
                    mma_commit(B_PV);
                    // the next MMA that writes these TMEM columns (S of the next head,
                    // or the next tile's QKV) waits until P.V has read P
                    ok = wait_or_abort(B_PV, ph_pv_m, st.wait_ns, abort_flag);
                    ph_pv_m ^= 1;
                    if (!ok) break;
                }
                if (!ok) break;
                // next tile's QKV as soon as this tile's softmax has freed its TMEM
                // columns and the next x tile has landed
                if (tile + gridDim.x < ntiles) {
                    if (!wait_or_abort(R_FREE, ph_free, st.wait_ns, abort_flag)) break;
                    ph_free ^= 1;
                    tc_fence_after();
                    issue_qkv(buf ^ 1);
                }
                if (!wait_or_abort(R_O, ph_o, st.wait_ns, abort_flag)) break;
                ph_o ^= 1;
                tc_fence_after();
                const uint32_t xb = base + xbuf(buf);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_Y, desc_kmajor_sw64(xb + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(base + F::WP + kb * (C * 64) + 32 * ks), id_y, (kb | ks) != 0);
                mma_commit(B_Y);
            }
        }
    } else {
        // ===================== compute warps =====================
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        uint32_t ph_qkv = 0, ph_s = 0, ph_pv = 0, ph_y = 0;
        bool failed = false;
        int k = 0;
#pragma unroll 1
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
            const int buf = k & 1;
            const bool has_next = tile + gridDim.x < ntiles;
            PHASE(k, 0);
            int *tok_cur = rowtok + (k % 3) * 128, *tok_next = rowtok + ((k + 1) % 3) * 128;
            // this tile's window geometry: key regions and whether a window is cut
            // by the shift; the next tile's row tokens
            if (tid < 128) {
                const int sl = tid >> 6, tt = tid & 63;
                const int win = (int)(2 * tile) + sl;
                int reg = -1;
                if (tt < N && win < g.nwin) {
                    const int rem = win % (g.nh * g.nw);
                    const int wi = rem / g.nw, wj = rem % g.nw;
                    reg = 0;
                    if (g.s > 0)
                        reg = 3 * shift_band(wi * M + tt / M, g.H, M, g.s) + shift_band(wj * M + tt % M, g.W, M, g.s);
                    if (tt == 0) slot_masked[sl] = g.s > 0 && (wi == g.nh - 1 || wj == g.nw - 1);
                } else if (tt == 0) {
                    slot_masked[sl] = 0;
                }
                key_region[sl * 64 + tt] = reg;
            }
            row_tokens(tile + gridDim.x, tok_next);
            if (compute_sync_or(failed)) { failed = true; break; }
            PHASE(k, 1);
            // prefetch the next tile into the other buffer (its o and staging
            // were consumed by the previous tile, which has completed)
            if (has_next) load_x(tok_next, buf ^ 1);
            PHASE(k, 2);

            if (!wait_or_abort(B_QKV, ph_qkv, st.wait_ns, abort_flag)) failed = true;
            ph_qkv ^= 1;
            tc_fence_after();
            PHASE(k, 3);

            // v^T drain: lane = v channel, this half's 64 token columns -> V^T K block `half`
            {
                float v0[32], v1[32];
                tmem_ld32(t_lane + F::T_VT + 64 * half, v0);
                tmem_ld32(t_lane + F::T_VT + 64 * half + 32, v1);
                tmem_wait_ld();
                if (row < C) {
                    const float bv = sbqkv[2 * C + row];
                    uint8_t *dst = sm + F::VT + half * F::VT_BLK;
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(dst + sw128_offset(row, c)) =
                            make_uint4(pack_bf16x2(v0[8 * c] + bv, v0[8 * c + 1] + bv),
                                       pack_bf16x2(v0[8 * c + 2] + bv, v0[8 * c + 3] + bv),
                                       pack_bf16x2(v0[8 * c + 4] + bv, v0[8 * c + 5] + bv),
                                       pack_bf16x2(v0[8 * c + 6] + bv, v0[8 * c + 7] + bv));
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4 *>(dst + sw128_offset(row, 4 + c)) =
                            make_uint4(pack_bf16x2(v1[8 * c] + bv, v1[8 * c + 1] + bv),
                                       pack_bf16x2(v1[8 * c + 2] + bv, v1[8 * c + 3] + bv),
                                       pack_bf16x2(v1[8 * c + 4] + bv, v1[8 * c + 5] + bv),
                                       pack_bf16x2(v1[8 * c + 6] + bv, v1[8 * c + 7] + bv));
                }
            }
            // q_h (half 0) or k_h (half 1) of head hd to shared memory
            auto drain_qk = [&](int hd) {
                const int col = half == 0 ? hd * 32 : C + hd * 32;
                float v[32];
                tmem_ld32(t_lane + F::T_QK + col, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] += sbqkv[col + e];
                if (a.mode == 1) {
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
                    const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= inv;
                }
                uint8_t *dst = sm + (half == 0 ? F::Q : F::K);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(dst + sw64_offset(row, c)) =
                        make_uint4(pack_bf16x2(v[8 * c], v[8 * c + 1]), pack_bf16x2(v[8 * c + 2], v[8 * c + 3]),
                                   pack_bf16x2(v[8 * c + 4], v[8 * c + 5]), pack_bf16x2(v[8 * c + 6], v[8 * c + 7]));
                fence_proxy_async_smem();
                warp_arrive(R_QK, lane);
            };
            drain_qk(0);

            const bool row_ok = key_region[slot * 64 + t] >= 0;
            // keys this row may attend to (bit j = key j of its window): all N keys,
            // or those in its own shift region; none for a padding row
            uint32_t allow_lo = 0, allow_hi = 0;
            if (row_ok) {
                if (slot_masked[slot]) {
                    const int my_region = key_region[slot * 64 + t];
                    for (int j = 0; j < N; ++j) {
                        if (key_region[slot * 64 + j] == my_region) {
                            if (j < 32) allow_lo |= 1u << j;
                            else allow_hi |= 1u << (j - 32);
                        }
                    }
                } else {
                    allow_lo = 0xffffffffu;
                    allow_hi = N >= 64 ? 0xffffffffu : ((1u << (N - 32)) - 1u);
                }
            }
            const uint32_t allow = half == 0 ? allow_lo : allow_hi;
            const int tb = row_ok ? t : 0;   // padding rows read a valid bias row (then masked)
            const int bias_base = (tb / M + M - 1) * L + (tb % M + M - 1);

#pragma unroll 1
            for (int hd = 0; hd < HEADS; ++hd) {
                PHASE(k, 4 + 4 * hd);
                if (!wait_or_abort(B_S, ph_s, st.wait_ns, abort_flag)) failed = true;
                ph_s ^= 1;
                tc_fence_after();
                PHASE(k, 5 + 4 * hd);

                // ---- softmax over this row's own window, keys 32*half .. +31 -------
                float s[32];
                tmem_ld32(t_lane + F::T_S + 64 * slot + 32 * half, s);
                tmem_wait_ld();
                const float scale = sscale[hd];
                const float *bias = sbias + hd * L * L + bias_base;
                float mx = -INFINITY;
                // key j of the row's window: relative-bias row bias_base - ((j/M)*L + j%M);
                // j is a compile-time constant in each unrolled loop
                if (half == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float v = fmaf(s[j], scale, bias[-((j / M) * L + j % M)]);
                        s[j] = (allow >> j) & 1u ? v : -INFINITY;
                        mx = fmaxf(mx, s[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 32; j < 64; ++j) {
                        if (j < N) {
                            const float v = fmaf(s[j - 32], scale, bias[-((j / M) * L + j % M)]);
                            s[j - 32] = (allow >> (j - 32)) & 1u ? v : -INFINITY;
                        } else {
                            s[j - 32] = -INFINITY;
                        }
                        mx = fmaxf(mx, s[j - 32]);
                    }
                }
                smax[half * 128 + row] = mx;
                if (hd == HEADS - 1 && has_next) {
                    // this tile's last TMEM reads of the QK and S columns are done, and
                    // the next x tile is in place: the MMA warp may start its QKV
                    cp_async_wait<0>();
                    fence_proxy_async_smem();
                    warp_arrive(R_FREE, lane);
                }
                if (compute_sync_or(failed)) { failed = true; break; }
                mx = row_ok ? fmaxf(smax[row], smax[128 + row]) : 0.f;   // padding rows: all -inf -> p = 0
                float sum = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const float p0 = ex2_approx(s[jj] - mx), p1 = ex2_approx(s[jj + 1] - mx);
                    sum += p0 + p1;
                    pk[jj / 2] = pack_bf16x2(p0, p1);
                }
                spart[(hd * 2 + half) * 128 + row] = sum;
                PHASE(k, 6 + 4 * hd);
                // P may be rewritten only once the previous head's P.V has read it
                if (hd > 0) {
                    if (!wait_or_abort(B_PV, ph_pv, st.wait_ns, abort_flag)) failed = true;
                    ph_pv ^= 1;
                }
                // P (bf16, two keys per 32-bit column) goes to TMEM over the first 64
                // columns of S, the A operand of the P.V MMA: row r holds its window's
                // keys in columns 32*slot .. +31 and zeros for the other window's
                {
                    tmem_st16(t_lane + F::T_S + 32 * slot + 16 * half, pk);
                    const uint32_t zero[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    tmem_st16(t_lane + F::T_S + 32 * (slot ^ 1) + 16 * half, zero);
                    tmem_wait_st();
                }
                warp_arrive(R_P, lane);
                PHASE(k, 7 + 4 * hd);
                if (hd + 1 < HEADS) drain_qk(hd + 1);
            }
            // (a failure here is not uniform across threads yet: carry on to the
            // next barrier-with-OR, which makes every compute thread leave together;
            // waits return at once once the abort flag is set)
            if (!wait_or_abort(B_PV, ph_pv, st.wait_ns, abort_flag)) failed = true;
            ph_pv ^= 1;
            tc_fence_after();
            PHASE(k, 17);

            // ---- o / rowsum -> bf16 -> X buffer (A operand of the projection) ------
#pragma unroll
            for (int hd = 0; hd < HEADS; ++hd) {
                float o[16];
                tmem_ld16(t_lane + F::T_O + 32 * hd + 16 * half, o);
                tmem_wait_ld();
                const float l = spart[(hd * 2) * 128 + row] + spart[(hd * 2 + 1) * 128 + row];
                const float inv = row_ok ? rcp_approx(l) : 0.f;
                uint8_t *dst = sm + xbuf(buf) + hd * (128 * 64);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    *reinterpret_cast<uint4 *>(dst + sw64_offset(row, 2 * half + c)) =
                        make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                   pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                   pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                   pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
            }
            fence_proxy_async_smem();
            warp_arrive(R_O, lane);
            PHASE(k, 18);
            if (!wait_or_abort(B_Y, ph_y, st.wait_ns, abort_flag)) failed = true;
            ph_y ^= 1;
            tc_fence_after();
            PHASE(k, 19);

            // ---- y + bproj -> bf16 staging rows -> out through window reverse + roll(+s) ----
            // (thread = row reads its half of y from TMEM into a staging row with a
            // padded, bank-conflict-free stride; then all compute threads copy the
            // rows out in 16-byte chunks, consecutive lanes on consecutive chunks,
            // so each warp store covers whole rows that are contiguous in out
            // within a window row)
            {
                constexpr int HC = C / 2;
                uint8_t *stage = sm + xbuf(buf);
                uint8_t *srow = stage + row * F::SROW + half * HC * 2;
#pragma unroll
                for (int c0 = 0; c0 < HC; c0 += 16) {
                    float y[16];
                    tmem_ld16(t_lane + F::T_Y + half * HC + c0, y);
                    tmem_wait_ld();
                    const float *bp = sbproj + half * HC + c0;
                    uint4 *d4 = reinterpret_cast<uint4 *>(srow + c0 * 2);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        d4[c] = make_uint4(pack_bf16x2(y[8 * c] + bp[8 * c], y[8 * c + 1] + bp[8 * c + 1]),
                                           pack_bf16x2(y[8 * c + 2] + bp[8 * c + 2], y[8 * c + 3] + bp[8 * c + 3]),
                                           pack_bf16x2(y[8 * c + 4] + bp[8 * c + 4], y[8 * c + 5] + bp[8 * c + 5]),
                                           pack_bf16x2(y[8 * c + 6] + bp[8 * c + 6], y[8 * c + 7] + bp[8 * c + 7]));
                }
                tc_fence_before();
                if (compute_sync_or(failed)) { failed = true; break; }
                constexpr int CH = C / 8;   // 16-byte chunks per row
#pragma unroll 1
                for (int q = tid; q < 128 * CH; q += NCOMPUTE) {
                    const int r = q / CH, c16 = q % CH;
                    const int tk = tok_cur[r];
                    if (tk >= 0)
                        *reinterpret_cast<uint4 *>(a.out + (int64_t)tk * C + c16 * 8) =
                            *reinterpret_cast<const uint4 *>(stage + r * F::SROW + c16 * 16);
                }
            }
            PHASE(k, 20);
        }
        cp_async_wait<0>();
        if (failed) *abort_flag = 1;
    }
#ifdef SWIN_PHASE_TRACE
    if (tid == 0) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_cta_trace[blockIdx.x * 4 + 1] = (long long)global_timer_ns();
        g_cta_trace[blockIdx.x * 4 + 3] = smid;
    }
#endif
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(st.err, ERR_TIMEOUT);
    if (is_mma) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

int num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    }
    return n;
}

template <int M, int C>
cudaError_t launch_fused_t(const FusedArgs &a, DeviceStatus st, cudaStream_t stream)
{
    using F = FusedCfg<M, C>;
    const size_t smem = F::BYTES + 1024;
    auto kern = fused_block_kernel<M, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.g.nwin + 1) / 2;
    const int grid = (int)(ntiles < num_sms() ? ntiles : num_sms());
    kern<<<grid, FTHREADS, smem, stream>>>(a, st);
    return cudaGetLastError();
}

} // namespace

#ifdef SWIN_PHASE_TRACE
extern "C" int swin_wattn_phase_trace(long long *host, int n)
{
    return (int)cudaMemcpyFromSymbol(host, g_phase_trace, sizeof(long long) * (size_t)n);
}
extern "C" int swin_wattn_cta_trace(long long *host, int n)
{
    return (int)cudaMemcpyFromSymbol(host, g_cta_trace, sizeof(long long) * (size_t)n);
}
#endif

bool fused_supported(int M, int C, int heads)
{
    return (M == 7 || M == 8) && (C == 64 || C == 96) && C == heads * 32;
}

cudaError_t launch_fused(const bf16 *x, const bf16 *Wqkv, const bf16 *bqkv, const bf16 *table, const float *tau,
                         const bf16 *Wproj, const bf16 *bproj, bf16 *out, int mode, const Geom &g, DeviceStatus st,
                         cudaStream_t stream)
{
    FusedArgs a{x, Wqkv, bqkv, table, Wproj, bproj, tau, out, mode, g};
    if (g.M == 7 && g.C == 96) return launch_fused_t<7, 96>(a, st, stream);
    if (g.M == 8 && g.C == 96) return launch_fused_t<8, 96>(a, st, stream);
    if (g.M == 7 && g.C == 64) return launch_fused_t<7, 64>(a, st, stream);
    if (g.M == 8 && g.C == 64) return launch_fused_t<8, 64>(a, st, stream);
    return cudaErrorInvalidValue;
}

} // namespace swin
