// The Swin block's MLP sub-layer as one persistent kernel (sm_103a, tcgen05 +
// TMEM) ("Swin Transformer V2" (neura.market), How It Works: pre-norm in the
// original Swin, residual post-norm in V2), on the block's residual stream z:
//   V1 (PRE)    y = z + GELU(LN(z) W1^T + b1) W2^T + b2
//   V2 (POST)   y = z + LN(GELU(z W1^T + b1) W2^T + b2)
// with the exact GELU of gelu.cuh and LayerNorm's own gain and shift.  The
// hidden activation (4C per token) never leaves the SM.  Per 128-row tile of
// tokens (z's rows by 2-D TMA into one of two buffers, read again for the
// residual) the hidden units go in chunks of 128: H = z W1[chunk]^T (128 x 128
// x C) into one of two TMEM buffers; sixteen compute warps (four per TMEM lane
// quarter, 32 columns each) add the bias, apply GELU and write H back as bf16
// over the first half of their own fp32 columns; Y += H W2[:, chunk]^T (128 x
// C x 128, H read from TMEM as the A operand) into one of two Y buffers (tiles
// alternate).  GEMM1 of chunk n is issued before GEMM2 of chunk n - 1, so the
// tensor cores work while the compute warps apply GELU.
// PRE folds LN into GEMM1: LN(z) W1^T + b1 = rstd (z W'^T - mean c) + b' with
// W' = W1 diag(gamma) (bf16, in shared memory), c its row sums and b' = W1 beta
// + b1; each row's mean and rstd are summed over the quarter's four warps (24
// or 16 channels each) through shared memory.  POST takes the LayerNorm of the
// row's C outputs the same way (mean, then mean square deviation).
// Warp roles: 0 loads z tiles, 1 issues every MMA and owns TMEM, 2 and 3 idle,
// 4..19 compute (four warps per scheduler: the work per element is short
// chains, so latency is hidden by warps).  Weights stay in shared memory (one
// CTA per SM, tiles round-robin).  Every wait is bounded.
#include "common.cuh"
#include "gelu.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int MT_THREADS = 20 * 32;
constexpr int MT_CWARPS = 16;
constexpr int MT_CWARP0 = 4;
constexpr float MT_EPS = 1e-5f;
enum { MLP_PRE = 1, MLP_POST = 2 };

template <int C, int R>
struct MlpCfg {
    static constexpr int KB = C / 32;    // 32-wide K blocks of z and W1 (64-byte swizzle)
    static constexpr int NC = R / 128;   // hidden chunks of 128
    static constexpr int CP = C / 4;     // a compute warp's columns of the row: 24 or 16
    static constexpr int HT = 128 * 64;  // one [128 rows][32] SW64 tile
    static constexpr int W1 = 0;                   // [R rows][C]: KB blocks of R * 64 bytes
    static constexpr int W2 = W1 + R * C * 2;      // [C rows][R]: R / 32 blocks of C * 64 bytes
    static constexpr int AT = W2 + C * R * 2;      // z tile buffer a at AT + a * KB * HT
    static constexpr int SMALL = AT + 2 * KB * HT;
    static constexpr int O_B1 = 0;                 // [R] f32 (PRE: b')
    static constexpr int O_C1 = O_B1 + R * 4;      // [R] f32 (PRE: row sums of W')
    static constexpr int O_B2 = O_C1 + R * 4;      // [C] f32
    static constexpr int O_LN = O_B2 + C * 4;      // [2][C] f32: gamma, beta
    static constexpr int O_XCH = O_LN + 2 * C * 4; // [2 sets][16 warps][32 lanes] float2: quarter sums
    static constexpr int O_BARS = O_XCH + 2 * MT_CWARPS * 32 * 8;
    static constexpr int NBARS = 18;
    static constexpr int O_END = O_BARS + NBARS * 8 + 16;
    static constexpr int BYTES = SMALL + O_END;
    // TMEM: H buffers at 128 b, Y buffers at 256 + C yb
    static constexpr int T_H = 0, T_Y = 256;
    static_assert(C % 32 == 0 && C <= 128 && R % 128 == 0 && CP % 8 == 0, "shapes");
    static_assert(T_Y + 2 * C <= 512, "TMEM budget");
    static_assert(BYTES + 1024 <= 232448, "shared memory budget");
};

enum {
    MB_AFULL = 0,    // + a: z tile landed (TMA bytes)
    MB_AFREE = 2,    // + a: the tile's last GEMM1 and every compute warp's epilogue have read it
    MB_HREADY = 4,   // + b: GEMM1 into H buffer b done
    MB_HBF = 6,      // + b: H buffer b holds GELU(H) as bf16 (compute warps)
    MB_HFREE = 8,    // + b: GEMM2 has read H buffer b
    MB_YREADY = 10,  // + yb: the tile's last GEMM2 done
    MB_YFREE = 12,   // + yb: Y buffer yb drained (compute warps)
    MB_XCH = 14      // + quarter: the quarter's four partial sums are in shared memory
};

struct MlpArgs {
    const bf16 *W1, *b1, *W2, *b2, *ln_g, *ln_b;
    bf16 *out;
    int64_t T;
};

__device__ __forceinline__ bool mt_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
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

__device__ __forceinline__ bool mt_warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
{
    const bool ok = mt_wait(bar, parity, limit_ns, abort);
    return __all_sync(0xffffffffu, ok);
}

// A shared-memory descriptor whose start address (16-byte units) is moved by `bytes`.
__device__ __forceinline__ uint64_t mt_desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ void mt_warp_arrive(uint32_t bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

template <int C, int R, int MODE>
__global__ void __launch_bounds__(MT_THREADS, 1)
    mlp_fused_kernel(MlpArgs a, DeviceStatus st, const __grid_constant__ CUtensorMap tmap_z)
// tmap_z: z as [T][C] bf16, boxes of 32 columns x 128 rows
{
    using F = MlpCfg<C, R>;
    constexpr int KB = F::KB, NC = F::NC, HT = F::HT, CP = F::CP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    uint8_t *small = sm + F::SMALL;
    float *sb1 = reinterpret_cast<float *>(small + F::O_B1);
    float *sc1 = reinterpret_cast<float *>(small + F::O_C1);
    float *sb2 = reinterpret_cast<float *>(small + F::O_B2);
    float *sln = reinterpret_cast<float *>(small + F::O_LN);
    float2 *sxch = reinterpret_cast<float2 *>(small + F::O_XCH);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + F::O_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + F::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);
    auto BAR = [&](int i) { return smem_u32(&bars[i]); };
    const int64_t ntiles = (a.T + 127) / 128;
    auto wrow = [&](int n, int c16) -> uint8_t * {   // W1 row n, 16-byte chunk c16
        return sm + F::W1 + (c16 >> 2) * (R * 64) + sw64_offset(n, c16 & 3);
    };

    // ---- once per CTA: weights (64-byte-swizzled K-major), bias vectors,
    // barriers, TMEM --------------------------------------------------------
    for (int q = tid; q < R * (C / 8); q += MT_THREADS) {   // W1 [R][C]
        const int r = q / (C / 8), c16 = q % (C / 8);
        cp_async16(smem_u32(wrow(r, c16)), a.W1 + (int64_t)r * C + c16 * 8, 16);
    }
    for (int q = tid; q < C * (R / 8); q += MT_THREADS) {   // W2 [C][R]
        const int r = q / (R / 8), c16 = q % (R / 8);
        cp_async16(base + F::W2 + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3), a.W2 + (int64_t)r * R + c16 * 8,
                   16);
    }
    cp_async_commit();
    for (int i = tid; i < R; i += MT_THREADS) sb1[i] = a.b1 ? __bfloat162float(a.b1[i]) : 0.f;
    for (int i = tid; i < C; i += MT_THREADS) {
        sb2[i] = a.b2 ? __bfloat162float(a.b2[i]) : 0.f;
        sln[i] = __bfloat162float(a.ln_g[i]);
        sln[C + i] = __bfloat162float(a.ln_b[i]);
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(MB_AFULL + i), 1);
            mbar_init(BAR(MB_AFREE + i), 1 + MT_CWARPS);
            mbar_init(BAR(MB_HREADY + i), 1);
            mbar_init(BAR(MB_HBF + i), MT_CWARPS);
            mbar_init(BAR(MB_HFREE + i), 1);
            mbar_init(BAR(MB_YREADY + i), 1);
            mbar_init(BAR(MB_YFREE + i), MT_CWARPS);
        }
        for (int q = 0; q < 4; ++q) mbar_init(BAR(MB_XCH + q), 4);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    cp_async_wait<0>();
    __syncthreads();   // weights, bias vectors
    if (MODE == MLP_PRE) {
        // b' = W1 beta + b1 (fp32, the unscaled weights, one thread per hidden
        // unit in a fixed order), then W' = W1 diag(gamma) in place (bf16),
        // then c = the row sums of W' as the MMAs see it
        for (int n = tid; n < R; n += MT_THREADS) {
            float acc = 0.f;
#pragma unroll 1
            for (int c16 = 0; c16 < C / 8; ++c16) {
                const uint4 w8 = *reinterpret_cast<const uint4 *>(wrow(n, c16));
                const uint32_t wd[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 w2 = unpack_bf16x2(wd[e]);
                    acc = fmaf(w2.x, sln[C + 8 * c16 + 2 * e], acc);
                    acc = fmaf(w2.y, sln[C + 8 * c16 + 2 * e + 1], acc);
                }
            }
            sb1[n] += acc;
        }
        __syncthreads();
#pragma unroll 1
        for (int q = tid; q < R * (C / 8); q += MT_THREADS) {
            const int n = q / (C / 8), c16 = q % (C / 8);
            uint4 *p = reinterpret_cast<uint4 *>(wrow(n, c16));
            const uint4 w8 = *p;
            const uint32_t wd[4] = {w8.x, w8.y, w8.z, w8.w};
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 w2 = unpack_bf16x2(wd[e]);
                o[e] = pack_bf16x2(w2.x * sln[8 * c16 + 2 * e], w2.y * sln[8 * c16 + 2 * e + 1]);
            }
            *p = make_uint4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
        for (int n = tid; n < R; n += MT_THREADS) {
            float acc = 0.f;
#pragma unroll 1
            for (int c16 = 0; c16 < C / 8; ++c16) {
                const uint4 w8 = *reinterpret_cast<const uint4 *>(wrow(n, c16));
                const uint32_t wd[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 w2 = unpack_bf16x2(wd[e]);
                    acc += w2.x;
                    acc += w2.y;
                }
            }
            sc1[n] = acc;
        }
    }
    fence_proxy_async_smem();   // the weights are read by the MMAs
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto A = [&](int buf) { return base + F::AT + buf * KB * HT; };

    // The prologue above reads only the parameters; z and out wait for the
    // kernels queued before this one (a no-op unless launched to overlap them),
    // and the next such kernel may start its own prologue.
    griddep_launch_dependents();
    griddep_wait();
    if (warp == 0) {
        // ===================== producer: z tiles =====================
        bool ok = true;
        if (lane == 0) {
#pragma unroll 1
            for (int j = 0;; ++j) {
                const int64_t tile = (int64_t)blockIdx.x + (int64_t)j * gridDim.x;
                if (tile >= ntiles) break;
                const int ab = j & 1;
                if (j >= 2 && !(ok = mt_wait(BAR(MB_AFREE + ab), ((j >> 1) - 1) & 1, st.wait_ns, abort_flag))) break;
                mbar_arrive_expect_tx(BAR(MB_AFULL + ab), KB * HT);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
                    tma_load_2d(A(ab) + kb * HT, &tmap_z, kb * 32, (int)(tile * 128), BAR(MB_AFULL + ab));
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (warp == 1) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            constexpr uint32_t id1 = idesc_bf16(128, 128), id2 = idesc_bf16(128, C);
            const uint64_t dw1 = desc_kmajor_sw64(base + F::W1), dw2 = desc_kmajor_sw64(base + F::W2);
            bool ok = true;
            // GEMM2 of global chunk m: Y[yb] (+)= GELU(H[b]) W2[:, chunk]^T
            auto gemm2 = [&](int m) -> bool {
                const int b = m & 1, cm = m % NC, jm = m / NC, yb = jm & 1;
                if (!mt_wait(BAR(MB_HBF + b), (m >> 1) & 1, st.wait_ns, abort_flag)) return false;
                if (cm == 0 && jm >= 2 && !mt_wait(BAR(MB_YFREE + yb), ((jm >> 1) - 1) & 1, st.wait_ns, abort_flag))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    // K step s (16 hidden units): bf16 pairs at column 32 (s / 2) + 8 (s % 2) of the buffer
                    const uint32_t at = tmem + F::T_H + 128 * b + 32 * (s >> 1) + 8 * (s & 1);
                    const uint64_t bd = mt_desc_add(dw2, (4 * cm + (s >> 1)) * (C * 64) + 32 * (s & 1));
                    mma_bf16_ts(tmem + F::T_Y + C * yb, at, bd, id2, (cm | s) != 0);
                }
                mma_commit(BAR(MB_HFREE + b));
                if (cm == NC - 1) mma_commit(BAR(MB_YREADY + yb));
                return true;
            };
            int n = 0;   // global chunk index
#pragma unroll 1
            for (int j = 0; ok; ++j) {
                const int64_t tile = (int64_t)blockIdx.x + (int64_t)j * gridDim.x;
                if (tile >= ntiles) break;
                const int ab = j & 1;
                if (!(ok = mt_wait(BAR(MB_AFULL + ab), (j >> 1) & 1, st.wait_ns, abort_flag))) break;
                const uint64_t da = desc_kmajor_sw64(A(ab));
#pragma unroll 1
                for (int c = 0; c < NC; ++c, ++n) {
                    const int b = n & 1;
                    if (n >= 2 && !(ok = mt_wait(BAR(MB_HFREE + b), ((n >> 1) - 1) & 1, st.wait_ns, abort_flag)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                        for (int ks = 0; ks < 2; ++ks)
                            mma_bf16(tmem + F::T_H + 128 * b, mt_desc_add(da, kb * HT + 32 * ks),
                                     mt_desc_add(dw1, kb * (R * 64) + c * (128 * 64) + 32 * ks), id1, (kb | ks) != 0);
                    mma_commit(BAR(MB_HREADY + b));
                    if (c == NC - 1) mma_commit(BAR(MB_AFREE + ab));
                    if (n >= 1 && !(ok = gemm2(n - 1))) break;
                }
            }
            if (ok && n >= 1) ok = gemm2(n - 1);
            if (!ok) *abort_flag = 1;
        }
    } else if (warp >= MT_CWARP0) {
        // ===================== compute warps =====================
        const int quarter = warp & 3, part = (warp - MT_CWARP0) >> 2;   // part: 0..3 within the quarter
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        int n = 0, xe = 0;   // chunk counter, exchange counter
        // the sum over the quarter's four warps of each lane's v, through
        // shared memory (slot set xe mod 2; a set is written again two
        // exchanges later, after every warp of the quarter has read it)
        auto qsum = [&](float2 v) -> float2 {
            float2 *set = sxch + (xe & 1) * (MT_CWARPS * 32);
            set[(quarter * 4 + part) * 32 + lane] = v;
            mt_warp_arrive(BAR(MB_XCH + quarter), lane);
            if (!(ok = mt_warp_wait(BAR(MB_XCH + quarter), xe & 1, st.wait_ns, abort_flag))) return make_float2(0.f, 1.f);
            ++xe;
            float2 s = make_float2(0.f, 0.f);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float2 w = set[(quarter * 4 + p) * 32 + lane];
                s.x += w.x;
                s.y += w.y;
            }
            return s;
        };
        auto tile_of = [&](int j) { return (int64_t)blockIdx.x + (int64_t)j * gridDim.x; };
        auto zchunk_of = [&](int ab, int col) {   // 8 channels from col (a multiple of 8) of z tile buffer ab
            return *reinterpret_cast<const uint4 *>(sm + F::AT + ab * KB * HT + (col >> 5) * HT +
                                                    sw64_offset(row, (col & 31) >> 3));
        };
        // ---- the start of tile j: its z tile landed; PRE: the row's LayerNorm
        // statistics (rstd and -rstd mean), shifted sums (shift: the row's first
        // channel) over this warp's channels, then over the quarter ----
        auto begin_tile = [&](int j, float &rstd, float &nms) -> bool {
            const int ab = j & 1;
            if (!(ok = mt_warp_wait(BAR(MB_AFULL + ab), (j >> 1) & 1, st.wait_ns, abort_flag))) return false;
            rstd = 1.f;
            nms = 0.f;
            if (MODE == MLP_PRE) {
                const float K = unpack_bf16x2(zchunk_of(ab, 0).x).x;
                float s1 = 0.f, s2 = 0.f;
#pragma unroll
                for (int q = 0; q < CP / 8; ++q) {
                    const uint4 u = zchunk_of(ab, CP * part + 8 * q);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(wd[e]);
                        const float d0 = f.x - K, d1 = f.y - K;
                        s1 += d0 + d1;
                        s2 = fmaf(d0, d0, fmaf(d1, d1, s2));
                    }
                }
                const float2 s = qsum(make_float2(s1, s2));
                if (!ok) return false;
                const float m1 = s.x / (float)C;   // mean - K
                rstd = rsqrtf(fmaxf(s.y / (float)C - m1 * m1, 0.f) + MT_EPS);
                nms = -rstd * (K + m1);
            }
            return true;
        };
        // ---- GELU of chunk c (the CTA's n-th) of a tile: this warp's 32 columns ----
        auto gelu_chunk = [&](int c, float rstd, float nms) -> bool {
            const int b = n & 1;
            if (!(ok = mt_warp_wait(BAR(MB_HREADY + b), (n >> 1) & 1, st.wait_ns, abort_flag))) return false;
            tc_fence_after();
            const uint32_t tcol = t_lane + F::T_H + 128 * b + 32 * part;
            float v[32];
            tmem_ld32(tcol, v);
            tmem_wait_ld();
            const float4 *b4 = reinterpret_cast<const float4 *>(sb1 + 128 * c + 32 * part);
            const float4 *c4 = reinterpret_cast<const float4 *>(sc1 + 128 * c + 32 * part);
            uint32_t pk[16];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
                const float4 bb = b4[e4];
                float x0, x1, x2, x3;
                if (MODE == MLP_PRE) {
                    // rstd acc + (c (-rstd mean) + b')
                    const float4 cc = c4[e4];
                    float t0, t1, t2, t3;
                    g2_fma(t0, t1, cc.x, cc.y, nms, nms, bb.x, bb.y);
                    g2_fma(t2, t3, cc.z, cc.w, nms, nms, bb.z, bb.w);
                    g2_fma(x0, x1, v[4 * e4], v[4 * e4 + 1], rstd, rstd, t0, t1);
                    g2_fma(x2, x3, v[4 * e4 + 2], v[4 * e4 + 3], rstd, rstd, t2, t3);
                } else {
                    x0 = v[4 * e4] + bb.x;
                    x1 = v[4 * e4 + 1] + bb.y;
                    x2 = v[4 * e4 + 2] + bb.z;
                    x3 = v[4 * e4 + 3] + bb.w;
                }
                gelu_exact2(x0, x1);
                gelu_exact2(x2, x3);
                pk[2 * e4] = pack_bf16x2(x0, x1);
                pk[2 * e4 + 1] = pack_bf16x2(x2, x3);
            }
            tmem_st16(tcol, pk);
            tmem_wait_st();
            mt_warp_arrive(BAR(MB_HBF + b), lane);   // read by GEMM2
            ++n;
            return true;
        };
        // ---- the end of tile j ----
        auto end_tile = [&](int j) -> bool {
            const int64_t tok = tile_of(j) * 128 + row;
            const bool valid = tok < a.T;
            const int ab = j & 1;
            auto zchunk = [&](int col) { return zchunk_of(ab, col); };
            // ---- this warp's CP columns: y = z + Y + b2 (POST: z + LN(Y + b2)) ----
            const int yb = j & 1;
            if (!(ok = mt_warp_wait(BAR(MB_YREADY + yb), (j >> 1) & 1, st.wait_ns, abort_flag))) return false;
            tc_fence_after();
            float y[24];
            const uint32_t ycol = t_lane + F::T_Y + C * yb + CP * part;
            tmem_ld16(ycol, *reinterpret_cast<float(*)[16]>(y));
            if (CP == 24) tmem_ld8(ycol + 16, *reinterpret_cast<float(*)[8]>(y + 16));
            tmem_wait_ld();
            mt_warp_arrive(BAR(MB_YFREE + yb), lane);
#pragma unroll
            for (int k = 0; k < CP; ++k) y[k] += sb2[CP * part + k];
            float scale = 1.f, shift = 0.f;   // POST: y -> y scale + shift, then gamma, beta
            if (MODE == MLP_POST) {
                float s1 = 0.f;
#pragma unroll
                for (int k = 0; k < CP; ++k) s1 += y[k];
                const float mean = qsum(make_float2(s1, 0.f)).x / (float)C;
                if (!ok) return false;
                float s2 = 0.f;
#pragma unroll
                for (int k = 0; k < CP; ++k) {
                    const float d = y[k] - mean;
                    s2 = fmaf(d, d, s2);
                }
                const float var = qsum(make_float2(s2, 0.f)).x / (float)C;
                if (!ok) return false;
                scale = rsqrtf(var + MT_EPS);
                shift = -mean * scale;
            }
            if (valid) {
                uint4 *dst = reinterpret_cast<uint4 *>(a.out + tok * C + CP * part);
#pragma unroll
                for (int q = 0; q < CP / 8; ++q) {
                    const uint4 u = zchunk(CP * part + 8 * q);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
                    uint32_t o[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 r2 = unpack_bf16x2(wd[e]);
                        const int k = 8 * q + 2 * e, kk = CP * part + k;
                        float v0 = y[k], v1 = y[k + 1];
                        if (MODE == MLP_POST) {
                            v0 = fmaf(fmaf(v0, scale, shift), sln[kk], sln[C + kk]);
                            v1 = fmaf(fmaf(v1, scale, shift), sln[kk + 1], sln[C + kk + 1]);
                        }
                        o[e] = pack_bf16x2(v0 + r2.x, v1 + r2.y);
                    }
                    dst[q] = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
            mt_warp_arrive(BAR(MB_AFREE + ab), lane);   // (this warp's reads of the z tile are done)
            return true;
        };
        // Software-pipelined over the CTA's tiles: after tile j's last chunk the
        // warps start tile j + 1 (its statistics and first chunk) and only then
        // take tile j's output, so that the wait for tile j's last GEMM2 runs
        // under that work.  (Chunks stay in order n = 0, 1, ...: GEMM1 of tile j
        // + 1's first chunk is issued before GEMM2 of tile j's last one.)
        float r_cur = 1.f, m_cur = 0.f;
        if (tile_of(0) < ntiles) ok = begin_tile(0, r_cur, m_cur) && gelu_chunk(0, r_cur, m_cur);
#pragma unroll 1
        for (int j = 0; ok && tile_of(j) < ntiles; ++j) {
#pragma unroll 1
            for (int c = 1; c < NC && ok; ++c) ok = gelu_chunk(c, r_cur, m_cur);
            if (!ok) break;
            float r_nxt = 1.f, m_nxt = 0.f;
            if (tile_of(j + 1) < ntiles && !(ok = begin_tile(j + 1, r_nxt, m_nxt) && gelu_chunk(0, r_nxt, m_nxt))) break;
            if (!(ok = end_tile(j))) break;
            r_cur = r_nxt;
            m_cur = m_nxt;
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(st.err, ERR_TIMEOUT);
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

int mlp_num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    }
    return n;
}

template <int C, int R, int MODE>
cudaError_t launch_mlp_t(const bf16 *z, const MlpArgs &a, DeviceStatus st, cudaStream_t stream, int overlap)
{
    using F = MlpCfg<C, R>;
    const size_t smem = F::BYTES + 1024;
    auto kern = mlp_fused_kernel<C, R, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tz;
    e = make_tensor_map_sw64(&tz, z, a.T, C, 128);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.T + 127) / 128;
    const int grid = (int)(ntiles < mlp_num_sms() ? ntiles : mlp_num_sms());
    // (overlap: programmatic stream serialization, see the prologue's end)
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(MT_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, st, tz);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace

bool mlp_fused_supported(int C, int R) { return (C == 96 && R == 384) || (C == 64 && R == 256); }

cudaError_t launch_mlp_fused(const bf16 *z, const bf16 *W1, const bf16 *b1, const bf16 *W2, const bf16 *b2,
                             const bf16 *ln_g, const bf16 *ln_b, bool post, bf16 *out, int64_t T, int C, int R,
                             DeviceStatus st, cudaStream_t stream, int overlap)
{
    if (!mlp_fused_supported(C, R) || !z || !W1 || !W2 || !ln_g || !ln_b || !out || T <= 0)
        return cudaErrorInvalidValue;
    const MlpArgs a{W1, b1, W2, b2, ln_g, ln_b, out, T};
    if (C == 96)
        return post ? launch_mlp_t<96, 384, MLP_POST>(z, a, st, stream, overlap)
                    : launch_mlp_t<96, 384, MLP_PRE>(z, a, st, stream, overlap);
    return post ? launch_mlp_t<64, 256, MLP_POST>(z, a, st, stream, overlap)
                : launch_mlp_t<64, 256, MLP_PRE>(z, a, st, stream, overlap);
}

} // namespace swin
