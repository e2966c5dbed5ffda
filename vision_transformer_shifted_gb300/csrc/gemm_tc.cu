// Tensor-core GEMM of the block's two projections, tcgen05 + TMEM on sm_103a.
//
//   D[r, n] = sum_k A[r, k] * Bw[n, k] + bias[n]      (bf16 in, fp32 accumulate)
//
// QKV projection ("Boosting Swin Transformer Speed", Inference Optimization:
// QKV GEMM fused with its bias, no separate transpose): the A rows are read
// straight from x through the cyclic-shift + window-partition map (Training
// Optimization: the partition/shift index maps), so no partitioned copy of x
// is ever written.  Output projection: the epilogue writes each row through
// the window-reverse + roll(+s) map into the original [B, H, W, C] layout.
//
// Tile: 128 rows x BN columns (BN <= 256, multiple of 16), K in blocks of BK
// (64: one 128-byte swizzle atom per row, 3-stage ring; 32: one 64-byte
// swizzle atom per row, 4-stage ring), cp.async into the K-major swizzled
// layout, one thread issuing tcgen05.mma, the fp32 accumulator in TMEM, and a
// 4-warp epilogue reading one TMEM lane (= one output row) per thread.
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"
#include "gelu.cuh"

namespace swin {

namespace {

constexpr int BM = 128;
constexpr int THREADS = 128;

template <int BK, int NSTAGES = (BK == 64 ? 3 : 4)>
struct GemmSmem {
    // dynamic layout: [A stages][B stages] (1024-aligned), then row offsets,
    // bias, barriers and the TMEM address.
    static constexpr int STAGES = NSTAGES;
    static constexpr int CPR = BK / 8;          // 16-byte chunks per row
    static constexpr int a_stage = BM * BK * 2;
    static size_t bytes(int BN)
    {
        return 1024 + (size_t)STAGES * (a_stage + BN * BK * 2) + BM * sizeof(int64_t) + 256 * sizeof(float) +
               STAGES * 8 + 8 + 16;
    }
    static __device__ __forceinline__ uint32_t offset(uint32_t row, uint32_t chunk)
    {
        return BK == 64 ? sw128_offset(row, chunk) : sw64_offset(row, chunk);
    }
    static __device__ __forceinline__ uint64_t desc(uint32_t addr)
    {
        return BK == 64 ? desc_kmajor_sw128(addr) : desc_kmajor_sw64(addr);
    }
};

__device__ __forceinline__ void store_row_bf16(bf16 *dst, const float *v, const float *bias, int n)
{
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    for (int q = 0; q < n / 8; ++q) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * q + 0] + bias[8 * q + 0], v[8 * q + 1] + bias[8 * q + 1]);
        u.y = pack_bf16x2(v[8 * q + 2] + bias[8 * q + 2], v[8 * q + 3] + bias[8 * q + 3]);
        u.z = pack_bf16x2(v[8 * q + 4] + bias[8 * q + 4], v[8 * q + 5] + bias[8 * q + 5]);
        u.w = pack_bf16x2(v[8 * q + 6] + bias[8 * q + 6], v[8 * q + 7] + bias[8 * q + 7]);
        d4[q] = u;
    }
}

// Epilogue of the block's MLP ("Swin Transformer V2" (neura.market), How It
// Works: the block's sub-layers): e = v + bias, then GELU(e) = e * Phi(e)
// (exact GELU, erf as above) or e + R[row, n] (the residual branch).
__device__ __forceinline__ void epilogue_op(const GemmArgs &a, int64_t R, int n, const float *v, const float *bias,
                                            float *e, int cnt)
{
    for (int i = 0; i < cnt; ++i) {
        float t = v[i] + bias[i];
        if (a.epi == EPI_GELU) t = gelu_exact(t);
        else if (a.epi == EPI_RESID && R < a.rows) t += __bfloat162float(a.R[R * a.ldr + n + i]);
        e[i] = t;
    }
}

template <int LOAD, int STORE, int BK, int NSTAGES>
__global__ void __launch_bounds__(THREADS) gemm_tc_kernel(GemmArgs a, int BN, DeviceStatus st)
{
    using L = GemmSmem<BK, NSTAGES>;
    constexpr int STAGES = L::STAGES, CPR = L::CPR;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align(smem_raw, 1024);
    const int b_stage = BN * BK * 2;
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * L::a_stage;
    int64_t *row_off = reinterpret_cast<int64_t *>(sB + STAGES * b_stage);
    float *sbias = reinterpret_cast<float *>(row_off + BM);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sbias + 256);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + STAGES + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int n0 = blockIdx.y * BN;
    const int KB = (a.K + BK - 1) / BK;
    const uint32_t tmem_cols = BN <= 32 ? 32 : BN <= 64 ? 64 : BN <= 128 ? 128 : 256;

    // source offset (elements) of each tile row; -1 past the end
    for (int r = tid; r < BM; r += THREADS) {
        const int64_t R = m0 + r;
        int64_t off = -1;
        if (R < a.rows) off = LOAD == LOAD_GATHER ? window_row_to_token(a.g, R) * a.K : R * a.lda;
        row_off[r] = off;
    }
    for (int n = tid; n < BN; n += THREADS) sbias[n] = a.bias ? __bfloat162float(a.bias[n0 + n]) : 0.f;
    if (tid == 0) {
        for (int s = 0; s < STAGES + 1; ++s) mbar_init(smem_u32(&bars[s]), 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // (every global read comes after: a no-op unless launched to overlap the
    // kernels before it)
    griddep_launch_dependents();
    griddep_wait();

    auto load_stage = [&](int kb, int s) {
        const uint32_t a_base = smem_u32(sA + s * L::a_stage);
        const uint32_t b_base = smem_u32(sB + s * b_stage);
        const int c = tid % CPR;
        const int k0 = kb * BK + c * 8;
        const bool kin = k0 < a.K;
#pragma unroll
        for (int i = 0; i < CPR; ++i) {
            const int r = tid / CPR + (THREADS / CPR) * i;
            const int64_t off = row_off[r];
            const bool ok = kin && off >= 0;
            const bf16 *src = ok ? a.A + off + k0 : a.A;
            cp_async16(a_base + L::offset(r, c), src, ok ? 16u : 0u);
        }
        for (int n = tid / CPR; n < BN; n += THREADS / CPR) {
            const bf16 *src = kin ? a.Bw + (int64_t)(n0 + n) * a.K + k0 : a.Bw;
            cp_async16(b_base + L::offset(n, c), src, kin ? 16u : 0u);
        }
    };

    const uint32_t idesc = idesc_bf16(BM, BN);
    bool failed = false;

#pragma unroll 1
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KB) load_stage(s, s);
        cp_async_commit();
    }
#pragma unroll 1
    for (int kb = 0; kb < KB; ++kb) {
        const int nk = kb + STAGES - 1;
        if (nk < KB) {
            // stage nk % STAGES was last read by the MMAs of block kb - 1
            if (kb >= 1 && !failed) {
                const int pk = kb - 1;
                if (!mbar_wait(smem_u32(&bars[pk % STAGES]), (pk / STAGES) & 1, st.wait_ns)) failed = true;
            }
            if (!failed) load_stage(nk, nk % STAGES);
        }
        cp_async_commit();
        cp_async_wait<STAGES - 1>();
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
        tc_fence_after();
        if (tid == 0) {
            const int s = kb % STAGES;
            const uint32_t a_base = smem_u32(sA + s * L::a_stage);
            const uint32_t b_base = smem_u32(sB + s * b_stage);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                if (kb * BK + k * 16 < a.K)
                    mma_bf16(tmem, L::desc(a_base + 32 * k), L::desc(b_base + 32 * k), idesc, (kb | k) != 0);
            }
            mma_commit(smem_u32(&bars[s]));
        }
    }
    cp_async_wait<0>();
    if (!failed) {
        const int lk = KB - 1;
        if (!mbar_wait(smem_u32(&bars[lk % STAGES]), (lk / STAGES) & 1, st.wait_ns)) failed = true;
    }
    if (__syncthreads_or(failed)) failed = true;
    tc_fence_after();

    if (!failed) {
        const int r = warp * 32 + lane;
        const int64_t R = m0 + r;
        bf16 *dst_row = nullptr;
        if (R < a.rows) {
            if (STORE == STORE_SCATTER) dst_row = a.D + window_row_to_token(a.g, R) * (int64_t)a.N + n0;
            else dst_row = a.D + R * a.ldd + n0;
        }
        const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
        int c0 = 0;
        for (; c0 + 32 <= BN; c0 += 32) {
            float v[32];
            tmem_ld32(t_lane + c0, v);
            tmem_wait_ld();
            if (n0 + c0 < a.norm_cols) {
                // V2: this 32-column chunk is one head's q or k; bias first, then
                // scale to unit length (norm clamped at 1e-12) before rounding
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] += sbias[c0 + i];
                    ss = fmaf(v[i], v[i], ss);
                }
                const float nrm = fmaxf(sqrtf(ss), 1e-12f), inv = 1.0f / nrm;
                float zero[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v[i] *= inv;
                    zero[i] = 0.f;
                }
                if (dst_row) store_row_bf16(dst_row + c0, v, zero, 32);
                if (a.norms && R < a.rows) a.norms[R * (a.norms_ld ? a.norms_ld : a.norm_cols / 32) + (n0 + c0) / 32] = nrm;
            } else if (dst_row) {
                if (a.epi == EPI_NONE) {
                    store_row_bf16(dst_row + c0, v, sbias + c0, 32);
                } else {
                    float e[32], zero[32];
                    epilogue_op(a, R, n0 + c0, v, sbias + c0, e, 32);
#pragma unroll
                    for (int i = 0; i < 32; ++i) zero[i] = 0.f;
                    store_row_bf16(dst_row + c0, e, zero, 32);
                }
            }
        }
        if (c0 < BN) { // 16-column tail
            float v[16];
            tmem_ld16(t_lane + c0, v);
            tmem_wait_ld();
            if (dst_row) {
                if (a.epi == EPI_NONE) {
                    store_row_bf16(dst_row + c0, v, sbias + c0, 16);
                } else {
                    float e[16], zero[16];
                    epilogue_op(a, R, n0 + c0, v, sbias + c0, e, 16);
#pragma unroll
                    for (int i = 0; i < 16; ++i) zero[i] = 0.f;
                    store_row_bf16(dst_row + c0, e, zero, 16);
                }
            }
        }
    } else if (tid == 0) {
        atomicOr(st.err, ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, tmem_cols);
}

// ---- persistent GEMM with the weight matrix resident in shared memory -----------
//
// For the block's projections the whole weight matrix Bw [N, K] fits in
// shared memory (K-major, 128-byte swizzle, 64-wide K blocks).  One CTA per
// SM keeps it there and walks over 128-row tiles (for N > 256 as two column
// halves from the same A stages), with three warp roles:
//   warp 0      producer: 128 x 64 A blocks into a ring of stages by TMA (plain
//               rows); for rows gathered through the window map, warps 0 and
//               10..16 each bring 16 rows of every block by cp.async
//   warp 1      one thread issues the MMAs of a tile into one of two TMEM
//               accumulators (N > 256: half 0 into one, half 1 into the other),
//               releasing each A stage by tcgen05.commit once the last half read it
//   warps 2..9  epilogue: two warps per TMEM lane quadrant (alternate 32-column
//               chunks) drain the other accumulator while the next tile runs.
// Every wait is bounded; a timeout sets the error word and ends the kernel.
constexpr int RS_NEPI = 8;
constexpr int RS_NPROD = 8; // producer warps for gathered rows (warp 0 and warps 10..16)
constexpr int RS_THREADS = 32 * (2 + RS_NEPI + RS_NPROD - 1);
constexpr int RS_DEPTH = 4; // cp.async groups a producer lane keeps in flight (gathered rows)
constexpr int RS_STAGE = BM * 128;

struct RsPlan {
    int BN, nbn, KB, stages;
    uint32_t tcols;
    size_t b_bytes, smem;
    int ng;   // column groups: CTA b does column chunk b % ng of every ng-th row block (1: none)
    // stores staged through shared memory (rs_warp_store): for epilogues that
    // only add the bias (and V2's unit length), whose time goes to the stores;
    // the GELU and residual epilogues store directly and keep the 16 KB for a
    // deeper A ring
    int staged;
};

// Column chunk c0 .. c0+n of a plain-store GEMM as a GEMM of its own (its
// weight rows, bias, output columns, residual columns and normalised chunks).
__host__ __device__ inline GemmArgs column_chunk(const GemmArgs &a, int c0, int n)
{
    GemmArgs c = a;
    c.Bw = a.Bw + (int64_t)c0 * a.K;
    if (a.bias) c.bias = a.bias + c0;
    c.D = a.D + c0;
    c.N = n;
    if (a.R) c.R = a.R + c0;
    if (a.norm_cols > 0) {
        c.norm_cols = a.norm_cols - c0 < 0 ? 0 : (a.norm_cols - c0 > n ? n : a.norm_cols - c0);
        c.norms_ld = a.norms_ld ? a.norms_ld : a.norm_cols / 32;
        c.norms = a.norms && c.norm_cols > 0 ? a.norms + c0 / 32 : nullptr;
    }
    return c;
}

// One 32-column chunk of this thread's output row, stored directly (the
// GELU and residual epilogues).
__device__ __forceinline__ void rs_epilogue_chunk32(const GemmArgs &a, int64_t R, int n, bf16 *dst, float (&v)[32],
                                                   const float *bias, bool norm)
{
    if (norm) {
        // V2: this 32-column chunk is one head's q or k; bias first, then scale
        // to unit length (norm clamped at 1e-12) before rounding
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] += bias[i];
            ss = fmaf(v[i], v[i], ss);
        }
        const float nrm = fmaxf(sqrtf(ss), 1e-12f), inv = 1.0f / nrm;
        if (a.norms) a.norms[R * (a.norms_ld ? a.norms_ld : a.norm_cols / 32) + n / 32] = nrm;
        float zero[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] *= inv;
            zero[i] = 0.f;
        }
        store_row_bf16(dst, v, zero, 32);
    } else if (a.epi == EPI_NONE) {
        store_row_bf16(dst, v, bias, 32);
    } else if (a.epi == EPI_RESID) {
        // residual row read 16 bytes at a time (R < rows here)
        const uint4 *res = reinterpret_cast<const uint4 *>(a.R + R * a.ldr + n);
        float e[32], zero[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = res[q];
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = unpack_bf16x2(w[t]);
                e[8 * q + 2 * t] = v[8 * q + 2 * t] + bias[8 * q + 2 * t] + f.x;
                e[8 * q + 2 * t + 1] = v[8 * q + 2 * t + 1] + bias[8 * q + 2 * t + 1] + f.y;
            }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
        store_row_bf16(dst, e, zero, 32);
    } else {
        float e[32], zero[32];
        epilogue_op(a, R, n, v, bias, e, 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) zero[i] = 0.f;
        store_row_bf16(dst, e, zero, 32);
    }
}

// One 32-column chunk of this thread's output row as 16 packed bf16 pairs:
// bias, then (V2) unit length, the residual or the MLP's activation.  (The
// additions of zero keep the bits of a plain bias-add store: -0 becomes +0.)
// `valid`: the row exists (rows past the end compute on whatever TMEM holds
// and are never stored).
__device__ __forceinline__ void rs_chunk_words(const GemmArgs &a, int64_t R, bool valid, int n, float (&v)[32],
                                               const float *bias, bool norm, uint32_t (&w)[16])
{
    if (norm) {
        // V2: this 32-column chunk is one head's q or k; bias first, then scale
        // to unit length (norm clamped at 1e-12) before rounding
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] += bias[i];
            ss = fmaf(v[i], v[i], ss);
        }
        const float nrm = fmaxf(sqrtf(ss), 1e-12f), inv = 1.0f / nrm;
        if (valid && a.norms) a.norms[R * (a.norms_ld ? a.norms_ld : a.norm_cols / 32) + n / 32] = nrm;
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i] * inv + 0.f, v[2 * i + 1] * inv + 0.f);
    } else if (a.epi == EPI_NONE) {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i] + bias[2 * i], v[2 * i + 1] + bias[2 * i + 1]);
    } else if (a.epi == EPI_RESID) {
        // residual row read 16 bytes at a time
        const uint4 *res = reinterpret_cast<const uint4 *>(a.R + R * a.ldr + n);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 u = valid ? res[q] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t wr[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float2 f = unpack_bf16x2(wr[t]);
                const int i = 8 * q + 2 * t;
                w[4 * q + t] = pack_bf16x2(v[i] + bias[i] + f.x + 0.f, v[i + 1] + bias[i + 1] + f.y + 0.f);
            }
        }
    } else {
        float e[32];
        epilogue_op(a, R, n, v, bias, e, 32);
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(e[2 * i] + 0.f, e[2 * i + 1] + 0.f);
    }
}

// The warp's 32 rows of one 32-column chunk (this thread's: w) to global
// memory: staged in the warp's 2 KB of shared memory (16-byte pieces XOR-
// swizzled by row: no bank conflicts either way), then written back with
// four lanes per row, 8 rows x 64 bytes per instruction, instead of 32 rows x
// 16 bytes (a quarter of the L2 write requests, whole sectors).  dk[k]: the
// output row of warp row 8k + lane / 4 (null: not stored), col its offset.
__device__ __forceinline__ void rs_warp_store(uint8_t *stage, const uint32_t (&w)[16], bf16 *const (&dk)[4], int col,
                                              int lane)
{
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4 *>(stage + lane * 64 + ((c ^ sw) << 4)) =
            make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    __syncwarp();
    const int c = lane & 3;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int rr = 8 * k + (lane >> 2);
        const uint4 u = *reinterpret_cast<const uint4 *>(stage + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4));
        if (dk[k]) *reinterpret_cast<uint4 *>(dk[k] + col + 8 * c) = u;
    }
    __syncwarp();   // (the stage is written again by the next chunk)
}

template <int LOAD, int STORE, bool GROUPS>
__global__ void __launch_bounds__(RS_THREADS, 1)
gemm_rs_kernel(GemmArgs a_full, RsPlan pl, DeviceStatus st, const __grid_constant__ CUtensorMap tmA)
{
    // GROUPS (column groups): this CTA's chunk of the output columns (its
    // weights stay resident), every ng-th row block; the ng CTAs of a row
    // block run about together, so its A rows come from DRAM once and from L2
    // after that.  (Without, the arguments stay in the parameter space.)
    const int ng = GROUPS ? pl.ng : 1;
    const int m_first = (int)(blockIdx.x / ng), m_step = (int)(gridDim.x / ng);
    GemmArgs a_chunk;
    if (GROUPS) a_chunk = column_chunk(a_full, (int)(blockIdx.x % ng) * (a_full.N / ng), a_full.N / ng);
    const GemmArgs &a = GROUPS ? a_chunk : a_full;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align(smem_raw, 1024);
    const int S = pl.stages, BN = pl.BN, nbn = pl.nbn, KB = pl.KB;
    uint8_t *sB = smem;
    uint8_t *sA = smem + pl.b_bytes;
    uint8_t *sstage = sA + (size_t)S * RS_STAGE;   // (staged) [RS_NEPI warps][32 rows][64 B]: the stores' staging
    float *sbias = reinterpret_cast<float *>(sstage + (pl.staged ? RS_NEPI * 2048 : 0));
    int64_t *rowoff = reinterpret_cast<int64_t *>(sbias + 512); // producer's gathered rows of the tile
    uint64_t *bars = reinterpret_cast<uint64_t *>(rowoff + BM);
    uint64_t *full = bars, *empty = bars + S, *tfull = bars + 2 * S, *tempty = bars + 2 * S + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + 2 * S + 4);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // row blocks of 128 rows; for N > 256 each block is done as two column
    // halves, one per TMEM accumulator, from the same A stages (loaded once)
    const int64_t mtiles = (a.rows + BM - 1) / BM;

    // the weight matrix, once (zero past K), and the bias
    for (int e = tid; e < a.N * KB * 8; e += RS_THREADS) {
        const int n = e / (KB * 8), rem = e - n * (KB * 8), kb = rem >> 3, c = rem & 7;
        const int k0 = kb * 64 + c * 8;
        const bool ok = k0 < a.K;
        cp_async16(smem_u32(sB) + (uint32_t)kb * (uint32_t)(a.N * 128) + sw128_offset(n, c),
                   ok ? a.Bw + (int64_t)n * a.K + k0 : a.Bw, ok ? 16u : 0u);
    }
    cp_async_commit();
    for (int n = tid; n < a.N; n += RS_THREADS) sbias[n] = a.bias ? __bfloat162float(a.bias[n]) : 0.f;
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full[s]), LOAD == LOAD_GATHER ? RS_NPROD : 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&tfull[b]), 1);
            mbar_init(smem_u32(&tempty[b]), RS_NEPI);
        }
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tslot), pl.tcols);
        tmem_relinquish();
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t half_cols = pl.tcols / 2;
    // the prologue read only the weights and the bias: A, R and D wait for the
    // kernels queued before this one (a no-op unless launched to overlap them)
    griddep_launch_dependents();
    griddep_wait();
    bool failed = false;

    if (warp == 0 || warp >= 2 + RS_NEPI) {
        // ---------------- producer(s) ----------------
        const int pw = warp == 0 ? 0 : warp - (1 + RS_NEPI); // 0..RS_NPROD-1
        int64_t it = 0;
        if (LOAD == LOAD_PLAIN) {
            if (warp == 0 && lane == 0) {
                for (int64_t m = m_first; m < mtiles && !failed; m += m_step) {
                    const int64_t m0 = m * BM;
                    for (int kb = 0; kb < KB; ++kb, ++it) {
                        const int s = (int)(it % S);
                        if (!mbar_wait(smem_u32(&empty[s]), (uint32_t)((it / S) & 1) ^ 1u, st.wait_ns)) {
                            failed = true;
                            break;
                        }
                        mbar_arrive_expect_tx(smem_u32(&full[s]), RS_STAGE);
                        tma_load_2d(smem_u32(sA + (size_t)s * RS_STAGE), &tmA, kb * 64, (int)m0, smem_u32(&full[s]));
                    }
                }
            }
        } else {
            for (int64_t m = m_first; m < mtiles && !failed; m += m_step) {
                const int64_t m0 = m * BM;
                // this warp's rows of the tile (BM / RS_NPROD of them): source
                // offsets (32-bit index map when it fits) into shared memory
                constexpr int RPW = BM / RS_NPROD;
                const bool small = a.g.T < ((int64_t)1 << 31);
                int64_t *myoff = rowoff + RPW * pw;
                __syncwarp();
                if (lane < RPW) {
                    const int64_t R = m0 + RPW * pw + lane;
                    const int64_t tok = R >= a.rows ? -1
                                        : small     ? (int64_t)window_row_to_token32(a.g, (int)R)
                                                    : window_row_to_token(a.g, R);
                    myoff[lane] = tok < 0 ? -1 : tok * a.K;
                }
                __syncwarp();
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = (int)(it % S);
                    // warp-uniform outcome: the lanes meet at __syncwarp below
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(smem_u32(&empty[s]), (uint32_t)((it / S) & 1) ^ 1u, st.wait_ns))) {
                        failed = true;
                        break;
                    }
                    const uint32_t dst = smem_u32(sA + (size_t)s * RS_STAGE);
                    // eight lanes per row (one 128-byte line), four rows per
                    // instruction; 16-byte chunks past K are never read by the MMAs
                    const int c = lane & 7, k0 = kb * 64 + c * 8;
                    if (k0 < a.K) {
#pragma unroll
                        for (int j = 0; j < RPW / 4; ++j) {
                            const int rl = 4 * j + (lane >> 3);
                            const int64_t off = myoff[rl];
                            cp_async16(dst + sw128_offset(RPW * pw + rl, c), off >= 0 ? a.A + off + k0 : a.A,
                                       off >= 0 ? 16u : 0u);
                        }
                    }
                    cp_async_commit();
                    if (it >= RS_DEPTH) {
                        // every lane's copies of that stage have landed: one arrival per warp
                        cp_async_wait<RS_DEPTH>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&full[(it - RS_DEPTH) % S]));
                    }
                }
            }
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (!failed && lane == 0)
                for (int64_t j = it - RS_DEPTH < 0 ? 0 : it - RS_DEPTH; j < it; ++j) mbar_arrive(smem_u32(&full[j % S]));
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(BM, BN);
            int64_t it = 0, lm = 0;
            for (int64_t m = m_first; m < mtiles && !failed; m += m_step, ++lm) {
                const int64_t it0 = it;
                for (int nb = 0; nb < nbn && !failed; ++nb) {
                    // accumulator: alternate per row block (one half), or one per half
                    const int buf = nbn == 2 ? nb : (int)(lm & 1);
                    const uint32_t par = nbn == 2 ? (uint32_t)(lm & 1) : (uint32_t)((lm >> 1) & 1);
                    if (!mbar_wait(smem_u32(&tempty[buf]), par ^ 1u, st.wait_ns)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)buf * half_cols;
                    const uint32_t b_col = (uint32_t)nb * (uint32_t)BN * 128u;
                    for (int kb = 0; kb < KB; ++kb) {
                        const int64_t i = it0 + kb;
                        const int s = (int)(i % S);
                        if (nb == 0) {
                            if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((i / S) & 1), st.wait_ns)) {
                                failed = true;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t a_base = smem_u32(sA + (size_t)s * RS_STAGE);
                        const uint32_t b_base = smem_u32(sB) + (uint32_t)kb * (uint32_t)(a.N * 128) + b_col;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if (kb * 64 + k * 16 < a.K)
                                mma_bf16(d, desc_kmajor_sw128(a_base + 32 * k), desc_kmajor_sw128(b_base + 32 * k), idesc,
                                         (kb | k) != 0);
                        // the stage is free once the last half has read it
                        if (nb == nbn - 1) mma_commit(smem_u32(&empty[s]));
                    }
                    if (failed) break;
                    mma_commit(smem_u32(&tfull[buf]));
                }
                it = it0 + KB;
            }
        }
    } else {
        // ---------------- epilogue ----------------
        const int quad = warp & 3, half = (warp - 2) >> 2;
        const int r = quad * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16);
        const int nchunks = BN / 32;
        int64_t lm = 0;
        for (int64_t m = m_first; m < mtiles && !failed; m += m_step, ++lm)
        for (int nb = 0; nb < nbn; ++nb) {
            const int buf = nbn == 2 ? nb : (int)(lm & 1);
            const uint32_t par = nbn == 2 ? (uint32_t)(lm & 1) : (uint32_t)((lm >> 1) & 1);
            // (warp-uniform outcome: the warp's TMEM loads, shuffles and staged
            // stores below are warp-collective)
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&tfull[buf]), par, st.wait_ns))) {
                failed = true;
                break;
            }
            tc_fence_after();
            int64_t R = m * BM + r;
            const int n0 = nb * BN;
            bf16 *dst_row = nullptr;
            if (R < a.rows) {
                if (STORE == STORE_SCATTER) {
                    dst_row = a.D + window_row_to_token(a.g, R) * (int64_t)a.N + n0;
                } else if (STORE == STORE_WINDOW) {
                    R = token_to_window_row(a.g, R);   // the output row (and its norms' row)
                    dst_row = a.D + R * a.ldd + n0;
                } else {
                    dst_row = a.D + R * a.ldd + n0;
                }
            }
            const uint32_t tb = t_lane + (uint32_t)buf * half_cols;
            // the output rows this lane writes back for the warp (rows 8k + lane / 4)
            bf16 *dk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                dk[k] = reinterpret_cast<bf16 *>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst_row), 8 * k + (lane >> 2)));
            uint8_t *stage = sstage + (warp - 2) * 2048;
            if (pl.staged) {   // (uniform over the CTA)
                for (int ci = half; ci < nchunks; ci += 2) {
                    float v[32];
                    uint32_t w[16];
                    tmem_ld32(tb + 32 * ci, v);
                    tmem_wait_ld();
                    rs_chunk_words(a, R, dst_row != nullptr, n0 + 32 * ci, v, sbias + n0 + 32 * ci,
                                   n0 + 32 * ci < a.norm_cols, w);
                    rs_warp_store(stage, w, dk, 32 * ci, lane);
                }
            } else {
                for (int ci = half; ci < nchunks; ci += 2) {
                    float v[32];
                    tmem_ld32(tb + 32 * ci, v);
                    tmem_wait_ld();
                    if (dst_row)
                        rs_epilogue_chunk32(a, R, n0 + 32 * ci, dst_row + 32 * ci, v, sbias + n0 + 32 * ci,
                                            n0 + 32 * ci < a.norm_cols);
                }
            }
            if ((BN & 31) && (nchunks & 1) == half) { // 16-column tail
                const int c0 = 32 * nchunks;
                float v[16];
                tmem_ld16(tb + c0, v);
                tmem_wait_ld();
                if (dst_row) {
                    if (a.epi == EPI_NONE) {
                        store_row_bf16(dst_row + c0, v, sbias + n0 + c0, 16);
                    } else {
                        float e[16], zero[16];
                        epilogue_op(a, R, n0 + c0, v, sbias + n0 + c0, e, 16);
#pragma unroll
                        for (int i = 0; i < 16; ++i) zero[i] = 0.f;
                        store_row_bf16(dst_row + c0, e, zero, 16);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&tempty[buf]));
        }
    }
    if (failed && lane == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, pl.tcols);
}

// The resident-weight plan, or false when the weights (or two accumulators)
// do not fit: N a multiple of 16, one tile column of N <= 256 or two halves,
// the V2 normalisation's 32-column chunks whole, Bw within 152 KB.
bool rs_plan(const GemmArgs &a, RsPlan &p)
{
    if (a.N <= 0 || a.N % 16 || a.N > 512 || a.K <= 0 || a.K % 16) return false;
    p.ng = 1;
    p.nbn = a.N <= 256 ? 1 : 2;
    p.BN = a.N / p.nbn;
    if (p.BN % 16 || (a.norm_cols > 0 && p.BN % 32)) return false;
    if (a.epi == EPI_RESID && ((a.ldr % 8) || (reinterpret_cast<uintptr_t>(a.R) & 15))) return false;
    p.KB = (a.K + 63) / 64;
    p.b_bytes = (size_t)a.N * p.KB * 128;
    if (p.b_bytes > 152 * 1024) return false;
    p.staged = a.epi == EPI_NONE;
    const size_t fixed = 1024 + p.b_bytes + (p.staged ? RS_NEPI * 2048 : 0) + 512 * 4 + BM * 8 + 256;
    p.stages = (int)((227 * 1024 - fixed) / RS_STAGE);
    if (p.stages > 8) p.stages = 8;
    if (p.stages < 3) return false;
    if (p.nbn == 2 && p.KB > p.stages) return false; // both halves read a block's stages
    p.tcols = 2 * p.BN <= 256 ? 256 : 512;
    p.smem = fixed + (size_t)p.stages * RS_STAGE;
    return true;
}

template <int LOAD, int STORE>
cudaError_t launch_rs(const GemmArgs &a, const RsPlan &pl, DeviceStatus st, cudaStream_t stream)
{
    CUtensorMap tmA;
    memset(&tmA, 0, sizeof(tmA));
    if (LOAD == LOAD_PLAIN) {
        if ((a.lda * 2) % 16 || (reinterpret_cast<uintptr_t>(a.A) & 15)) return cudaErrorInvalidValue;
        cudaError_t e = make_tensor_map_sw128(&tmA, a.A, a.rows, a.K, a.lda, BM);
        if (e != cudaSuccess) return e;
    }
    auto kern = pl.ng > 1 ? gemm_rs_kernel<LOAD, STORE, true> : gemm_rs_kernel<LOAD, STORE, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    }
    const int64_t mtiles = (a.rows + BM - 1) / BM;
    const int ng = pl.ng > 1 ? pl.ng : 1;
    const int64_t per = sms / ng;   // CTAs per column group
    const unsigned grid = (unsigned)((mtiles < per ? mtiles : per) * ng);
    e = launch_maybe_overlapped(kern, dim3(grid), dim3(RS_THREADS), pl.smem, stream, a.overlap, a, pl, st, tmA);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Largest N tile <= 128 that divides N and is a multiple of `step` (16, or
// 32 when 32-column chunks must stay whole); larger only when nothing <= 128
// divides N.  (At most 128 columns keep a CTA's 3-stage ring under 100 KB,
// so that two CTAs share an SM and one's epilogue overlaps the other's
// loads.)
int pick_bn(int N, int step)
{
    for (int bn = 128 / step * step; bn >= step; bn -= step)
        if (N % bn == 0) return bn;
    for (int bn = 256 / step * step; bn > 128; bn -= step)
        if (N % bn == 0) return bn;
    return 0;
}

template <int LOAD, int STORE, int BK, int NSTAGES>
cudaError_t launch_stages(const GemmArgs &a, int BN, DeviceStatus st, cudaStream_t stream)
{
    const size_t smem = GemmSmem<BK, NSTAGES>::bytes(BN);
    auto kern = gemm_tc_kernel<LOAD, STORE, BK, NSTAGES>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.rows + BM - 1) / BM), (unsigned)(a.N / BN));
    e = launch_maybe_overlapped(kern, grid, dim3(THREADS), smem, stream, a.overlap, a, BN, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// A K of at most two 64-wide blocks gets a 2-stage ring: the smaller shared
// footprint lets a third CTA share the SM (its loads and epilogue overlap the
// others').
template <int LOAD, int STORE, int BK = 64>
cudaError_t launch_impl(const GemmArgs &a, DeviceStatus st, cudaStream_t stream)
{
    const int BN = pick_bn(a.N, a.norm_cols > 0 ? 32 : 16);
    if (BN == 0 || a.K % 16 != 0 || a.rows <= 0) return cudaErrorInvalidValue;
    if (BK == 64 && (a.K + BK - 1) / BK <= 2) return launch_stages<LOAD, STORE, BK, 2>(a, BN, st, stream);
    return launch_stages<LOAD, STORE, BK, GemmSmem<BK>::STAGES>(a, BN, st, stream);
}

// Test kernel of the TMEM-A form of the MMA: each thread writes its A row
// (K <= 128 bf16, packed in pairs) into TMEM columns 256.., B (N <= 256 rows,
// K-major, 128-byte swizzle) goes to shared memory, then K/16 MMAs read A from
// TMEM and accumulate D in columns 0..N-1.
__global__ void __launch_bounds__(THREADS) gemm_ts_test_kernel(GemmArgs a, DeviceStatus st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align(smem_raw, 1024);
    uint8_t *sB = smem;                                          // 2 K blocks x [N rows][128 B]
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * 256 * 128);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int N = a.N, K = a.K;
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init_fence();
    }
    // B rows -> shared memory (zero past K)
    for (int q = tid; q < N * 16; q += THREADS) {
        const int n = q / 16, c16 = q % 16;
        const int k0 = c16 * 8;
        const bool ok = k0 < K;
        cp_async16(smem_u32(sB) + (c16 >> 3) * (256 * 128) + sw128_offset(n, c16 & 7),
                   ok ? a.Bw + (int64_t)n * K + k0 : a.Bw, ok ? 16u : 0u);
    }
    cp_async_commit();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    // A row of this thread -> TMEM columns 256 + (K/2), zeros past the end
    {
        const int64_t R = m0 + tid;
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int k = 2 * (c0 + i);
                r[i] = R < a.rows ? *reinterpret_cast<const uint32_t *>(a.A + R * a.lda + k) : 0u;
            }
            tmem_st16(t_lane + 256 + c0, r);
        }
        tmem_wait_st();
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint32_t id = idesc_bf16(BM, N);
        for (int kk = 0; kk < K / 16; ++kk)
            mma_bf16_ts(tmem, tmem + 256 + 8 * kk,
                        desc_kmajor_sw128(smem_u32(sB) + (kk >> 2) * (256 * 128) + 32 * (kk & 3)), id, kk != 0);
        mma_commit(smem_u32(bar));
    }
    const bool ok = mbar_wait(smem_u32(bar), 0, st.wait_ns);
    tc_fence_after();
    const int64_t R = m0 + tid;
    for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld16(t_lane + c0, v);
        tmem_wait_ld();
        if (R < a.rows && ok) {
            float b[16];
            for (int i = 0; i < 16; ++i) b[i] = a.bias ? __bfloat162float(a.bias[c0 + i]) : 0.f;
            store_row_bf16(a.D + R * a.ldd + c0, v, b, 16);
        }
    }
    if (!ok && tid == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// Test kernel of an MN-major B operand: Bmn is [K, N] row-major (N = 32 or
// 64); each K row of a 32-wide N group is one 64-byte row of a 64B-swizzled
// tile, K groups of 8 rows 512 B apart, N groups K*64 bytes apart.  A is
// K-major (128-byte swizzle), K <= 128.
__global__ void __launch_bounds__(THREADS) gemm_mn_test_kernel(GemmArgs a, DeviceStatus st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align(smem_raw, 1024);
    uint8_t *sA = smem;                                          // 2 K blocks x [128 rows][128 B]
    uint8_t *sB = smem + 2 * 128 * 128;                          // 2 N groups x [128 K rows][64 B]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + 2 * 128 * 64);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int N = a.N, K = a.K;
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 64);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init_fence();
    }
    for (int q = tid; q < 128 * 16; q += THREADS) {               // A rows (zero past rows / K)
        const int r = q / 16, c16 = q % 16;
        const int64_t R = m0 + r;
        const bool ok = R < a.rows && c16 * 8 < K;
        cp_async16(smem_u32(sA) + (c16 >> 3) * (128 * 128) + sw128_offset(r, c16 & 7),
                   ok ? a.A + R * a.lda + c16 * 8 : a.A, ok ? 16u : 0u);
    }
    for (int q = tid; q < K * (N / 8); q += THREADS) {            // B rows k, 16-byte chunks of N
        const int k = q / (N / 8), c16 = q % (N / 8);
        cp_async16(smem_u32(sB) + (c16 >> 2) * (K * 64) + sw64_offset(k, c16 & 3), a.Bw + (int64_t)k * N + c16 * 8,
                   16);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (tid == 0) {
        const uint32_t id = idesc_bf16_bmn(BM, N);
        for (int kk = 0; kk < K / 16; ++kk)
            mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sA) + (kk >> 2) * (128 * 128) + 32 * (kk & 3)),
                     desc_mnmajor_sw64(smem_u32(sB) + kk * 1024, K * 64), id, kk != 0);
        mma_commit(smem_u32(bar));
    }
    const bool ok = mbar_wait(smem_u32(bar), 0, st.wait_ns);
    tc_fence_after();
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    const int64_t R = m0 + tid;
    for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
        tmem_ld16(t_lane + c0, v);
        tmem_wait_ld();
        if (R < a.rows && ok) {
            float b[16];
            for (int i = 0; i < 16; ++i) b[i] = a.bias ? __bfloat162float(a.bias[c0 + i]) : 0.f;
            store_row_bf16(a.D + R * a.ldd + c0, v, b, 16);
        }
    }
    if (!ok && tid == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

// Test kernel of the lane-masked MMA forms: every 128-row block is two halves
// that each see their own B.  Bw is [2N, K]; rows 0..63 of a block multiply
// B0 = Bw[0:N], rows 64..127 B1 = Bw[N:2N], written into the same N columns
// by two MMAs with complementary lane masks -- once with A from shared memory
// (D columns 0..N-1 of the output) and once with A from TMEM (columns N..2N-1).
// K <= 128 (multiple of 32), N <= 128 (multiple of 16).
__global__ void __launch_bounds__(THREADS) gemm_pair_test_kernel(GemmArgs a, DeviceStatus st)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align(smem_raw, 1024);
    uint8_t *sA = smem;                                          // 2 K blocks x [128 rows][128 B]
    uint8_t *sB = smem + 2 * 128 * 128;                          // 2 K blocks x [256 rows][128 B]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sB + 2 * 256 * 128);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int64_t m0 = (int64_t)blockIdx.x * BM;
    const int N = a.N, K = a.K;
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_u32(bar), 1);
        mbar_init_fence();
    }
    for (int q = tid; q < 128 * 16; q += THREADS) {               // A rows (zero past rows / K)
        const int r = q / 16, c16 = q % 16;
        const int64_t R = m0 + r;
        const bool ok = R < a.rows && c16 * 8 < K;
        cp_async16(smem_u32(sA) + (c16 >> 3) * (128 * 128) + sw128_offset(r, c16 & 7),
                   ok ? a.A + R * a.lda + c16 * 8 : a.A, ok ? 16u : 0u);
    }
    for (int q = tid; q < 2 * N * 16; q += THREADS) {             // B0 and B1 rows (zero past K)
        const int n = q / 16, c16 = q % 16;
        const bool ok = c16 * 8 < K;
        cp_async16(smem_u32(sB) + (c16 >> 3) * (256 * 128) + sw128_offset(n, c16 & 7),
                   ok ? a.Bw + (int64_t)n * K + c16 * 8 : a.Bw, ok ? 16u : 0u);
    }
    cp_async_commit();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);
    {   // A row of this thread -> TMEM columns 256 + (K/2)
        const int64_t R = m0 + tid;
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[i] = R < a.rows ? *reinterpret_cast<const uint32_t *>(a.A + R * a.lda + 2 * (c0 + i)) : 0u;
            tmem_st16(t_lane + 256 + c0, r);
        }
        tmem_wait_st();
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint32_t id = idesc_bf16(BM, N);
        const uint32_t keep_top[4] = {0u, 0u, ~0u, ~0u};   // lanes 64..127 masked
        const uint32_t keep_bot[4] = {~0u, ~0u, 0u, 0u};   // lanes 0..63 masked
        for (int half = 0; half < 2; ++half) {
            const uint32_t b0 = smem_u32(sB) + half * N * 128;   // B row offset N: whole 8-row groups
            for (int kk = 0; kk < K / 16; ++kk) {
                const uint64_t bd = desc_kmajor_sw128(b0 + (kk >> 2) * (256 * 128) + 32 * (kk & 3));
                mma_bf16_mask(tmem, desc_kmajor_sw128(smem_u32(sA) + (kk >> 2) * (128 * 128) + 32 * (kk & 3)), bd,
                              id, kk != 0, half ? keep_bot : keep_top);
                mma_bf16_ts_mask(tmem + 128, tmem + 256 + 8 * kk, bd, id, kk != 0, half ? keep_bot : keep_top);
            }
        }
        mma_commit(smem_u32(bar));
    }
    const bool ok = mbar_wait(smem_u32(bar), 0, st.wait_ns);
    tc_fence_after();
    const int64_t R = m0 + tid;
    for (int part = 0; part < 2; ++part)
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(t_lane + 128 * part + c0, v);
            tmem_wait_ld();
            if (R < a.rows && ok) {
                float b[16];
                for (int i = 0; i < 16; ++i) b[i] = 0.f;
                store_row_bf16(a.D + R * a.ldd + part * N + c0, v, b, 16);
            }
        }
    if (!ok && tid == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

} // namespace

cudaError_t launch_gemm_pair_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream)
{
    if (a.K % 32 || a.K > 128 || a.N % 16 || a.N > 128 || a.N < 16 || a.rows <= 0) return cudaErrorInvalidValue;
    const size_t smem = 1024 + 2 * 128 * 128 + 2 * 256 * 128 + 64;
    cudaError_t e = cudaFuncSetAttribute(gemm_pair_test_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gemm_pair_test_kernel<<<(unsigned)((a.rows + BM - 1) / BM), THREADS, smem, stream>>>(a, st);
    return cudaGetLastError();
}

cudaError_t launch_gemm_mn_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream)
{
    if (a.K % 16 || a.K > 128 || (a.N != 32 && a.N != 64) || a.rows <= 0) return cudaErrorInvalidValue;
    const size_t smem = 1024 + 2 * 128 * 128 + 2 * 128 * 64 + 64;
    cudaError_t e = cudaFuncSetAttribute(gemm_mn_test_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gemm_mn_test_kernel<<<(unsigned)((a.rows + BM - 1) / BM), THREADS, smem, stream>>>(a, st);
    return cudaGetLastError();
}

cudaError_t launch_gemm_ts_test(const GemmArgs &a, DeviceStatus st, cudaStream_t stream)
{
    if (a.K % 32 || a.K > 128 || a.N % 16 || a.N > 256 || a.rows <= 0) return cudaErrorInvalidValue;
    const size_t smem = 1024 + 2 * 256 * 128 + 64;
    cudaError_t e = cudaFuncSetAttribute(gemm_ts_test_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gemm_ts_test_kernel<<<(unsigned)((a.rows + BM - 1) / BM), THREADS, smem, stream>>>(a, st);
    return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmArgs &a, int load_mode, int store_mode, DeviceStatus st, cudaStream_t stream)
{
    RsPlan pl;
    // (gathered rows: the producer keeps RS_DEPTH stages in flight)
    auto rs_ok = [&](const GemmArgs &x, RsPlan &p) {
        return x.rows > 0 && rs_plan(x, p) && (load_mode != LOAD_GATHER || p.stages >= RS_DEPTH + 1);
    };
    // gathered rows with a plain store: plain token-order loads, output rows
    // sent to their window-order places (same result, no gathered loads)
    GemmArgs aw = a;
    if (load_mode == LOAD_GATHER && store_mode == STORE_PLAIN) aw.lda = a.K;
    const bool to_window = load_mode == LOAD_GATHER && store_mode == STORE_PLAIN && a.epi != EPI_RESID;
    if (to_window && a.rows > 0 && rs_plan(aw, pl)) return launch_rs<LOAD_PLAIN, STORE_WINDOW>(aw, pl, st, stream);
    if (rs_ok(a, pl)) {
        if (load_mode == LOAD_GATHER && store_mode == STORE_PLAIN) return launch_rs<LOAD_GATHER, STORE_PLAIN>(a, pl, st, stream);
        if (load_mode == LOAD_PLAIN && store_mode == STORE_SCATTER) return launch_rs<LOAD_PLAIN, STORE_SCATTER>(a, pl, st, stream);
        if (load_mode == LOAD_PLAIN && store_mode == STORE_PLAIN) return launch_rs<LOAD_PLAIN, STORE_PLAIN>(a, pl, st, stream);
    }
    // weights too large to stay resident: 2 to 4 (16) column chunks that each fit,
    // one column group of CTAs per chunk in one launch (the groups walk the
    // row blocks together, so A is read from DRAM about once); only where A
    // is no wider than the output (the QKV and the first MLP projections).
    if (store_mode == STORE_PLAIN && a.rows > 0 && a.K <= a.N) {
        // (more than four groups only while A stays in L2 for all of them)
        const bool a_in_l2 = a.rows * a.K * 2 <= ((int64_t)64 << 20);
        for (int nc = 2; nc <= (a_in_l2 ? 16 : 4); ++nc) {
            if (a.N % nc || (a.N / nc) % 16) continue;
            const int n = a.N / nc;
            if (a.norm_cols > 0 && (n % 32 || a.norm_cols % 32)) continue;
            GemmArgs c0 = column_chunk(aw, 0, n);
            if (!(to_window ? rs_plan(c0, pl) : rs_ok(c0, pl))) continue;
            pl.ng = nc;
            return to_window ? launch_rs<LOAD_PLAIN, STORE_WINDOW>(aw, pl, st, stream)
                   : load_mode == LOAD_GATHER ? launch_rs<LOAD_GATHER, STORE_PLAIN>(aw, pl, st, stream)
                                              : launch_rs<LOAD_PLAIN, STORE_PLAIN>(aw, pl, st, stream);
        }
    }
    if (load_mode == LOAD_GATHER && store_mode == STORE_PLAIN) return launch_impl<LOAD_GATHER, STORE_PLAIN>(a, st, stream);
    if (load_mode == LOAD_PLAIN && store_mode == STORE_SCATTER) return launch_impl<LOAD_PLAIN, STORE_SCATTER>(a, st, stream);
    if (load_mode == LOAD_PLAIN && store_mode == STORE_PLAIN) return launch_impl<LOAD_PLAIN, STORE_PLAIN>(a, st, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_sw64(const GemmArgs &a, DeviceStatus st, cudaStream_t stream)
{
    return launch_impl<LOAD_PLAIN, STORE_PLAIN, 32>(a, st, stream);
}

} // namespace swin
