// Window attention on tcgen05 tensor cores, sm_103a.
//
// Per window and head (pages "Boosting Swin Transformer Speed",
// Introduction and Training Optimization -- attention inside shifted windows;
// "Swin Transformer V2" (neura.market), How It Works -- relative position
// bias, scaled cosine attention with tau clipped at 0.01):
//   V1:  a_ij = q_i.k_j / sqrt(d) + table[idx(i,j), head]
//   V2:  a_ij = cos(q_i, k_j) / max(tau, 0.01) + table[idx(i,j), head]
//   a_ij = -inf when i, j lie in different shift regions (shift > 0)
//   o_i  = softmax_j(a_ij) . v_j
// idx(i,j) = (ri-rj+M-1)*(2M-1) + (ci-cj+M-1) (query minus key, in-window
// coordinates).  The mask and the relative index are computed from window
// coordinates; neither is loaded.  Softmax in fp32 with exp2 (logits carry
// a log2(e) factor), P rounded to bf16 for the P.V MMA, 1/rowsum applied to
// the fp32 P.V result.  In V2 the QKV projection has already scaled every q
// and k head to unit length, so q.k is the cosine.
//
// Windows of at most 64 tokens (M = 7 or 8) go to the tcgen05 attention
// kernel shared with the backward pass (csrc/backward.cu, forward mode: two
// windows of one head per 128-row tile, TMA loads, P.V with P block-diagonal).
// This file holds the large-window kernel (N > 64, e.g. M = 24, N = 576): one
// CTA of 256 threads takes 128 queries of one window and head (two threads per
// query row, 64 keys each) and walks the keys in double-buffered tiles of 128
// loaded by 2-D TMA into 64-byte-swizzled tiles, with an online softmax; P goes
// back into TMEM and P.V reads it from there, v used in its [key][d] layout as
// an N-major B operand (no transpose is ever written).
#include <cuda.h>

#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr float LOG2E = 1.4426950408889634f;

// Region id (row band * 3 + column band) of in-window token (ti, tj) of
// window (wi, wj); 0 everywhere when shift == 0.
__device__ __forceinline__ int token_region(const Geom &g, int wi, int wj, int ti, int tj)
{
    if (g.s == 0) return 0;
    return 3 * shift_band(wi * g.M + ti, g.H, g.M, g.s) + shift_band(wj * g.M + tj, g.W, g.M, g.s);
}

// Stores n o values (fp32 scaled by inv_l) as bf16 to attn.
template <int NV>
__device__ __forceinline__ void store_o(bf16 *dst, const float *o, float inv_l)
{
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < NV / 8; ++q)
        d4[q] = make_uint4(pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l),
                           pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l),
                           pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l),
                           pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l));
}

// ---------------------------------------------------------------------------
// Large windows: 128 queries per CTA, 256 threads (two per query row), keys
// in double-buffered tiles of 128, online softmax, P in TMEM.
// ---------------------------------------------------------------------------
constexpr int FL_THREADS = 256;

struct FlashSmem {
    static constexpr int q_off = 0;                    // [128][64 B] SW64
    static constexpr int k_off = q_off + 128 * 64;     // 2 x [128][64 B] SW64
    static constexpr int v_off = k_off + 2 * 128 * 64; // 2 x [128 keys][64 B] SW64 (N-major B)
    static constexpr int end = v_off + 2 * 128 * 64;
    // per-key metadata of the whole window (key_off, key_region: keys rounded
    // up to whole 128-key tiles), smax and spart, the bias table, barriers
    static size_t bytes(int M)
    {
        const size_t keys = (size_t)((M * M + 127) / 128) * 128;
        return 1024 + end + keys * 4 * 2 + 2 * 2 * 128 * 4 + (size_t)(2 * M - 1) * (2 * M - 1) * 4 + 64;
    }
};

// (two CTAs per SM: 2 x 8 warps at <= 128 registers fit each sub-partition's
// register file, and 2 x 256 TMEM columns fit the SM's 512)
__global__ void __launch_bounds__(FL_THREADS, 2)
    attn_flash_kernel(AttnArgs a, DeviceStatus st, const __grid_constant__ CUtensorMap tmap)
{
    extern __shared__ uint8_t smem_raw[];
    const Geom g = a.g;
    const int M = g.M, N = g.N, C = g.C, L = 2 * M - 1;
    uint8_t *sm = smem_align(smem_raw, 1024);
    // after the tiles (1024-aligned): key_off first, so that its int4 loads are
    // 16-byte aligned, then the other per-key and per-row arrays, then the bias
    const int kpad = ((N + 127) / 128) * 128;
    int *key_off = reinterpret_cast<int *>(sm + FlashSmem::end);        // [kpad], relative-bias offset of key
    int *key_region = key_off + kpad;                                    // [kpad], -1 past N
    float *smax = reinterpret_cast<float *>(key_region + kpad);          // [2][128]
    float *spart = smax + 2 * 128;                                       // [2][128]
    float *sbias = spart + 2 * 128;                                      // [L*L], times log2(e)
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_align(reinterpret_cast<uint8_t *>(sbias + L * L), 8));
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 4);
    const uint32_t sQ = smem_u32(sm + FlashSmem::q_off), sK = smem_u32(sm + FlashSmem::k_off),
                   sV = smem_u32(sm + FlashSmem::v_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = quarter * 32 + lane;
    const int head = blockIdx.y;
    const int qtiles = (N + 127) / 128;
    const int64_t win = blockIdx.x / qtiles;
    const int q0 = (int)(blockIdx.x % qtiles) * 128;
    const int per = g.nh * g.nw;
    const int rem = (int)(win % per);
    const int wi = rem / g.nw, wj = rem % g.nw;
    const bool masked = g.s > 0 && (wi == g.nh - 1 || wj == g.nw - 1);
    const int qt = q0 + row;
    const bool row_ok = qt < N;
    const int qi = row_ok ? qt / M : 0, qj = row_ok ? qt % M : 0;
    const int my_region = token_region(g, wi, wj, qi, qj);
    const int base = (qi + M - 1) * L + (qj + M - 1);
    const int ktiles = (N + 127) / 128;

    for (int i = tid; i < L * L; i += FL_THREADS)
        sbias[i] = __bfloat162float(a.table[(int64_t)i * a.heads + head]) * LOG2E;
    // every key of the window: its offset into the relative-bias table and its
    // shift region (once per CTA, not per key tile)
    for (int kj = tid; kj < kpad; kj += FL_THREADS) {
        const bool ok = kj < N;
        const int ki = ok ? kj / M : 0, kc = ok ? kj - ki * M : 0;
        key_off[kj] = ki * L + kc;
        key_region[kj] = ok ? token_region(g, wi, wj, ki, kc) : -1;
    }
    // bars: 0 = S done, 1 = P.V done (two committing threads), 2 + b = key
    // buffer b full (TMA transactions)
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), i == 1 ? 2 : 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    // key tile kt into buffer b: the k and v boxes (128 rows x 32 columns of
    // the qkv buffer, 64-byte swizzled, rows past the tensor zero-filled) by
    // TMA from thread 0, and the key metadata; rows past this window's N are
    // masked below
    const int64_t row0 = win * N;
    // (tile 0 also brings the q rows: one arrival with all three boxes' bytes)
    auto load_keys = [&](int kt, int b) {
        if (tid == 0) {
            const uint32_t full = smem_u32(&bars[2 + b]);
            mbar_arrive_expect_tx(full, (kt == 0 ? 3 : 2) * 128 * 64);
            if (kt == 0) tma_load_2d(sQ, &tmap, head * 32, (int)(row0 + q0), full);
            tma_load_2d(sK + b * (128 * 64), &tmap, C + head * 32, (int)(row0 + kt * 128), full);
            tma_load_2d(sV + b * (128 * 64), &tmap, 2 * C + head * 32, (int)(row0 + kt * 128), full);
        }
    };
    __syncthreads();   // barrier initialisation is visible before any TMA completes on it
    load_keys(0, 0);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t bar_s = smem_u32(&bars[0]), bar_pv = smem_u32(&bars[1]);
    const float scale = a.mode == 1 ? LOG2E / fmaxf(a.tau[head], 0.01f) : LOG2E * rsqrtf(32.0f);

    float o[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool failed = false;
    uint32_t phase = 0;

#pragma unroll 1
    for (int kt = 0; kt < ktiles; ++kt) {
        const int b = kt & 1;
        if (kt + 1 < ktiles) load_keys(kt + 1, b ^ 1);
        // tile kt (and, for kt = 0, the q rows) have landed.  (No CTA barrier
        // here: the S MMA overwrites TMEM columns that every thread finished
        // reading before the previous tile's P store barrier, and a failed
        // wait becomes uniform at the next barrier.)
        if (!mbar_wait(smem_u32(&bars[2 + b]), (kt >> 1) & 1, st.wait_ns)) failed = true;
        if (tid == 0 && !failed) {
            const uint32_t id = idesc_bf16(128, 128);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tmem, desc_kmajor_sw64(sQ + 32 * k), desc_kmajor_sw64(sK + b * (128 * 64) + 32 * k), id, k);
            mma_commit(bar_s);
        }
        if (!mbar_wait(bar_s, phase, st.wait_ns)) failed = true;
        tc_fence_after();

        // logits of this thread's 64 keys (64*half .. +63 of the tile)
        float sv[64];
        {
            float c0[32], c1[32];
            tmem_ld32(t_lane + 64 * half, c0);
            tmem_ld32(t_lane + 64 * half + 32, c1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) { sv[j] = c0[j]; sv[32 + j] = c1[j]; }
        }
        const int *koff = key_off + kt * 128 + 64 * half;
        const int nvalid = N - kt * 128 - 64 * half;   // keys of this thread's 64 that exist
        // four partial maxima (short dependency chains), combined below
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (masked) {
            const int *kreg = key_region + kt * 128 + 64 * half;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float lv = fmaf(sv[j], scale, sbias[base - koff[j]]);
                sv[j] = kreg[j] == my_region ? lv : -INFINITY;
                mq[j & 3] = fmaxf(mq[j & 3], sv[j]);
            }
        } else if (nvalid >= 64) {
            // the common case: every key exists and no shift region cuts the window
#pragma unroll
            for (int j4 = 0; j4 < 16; ++j4) {
                const int4 o4 = reinterpret_cast<const int4 *>(koff)[j4];
                const int oo[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = 4 * j4 + i;
                    sv[j] = fmaf(sv[j], scale, sbias[base - oo[i]]);
                    mq[j & 3] = fmaxf(mq[j & 3], sv[j]);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const float lv = fmaf(sv[j], scale, sbias[base - koff[j]]);
                sv[j] = j < nvalid ? lv : -INFINITY;
                mq[j & 3] = fmaxf(mq[j & 3], sv[j]);
            }
        }
        float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        smax[half * 128 + row] = mt;
        if (__syncthreads_or(failed)) { failed = true; break; }
        mt = fmaxf(smax[row], smax[128 + row]);
        const float m_new = fmaxf(m_run, mt);
        // no key seen yet: 0 as the reference (every p is then 0, and alpha = 0
        // leaves o = 0 and l = 0 as they are)
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2_approx(m_run - m_use);
        float sq[4] = {0.f, 0.f, 0.f, 0.f};   // four partial sums
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
            const float p0 = ex2_approx(sv[j] - m_use), p1 = ex2_approx(sv[j + 1] - m_use);
            sq[(j >> 1) & 3] += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + ((sq[0] + sq[1]) + (sq[2] + sq[3]));   // this half's share of the row sum
        m_run = m_new;
        // P (bf16 pairs) over TMEM columns 32*half .. +31 (keys 64*half ..)
        {
            uint32_t lo[16], hi[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) { lo[i] = pk[i]; hi[i] = pk[16 + i]; }
            tmem_st16(t_lane + 32 * half, lo);
            tmem_st16(t_lane + 32 * half + 16, hi);
            tmem_wait_st();
        }
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
        tc_fence_after();
        // P.V in two halves over the tile's keys, issued by two threads (an MMA
        // costs its issuing thread the same whatever its size): keys 0..63 into
        // TMEM columns 128.., keys 64..127 into 160..; both commit to bar_pv
        if (tid == 0 || tid == 32) {
            const int kh = tid >> 5;
            const uint32_t id = idesc_bf16_bmn(128, 32);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                mma_bf16_ts(tmem + 128 + 32 * kh, tmem + 32 * kh + 8 * k,
                            desc_mnmajor_sw64(sV + b * (128 * 64) + 4096 * kh + 1024 * k, 128 * 64), id, k);
            mma_commit(bar_pv);
        }
        if (!mbar_wait(bar_pv, phase, st.wait_ns)) failed = true;
        phase ^= 1;
        tc_fence_after();
        float ot[16], ou[16];
        tmem_ld16(t_lane + 128 + 16 * half, ot);
        tmem_ld16(t_lane + 160 + 16 * half, ou);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = fmaf(o[e], alpha, ot[e] + ou[e]);
        // (no CTA barrier: the next tile's max exchange and P store barriers
        // order every reuse of TMEM and of the shared row maxima)
        tc_fence_before();
    }
    spart[half * 128 + row] = l_run;
    __syncthreads();
    if (!failed && row_ok) {
        const float l = spart[row] + spart[128 + row];
        const int64_t orow = a.o_token_order ? window_row_to_token(g, win * N + qt) : win * N + qt;
        store_o<16>(a.attn + orow * (int64_t)C + head * 32 + 16 * half, o, rcp_approx(l));
        // log2 of the normaliser: p = exp2(logit2 - lse) for the log2-scaled logits
        if (a.lse && half == 0) a.lse[(win * N + qt) * a.heads + head] = m_run + log2f(l);
    }
    if (failed && tid == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

} // namespace

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return encode;
}

// Tensor map over a row-major bf16 matrix [rows, cols]: boxes of 32 columns x
// box_rows rows, 64-byte swizzle, zero fill past the last row.
cudaError_t make_tensor_map_sw64(CUtensorMap *map, const void *ptr, int64_t rows, int cols, int box_rows,
                                 bool promote128)
{
    const EncodeTiledFn encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        promote128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map over a row-major bf16 matrix [rows, cols] with a row stride of
// ld elements (ld * 2 a multiple of 16): boxes of 64 columns x box_rows rows,
// 128-byte swizzle, zero fill past the last row or column.
cudaError_t make_tensor_map_sw128(CUtensorMap *map, const void *ptr, int64_t rows, int cols, int64_t ld, int box_rows)
{
    const EncodeTiledFn encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t elem[2] = {1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Tensor map over a bf16 image batch [rows, width, cols] (rows = B*H image
// rows, width = W tokens, cols = C channels, row-major): boxes of 32 channels
// x box_w tokens x box_h image rows, 64-byte swizzle, zero fill outside.
cudaError_t make_tensor_map_sw64_3d(CUtensorMap *map, const void *ptr, int64_t rows, int width, int cols, int box_w,
                                    int box_h)
{
    const EncodeTiledFn encode = encode_fn();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)width, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)width * cols * 2};
    const cuuint32_t box[3] = {32, (cuuint32_t)box_w, (cuuint32_t)box_h};
    const cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_attention(const AttnArgs &a, DeviceStatus st, cudaStream_t stream)
{
    const Geom &g = a.g;
    if (g.C != a.heads * 32) return cudaErrorInvalidValue;
    if (g.N <= 64) {
        return launch_attn_forward_tc(a.qkv, a.table, a.tau, a.heads, a.mode == 1 ? 1 : 0, g, a.attn, st, stream,
                                      a.overlap);
    } else if (attn_window_supported(g.M, a.heads)) {
        return launch_attn_window(a, st, stream);
    } else {
        const size_t smem = FlashSmem::bytes(g.M);
        cudaError_t e = cudaFuncSetAttribute(attn_flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        CUtensorMap tmap;
        // CTAs of one head run together (grid y = head): the neighbouring
        // head's 64 bytes of a row are read much later, so no 128-byte promotion
        e = make_tensor_map_sw64(&tmap, a.qkv, g.T, 3 * g.C, 128, false);
        if (e != cudaSuccess) return e;
        const int qtiles = (g.N + 127) / 128;
        dim3 grid((unsigned)(g.nwin * qtiles), (unsigned)a.heads);
        attn_flash_kernel<<<grid, FL_THREADS, smem, stream>>>(a, st, tmap);
    }
    return cudaGetLastError();
}

} // namespace swin
