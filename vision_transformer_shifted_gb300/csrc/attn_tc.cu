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
// the fp32 P.V result.
//
// Small windows (N <= 64, e.g. M = 7 or 8): one CTA takes two windows of one
// head; window A fills rows 0..63 and window B rows 64..127 of a 128-row MMA
// tile, so QK^T is one 128x128x32 MMA whose off-diagonal blocks are ignored,
// and P.V is one 128x32x128 MMA with P zero outside each row's own window.
// Large windows (N > 64, e.g. M = 24, N = 576): one CTA takes 128 queries of
// one window and head and walks the keys in tiles of 128 with an online
// softmax, accumulating o in registers.
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int THREADS = 128;
constexpr float LOG2E = 1.4426950408889634f;

// Shared memory: Q and K tiles as 128 rows x 128 B (first 64 B = d 32 used),
// V^T as 32 rows x 128 keys (two 64-key K blocks), P as 128 rows x 128 keys
// (two K blocks), all K-major 128B-swizzled.
struct AttnSmem {
    static constexpr int q_off = 0;
    static constexpr int k_off = q_off + 128 * 128;
    static constexpr int vt_off = k_off + 128 * 128;
    static constexpr int p_off = vt_off + 2 * 32 * 128;
    static constexpr int end = p_off + 2 * 128 * 128;
    static size_t bytes(int M) { return 1024 + end + (size_t)(2 * M - 1) * (2 * M - 1) * 4 + 128 * 8 + 64; }
};

// Loads one 32-wide head slice (64 bytes) of a qkv row.
__device__ __forceinline__ void load_head_row(const bf16 *src, bool valid, uint4 (&v)[4])
{
    if (valid) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = s4[i];
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = make_uint4(0, 0, 0, 0);
    }
}

// V2: scales a 32-element bf16 row to unit L2 norm (norm clamped at 1e-12)
// in fp32 and rounds it back to bf16.
__device__ __forceinline__ void l2_normalise(uint4 (&v)[4])
{
    float f[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 p = unpack_bf16x2(w[j]);
            f[8 * i + 2 * j] = p.x;
            f[8 * i + 2 * j + 1] = p.y;
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) ss = fmaf(f[i], f[i], ss);
    const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i].x = pack_bf16x2(f[8 * i + 0] * inv, f[8 * i + 1] * inv);
        v[i].y = pack_bf16x2(f[8 * i + 2] * inv, f[8 * i + 3] * inv);
        v[i].z = pack_bf16x2(f[8 * i + 4] * inv, f[8 * i + 5] * inv);
        v[i].w = pack_bf16x2(f[8 * i + 6] * inv, f[8 * i + 7] * inv);
    }
}

// Writes a 32-element row (4 x 16 B) into row `row` of a 128B-swizzled tile.
__device__ __forceinline__ void store_row_sw128(uint8_t *tile, int row, const uint4 (&v)[4])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4 *>(tile + sw128_offset(row, c)) = v[c];
}

// Writes v (32 elements of key `key`, 0..127) as column `key` of V^T
// (32 rows e x 128 keys, two 64-key K blocks of 32 x 128 B).
__device__ __forceinline__ void store_vt_column(uint8_t *vt, int key, const uint4 (&v)[4])
{
    uint8_t *blk = vt + (key >> 6) * (32 * 128);
    const int kk = key & 63;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e0 = 8 * i + 2 * j;
            *reinterpret_cast<uint16_t *>(blk + sw128_offset(e0, kk >> 3) + (kk & 7) * 2) = (uint16_t)(w[j] & 0xFFFF);
            *reinterpret_cast<uint16_t *>(blk + sw128_offset(e0 + 1, kk >> 3) + (kk & 7) * 2) = (uint16_t)(w[j] >> 16);
        }
    }
}

// Writes 64 probabilities (bf16-packed in pairs) as the 64-key K block `kb`
// of row `row` of the P tile.
__device__ __forceinline__ void store_p_block(uint8_t *ptile, int row, int kb, const uint32_t (&pk)[32])
{
    uint8_t *blk = ptile + kb * (128 * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
}

__device__ __forceinline__ void zero_p_block(uint8_t *ptile, int row, int kb)
{
    uint8_t *blk = ptile + kb * (128 * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(blk + sw128_offset(row, c)) = make_uint4(0, 0, 0, 0);
}

// Region id (row band * 3 + column band) of in-window token (ti, tj) of
// window (wi, wj); 0 everywhere when shift == 0.
__device__ __forceinline__ int token_region(const Geom &g, int wi, int wj, int ti, int tj)
{
    if (g.s == 0) return 0;
    return 3 * shift_band(wi * g.M + ti, g.H, g.M, g.s) + shift_band(wj * g.M + tj, g.W, g.M, g.s);
}

// Stores an o row (32 fp32 scaled by inv_l) as bf16 to attn.
__device__ __forceinline__ void store_o_row(bf16 *dst, const float (&o)[32], float inv_l)
{
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 u;
        u.x = pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l);
        u.y = pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l);
        u.z = pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l);
        u.w = pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l);
        d4[q] = u;
    }
}

struct KernelCommon {
    uint8_t *smem;
    float *sbias;
    uint64_t *bar;
    uint32_t *tmem_slot;
};

__device__ __forceinline__ KernelCommon setup_smem(uint8_t *smem_raw, int M)
{
    KernelCommon k;
    k.smem = smem_align(smem_raw, 1024);
    k.sbias = reinterpret_cast<float *>(k.smem + AttnSmem::end);
    const int L2 = (2 * M - 1) * (2 * M - 1);
    uint8_t *after = reinterpret_cast<uint8_t *>(k.sbias + L2);
    after = smem_align(after, 8);
    k.bar = reinterpret_cast<uint64_t *>(after);
    k.tmem_slot = reinterpret_cast<uint32_t *>(k.bar + 1);
    return k;
}

// ---------------------------------------------------------------------------
// Two windows per CTA, N <= 64.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS) attn_pack2_kernel(AttnArgs a, DeviceStatus st)
{
    extern __shared__ uint8_t smem_raw[];
    const Geom g = a.g;
    const int M = g.M, N = g.N, C = g.C, L = 2 * M - 1;
    KernelCommon kc = setup_smem(smem_raw, M);
    uint8_t *sQ = kc.smem + AttnSmem::q_off;
    uint8_t *sK = kc.smem + AttnSmem::k_off;
    uint8_t *sVt = kc.smem + AttnSmem::vt_off;
    uint8_t *sP = kc.smem + AttnSmem::p_off;
    __shared__ int8_t key_region[2][64];
    __shared__ int16_t key_off[64];

    const int tid = threadIdx.x, warp = tid >> 5;
    const int head = blockIdx.y;
    const int slot = tid >> 6, t = tid & 63;
    const int64_t win = 2 * (int64_t)blockIdx.x + slot;
    const bool win_ok = win < g.nwin;
    const bool row_ok = win_ok && t < N;
    const int per = g.nh * g.nw;
    const int rem = win_ok ? (int)(win % per) : 0;
    const int wi = rem / g.nw, wj = rem % g.nw;
    const int ti = t / M, tj = t % M;

    // bias column of this head, times log2(e)
    for (int i = tid; i < L * L; i += THREADS) kc.sbias[i] = __bfloat162float(a.table[(int64_t)i * a.heads + head]) * LOG2E;
    // this thread's token as a key: its region in its window (-1 for padding), its offset
    key_region[slot][t] = (int8_t)(t < N ? token_region(g, wi, wj, ti, tj) : -1);
    if (slot == 0) key_off[t] = (int16_t)(ti * L + tj);
    if (tid == 0) {
        mbar_init(smem_u32(kc.bar), 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(kc.tmem_slot), 128);
        tmem_relinquish();
    }

    // q, k, v rows of this thread's token (zeros for padding rows)
    {
        const bf16 *base = a.qkv + ((win_ok ? win : 0) * N + (t < N ? t : 0)) * (int64_t)(3 * C) + head * 32;
        uint4 q[4], k[4], v[4];
        load_head_row(base, row_ok, q);
        load_head_row(base + C, row_ok, k);
        load_head_row(base + 2 * C, row_ok, v);
        if (a.mode == 1 && row_ok) {
            l2_normalise(q);
            l2_normalise(k);
        }
        store_row_sw128(sQ, tid, q);
        store_row_sw128(sK, tid, k);
        store_vt_column(sVt, tid, v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *kc.tmem_slot;
    const uint32_t bar = smem_u32(kc.bar);

    if (tid == 0) {
        const uint32_t id = idesc_bf16(128, 128);
#pragma unroll
        for (int k = 0; k < 2; ++k)
            mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sQ) + 32 * k), desc_kmajor_sw128(smem_u32(sK) + 32 * k), id, k);
        mma_commit(bar);
    }
    bool failed = !mbar_wait(bar, 0, st.wait_ns);
    tc_fence_after();

    // ---- softmax of this thread's row over its own window's 64 key columns ----
    float scale;
    if (a.mode == 1) scale = LOG2E / fmaxf(a.tau[head], 0.01f);
    else scale = LOG2E * rsqrtf(32.0f);
    float l = 1.f;
    {
        float s[64];
        const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(slot * 64);
        {
            float c0[32], c1[32];
            tmem_ld32(t_row, c0);
            tmem_ld32(t_row + 32, c1);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) { s[j] = c0[j]; s[32 + j] = c1[j]; }
        }
        const int my_region = key_region[slot][t];   // -1 for a padding row: nothing matches
        const int tb = row_ok ? t : 0;                 // padding rows read a valid bias row
        const int base = (tb / M + M - 1) * L + (tb % M + M - 1);
        float mx = -INFINITY;
        // branch-free over the lanes: every lane computes the logit and a select
        // applies the mask (j < N is the same for the whole warp)
#pragma unroll
        for (int j = 0; j < 64; ++j) {
            float v = -INFINITY;
            if (j < N) {
                const float lv = fmaf(s[j], scale, kc.sbias[base - key_off[j]]);
                v = key_region[slot][j] == my_region ? lv : -INFINITY;
            }
            s[j] = v;
            mx = fmaxf(mx, v);
        }
        if (!row_ok) mx = 0.f;
        float sum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 64; j += 2) {
            const float p0 = ex2_approx(s[j] - mx), p1 = ex2_approx(s[j + 1] - mx);
            sum += p0 + p1;
            pk[j / 2] = pack_bf16x2(p0, p1);
        }
        l = sum;
        if (row_ok) store_p_block(sP, tid, slot, pk);
        else zero_p_block(sP, tid, slot);
        zero_p_block(sP, tid, slot ^ 1);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(failed)) failed = true;
    tc_fence_after();

    if (!failed) {
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int kb = k >> 2, ks = k & 3;
                mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sP) + kb * 16384 + 32 * ks),
                         desc_kmajor_sw128(smem_u32(sVt) + kb * 4096 + 32 * ks), id, k);
            }
            mma_commit(bar);
        }
        failed = !mbar_wait(bar, 1, st.wait_ns);
        tc_fence_after();
        float o[32];
        tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), o);
        tmem_wait_ld();
        if (row_ok && !failed) store_o_row(a.attn + (win * N + t) * (int64_t)C + head * 32, o, rcp_approx(l));
    }
    if (failed) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// Large windows: 128 queries per CTA, keys in tiles of 128, online softmax.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS) attn_flash_kernel(AttnArgs a, DeviceStatus st)
{
    extern __shared__ uint8_t smem_raw[];
    const Geom g = a.g;
    const int M = g.M, N = g.N, C = g.C, L = 2 * M - 1;
    KernelCommon kc = setup_smem(smem_raw, M);
    uint8_t *sQ = kc.smem + AttnSmem::q_off;
    uint8_t *sK = kc.smem + AttnSmem::k_off;
    uint8_t *sVt = kc.smem + AttnSmem::vt_off;
    uint8_t *sP = kc.smem + AttnSmem::p_off;
    __shared__ int key_region[128];
    __shared__ int key_off[128];

    const int tid = threadIdx.x, warp = tid >> 5;
    const int head = blockIdx.y;
    const int qtiles = (N + 127) / 128;
    const int64_t win = blockIdx.x / qtiles;
    const int q0 = (blockIdx.x % qtiles) * 128;
    const int per = g.nh * g.nw;
    const int rem = (int)(win % per);
    const int wi = rem / g.nw, wj = rem % g.nw;
    const int qt = q0 + tid;
    const bool row_ok = qt < N;
    const int qi = row_ok ? qt / M : 0, qj = row_ok ? qt % M : 0;
    const int my_region = token_region(g, wi, wj, qi, qj);
    const int base = (qi + M - 1) * L + (qj + M - 1);
    const bf16 *wbase = a.qkv + win * N * (int64_t)(3 * C) + head * 32;

    for (int i = tid; i < L * L; i += THREADS) kc.sbias[i] = __bfloat162float(a.table[(int64_t)i * a.heads + head]) * LOG2E;
    if (tid == 0) {
        mbar_init(smem_u32(kc.bar), 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(kc.tmem_slot), 256);
        tmem_relinquish();
    }
    {
        uint4 q[4];
        load_head_row(wbase + (int64_t)(row_ok ? qt : 0) * (3 * C), row_ok, q);
        if (a.mode == 1 && row_ok) l2_normalise(q);
        store_row_sw128(sQ, tid, q);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *kc.tmem_slot;
    const uint32_t bar = smem_u32(kc.bar);
    const uint32_t t_lane = tmem + ((uint32_t)(warp * 32) << 16);

    float scale;
    if (a.mode == 1) scale = LOG2E / fmaxf(a.tau[head], 0.01f);
    else scale = LOG2E * rsqrtf(32.0f);

    float o[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    bool failed = false;
    uint32_t phase = 0;
    const int ktiles = (N + 127) / 128;

#pragma unroll 1
    for (int kt = 0; kt < ktiles; ++kt) {
        // K and V rows of key kt*128 + tid; the previous tile's MMAs have
        // completed (awaited before its o update)
        const int kj = kt * 128 + tid;
        const bool kok = kj < N;
        {
            const bf16 *src = wbase + (int64_t)(kok ? kj : 0) * (3 * C);
            uint4 k[4], v[4];
            load_head_row(src + C, kok, k);
            load_head_row(src + 2 * C, kok, v);
            if (a.mode == 1 && kok) l2_normalise(k);
            store_row_sw128(sK, tid, k);
            store_vt_column(sVt, tid, v);
            key_region[tid] = kok ? token_region(g, wi, wj, kj / M, kj % M) : -1;
            key_off[tid] = kok ? (kj / M) * L + (kj % M) : 0;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
        tc_fence_after();
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 128);
#pragma unroll
            for (int k = 0; k < 2; ++k)
                mma_bf16(tmem, desc_kmajor_sw128(smem_u32(sQ) + 32 * k), desc_kmajor_sw128(smem_u32(sK) + 32 * k), id, k);
            mma_commit(bar);
        }
        if (!mbar_wait(bar, phase, st.wait_ns)) failed = true;
        phase ^= 1;
        tc_fence_after();

        // logits of the tile's 128 keys in registers; mask by select, not by branch
        float sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float s[32];
            tmem_ld32(t_lane + 32 * c, s);
#pragma unroll
            for (int j = 0; j < 32; ++j) sv[32 * c + j] = s[j];
        }
        tmem_wait_ld();
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; ++j) {
            const float lv = fmaf(sv[j], scale, kc.sbias[base - key_off[j]]);
            sv[j] = key_region[j] == my_region ? lv : -INFINITY;
            mt = fmaxf(mt, sv[j]);
        }
        const float m_new = fmaxf(m_run, mt);
        // no key seen yet: use 0 as the reference (every p below is then 0, and
        // alpha = 0 leaves o = 0, l = 0 as they are)
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2_approx(m_run - m_use);
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
                const float p0 = ex2_approx(sv[32 * c + j] - m_use), p1 = ex2_approx(sv[32 * c + j + 1] - m_use);
                sum += p0 + p1;
                pk[j / 2] = pack_bf16x2(p0, p1);
            }
            // chunk c holds keys 32c..32c+31: K block c/2, 16-byte chunks 4*(c%2)..+3
            uint8_t *blk = sP + (c >> 1) * (128 * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4 *>(blk + sw128_offset(tid, 4 * (c & 1) + q)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
        tc_fence_after();
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 32);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int kb = k >> 2, ks = k & 3;
                mma_bf16(tmem + 128, desc_kmajor_sw128(smem_u32(sP) + kb * 16384 + 32 * ks),
                         desc_kmajor_sw128(smem_u32(sVt) + kb * 4096 + 32 * ks), id, k);
            }
            mma_commit(bar);
        }
        if (!mbar_wait(bar, phase, st.wait_ns)) failed = true;
        phase ^= 1;
        tc_fence_after();
        float ot[32];
        tmem_ld32(t_lane + 128, ot);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = fmaf(o[e], alpha, ot[e]);
        tc_fence_before();
        if (__syncthreads_or(failed)) { failed = true; break; }
    }
    if (!failed && row_ok) store_o_row(a.attn + (win * N + qt) * (int64_t)C + head * 32, o, rcp_approx(l_run));
    if (failed && tid == 0) atomicOr(st.err, ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

} // namespace

cudaError_t launch_attention(const AttnArgs &a, DeviceStatus st, cudaStream_t stream)
{
    const Geom &g = a.g;
    if (g.C != a.heads * 32) return cudaErrorInvalidValue;
    const size_t smem = AttnSmem::bytes(g.M);
    if (g.N <= 64) {
        cudaError_t e = cudaFuncSetAttribute(attn_pack2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        dim3 grid((unsigned)((g.nwin + 1) / 2), (unsigned)a.heads);
        attn_pack2_kernel<<<grid, THREADS, smem, stream>>>(a, st);
    } else {
        cudaError_t e = cudaFuncSetAttribute(attn_flash_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const int qtiles = (g.N + 127) / 128;
        dim3 grid((unsigned)(g.nwin * qtiles), (unsigned)a.heads);
        attn_flash_kernel<<<grid, THREADS, smem, stream>>>(a, st);
    }
    return cudaGetLastError();
}

} // namespace swin
