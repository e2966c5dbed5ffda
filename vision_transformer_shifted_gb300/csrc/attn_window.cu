// Window attention for large windows (M = 12, 16, 20 or 24: N = M*M tokens
// per window, 32 channels per head), sm_103a tcgen05 + TMEM.
//
// Per window and head (pages "Boosting Swin Transformer Speed",
// Introduction and Training Optimization -- attention inside shifted
// windows; "Swin Transformer V2" (neura.market), How It Works -- relative
// position bias, scaled cosine attention with tau clipped at 0.01):
//   V1:  a_ij = q_i.k_j / sqrt(d) + table[idx(i,j), head]
//   V2:  a_ij = cos(q_i, k_j) / max(tau, 0.01) + table[idx(i,j), head]
//   a_ij = -inf when i, j lie in different shift regions (shift > 0)
//   o_i  = softmax_j(a_ij) . v_j
// idx(i,j) = (ri-rj+M-1)*(2M-1) + (ci-cj+M-1), query minus key, in-window
// coordinates; the mask and the index are computed, never loaded.  In V2 the
// QKV projection has already scaled q and k to unit length.
//
// A persistent CTA walks over units (head, window), head-major, so that a
// CTA's consecutive units mostly share a head and its relative-bias table.  A
// unit's k and v (all N keys, 64 bytes a row) come into shared memory once by
// TMA (two unit buffers: the next unit's keys load while this one's queries
// run) and serve all of the unit's query tiles of 128 rows.  The query tiles
// alternate between two groups of four compute warps (one thread per query
// row), so that one group's softmax overlaps the other group's MMAs.  Keys go
// in tiles of four window rows (4M keys: a multiple of 16, and whole window
// rows, so that the relative-bias offsets inside a tile are compile-time
// constants): per key tile, S = q k^T (128 x 4M x 32) into one of two TMEM
// buffers; an online softmax in fp32 (exp2, the running maximum and sum of a
// row in its thread's registers); P (bf16) back over the S columns; P.V (128
// x 32 x 4M, P read from TMEM as the A operand, v as an N-major B operand)
// into one of two 32-column buffers, added to the row's output one key tile
// later, while the next tile's softmax has already run.
// Warp roles: warp 0 loads (k, v of a unit; a q tile per group),
// warp 1 owns the TMEM allocation, warps 2 and 3 issue group 0's / group 1's
// MMAs, warps 4..7 and 8..11 compute.  Every wait is bounded.
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int AW_THREADS = 12 * 32;
constexpr int AW_CWARP0 = 4;
constexpr float AW_LOG2E = 1.4426950408889634f;

template <int M>
struct WinCfg {
    static constexpr int N = M * M;            // keys (and queries) of a window
    static constexpr int L = 2 * M - 1;
    static constexpr int KT = 4 * M;           // keys per key tile (four window rows)
    static constexpr int NKT = M / 4;          // key tiles per window
    static constexpr int QT = (N + 127) / 128; // query tiles per window
    static constexpr int KVB = N * 64;         // k (or v) of a unit: N rows of 32 bf16, SW64
    // bias table rows padded to BS floats, BS = M (mod 32): the bias loads of 32
    // consecutive queries (the lanes of a warp) then fall in 32 distinct banks
    static constexpr int BS = L + ((M - L) % 32 + 32) % 32;
    static constexpr int LL = L * BS;
    // shared memory: [2 units][k, v] KVB each; [2 groups][128][32] q tiles
    // (SW64); barriers; then every head's relative-bias table ([heads][L][BS]
    // f32, times log2(e))
    static constexpr int O_KV = 0;
    static constexpr int O_Q = O_KV + 4 * KVB;
    static constexpr int O_BARS = O_Q + 2 * 128 * 64;
    static constexpr int NBARS = 24;
    static constexpr int O_HEAD = O_BARS + NBARS * 8 + 16;    // [64] f32: per head, the fixed reference (or NaN)
    static constexpr int O_BIAS = O_HEAD + 64 * 4;
    static int bytes(int heads) { return O_BIAS + heads * LL * 4; }
    static_assert(M % 4 == 0 && KT % 16 == 0 && KT <= 128, "key tiles of four window rows");
    static_assert(2 * KT + 64 <= 256, "TMEM budget of a group");
};

// barriers
enum {
    AB_KVFULL = 0,   // + u: k, v of unit buffer u landed (TMA bytes)
    AB_KVFREE = 2,   // + u: both groups' MMAs on unit buffer u done (two commits)
    AB_QFULL = 4,    // + g: q tile of group g landed
    AB_QFREE = 6,    // + g: the S MMAs reading group g's q tile done
    AB_S = 8,        // + 8 g + r: S in buffer r done
    AB_P = 10,       // + 8 g + r: P in buffer r (compute warps)
    AB_PV = 12,      // + 8 g + r: P.V into buffer r done
    AB_PVC = 14      // + 8 g + r: P.V buffer r read (compute warps)
};

__device__ __forceinline__ bool aw_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
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

// The same from every lane of a warp, with a warp-uniform result.
__device__ __forceinline__ bool aw_warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
{
    const bool ok = aw_wait(bar, parity, limit_ns, abort);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void aw_arrive(uint32_t bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

__device__ __forceinline__ uint64_t aw_desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

__device__ __forceinline__ float aw_max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// x0 = x0 * m + b0, x1 = x1 * m + b1 (fma.rn.f32x2)
__device__ __forceinline__ void aw_ffma2(float &x0, float &x1, float m, float b0, float b1)
{
    asm("{\n\t.reg .b64 p, q, r;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\t"
        "mov.b64 r, {%3, %4};\n\tfma.rn.f32x2 p, p, q, r;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(m), "f"(b0), "f"(b1));
}

// x0 += b0, x1 += b1 (add.rn.f32x2)
__device__ __forceinline__ void aw_fadd2(float &x0, float &x1, float b0, float b1)
{
    asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
        "add.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(b0), "f"(b1));
}

// P = exp2(s - m) (SUB; s itself otherwise), bf16, two keys a column, into
// the KT/2 TMEM columns at taddr, 32 keys at a time; returns the sum of the p.
template <int KT, bool SUB>
__device__ __forceinline__ float aw_exp_store(float (&s)[KT], float m, uint32_t taddr)
{
    float sq0 = 0.f, sq1 = 0.f, sq2 = 0.f, sq3 = 0.f;
    const float nm = -m;
#pragma unroll
    for (int c0 = 0; c0 < KT; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int jj = c0; jj < c0 + 32 && jj < KT; jj += 2) {
            float d0 = s[jj], d1 = s[jj + 1];
            if (SUB) aw_fadd2(d0, d1, nm, nm);
            const float p0 = ex2_approx(d0), p1 = ex2_approx(d1);
            if ((jj >> 1) & 1)
                aw_fadd2(sq2, sq3, p0, p1);
            else
                aw_fadd2(sq0, sq1, p0, p1);
            pk[(jj - c0) >> 1] = pack_bf16x2(p0, p1);
        }
        if (c0 + 32 <= KT)
            tmem_st16(taddr + c0 / 2, pk);
        else
            tmem_st8(taddr + c0 / 2, *reinterpret_cast<uint32_t(*)[8]>(pk));
    }
    return (sq0 + sq1) + (sq2 + sq3);
}

// A unit (head-major): its head and window (b, wi, wj).
struct AwUnit {
    int64_t win;
    int head, wi, wj;
};

__device__ __forceinline__ AwUnit aw_unit(const Geom &g, int64_t u)
{
    AwUnit x;
    x.head = (int)(u / g.nwin);
    x.win = u - (int64_t)x.head * g.nwin;
    const int per = g.nh * g.nw;
    const int rem = (int)(x.win % per);
    x.wi = rem / g.nw;
    x.wj = rem - x.wi * g.nw;
    return x;
}

template <int M>
__global__ void __launch_bounds__(AW_THREADS, 1)
    attn_window_kernel(AttnArgs a, DeviceStatus st, const __grid_constant__ CUtensorMap tmap_q,
                       const __grid_constant__ CUtensorMap tmap_kv)
// tmap_q: qkv [T, 3C] bf16, boxes of 32 columns x 128 rows; tmap_kv: the same,
// boxes of 32 columns x 4M rows; both 64-byte swizzled
{
    using F = WinCfg<M>;
    constexpr int N = F::N, L = F::L, KT = F::KT, NKT = F::NKT, QT = F::QT, KVB = F::KVB, LL = F::LL, BS = F::BS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + F::O_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + F::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    float *sbias = reinterpret_cast<float *>(sm + F::O_BIAS);
    float *sref = reinterpret_cast<float *>(sm + F::O_HEAD);
    const Geom g = a.g;
    const int C = g.C;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);
    auto BAR = [&](int i) { return smem_u32(&bars[i]); };
    const int64_t nunits = g.nwin * a.heads;
    const int64_t my_units =
        nunits > (int64_t)blockIdx.x ? (nunits - 1 - (int64_t)blockIdx.x) / (int64_t)gridDim.x + 1 : 0;
    const int64_t my_qtiles = my_units * QT;   // the CTA's q tiles: lu * QT + qt, group = index % 2

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(AB_KVFULL + i), 1);
            mbar_init(BAR(AB_KVFREE + i), 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(BAR(AB_QFULL + i), 1);
            mbar_init(BAR(AB_QFREE + i), 1);
        }
        for (int grp = 0; grp < 2; ++grp)
            for (int r = 0; r < 2; ++r) {
                mbar_init(BAR(AB_S + 8 * grp + r), 1);
                mbar_init(BAR(AB_P + 8 * grp + r), 4);
                mbar_init(BAR(AB_PV + 8 * grp + r), 1);
                mbar_init(BAR(AB_PVC + 8 * grp + r), 4);
            }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    // every head's relative-bias table, times log2(e), once per CTA
    for (int i = tid; i < a.heads * LL; i += AW_THREADS) {
        const int hd = i / LL, e = i - hd * LL, dr = e / F::BS, dc = e - dr * F::BS;
        sbias[i] = dc < L ? __bfloat162float(a.table[(int64_t)(dr * L + dc) * a.heads + hd]) * AW_LOG2E : 0.f;
    }
    __syncthreads();
    // A fixed softmax reference per head where the logits are bounded.  In V2 a
    // logit (log2 units) is cos * sigma + bias with |cos| <= 1, sigma =
    // log2(e) / max(tau, 0.01): every logit of the head lies in [-sigma +
    // min(bias), sigma + max(bias)].  Softmax is the same for any common
    // shift of a row, so with the reference m = sigma + max(bias) every p =
    // exp2(logit - m) <= 1, and a row's largest p >= exp2(-(2 sigma + max -
    // min)).  When that span is at most 96 (p >= 2^-96, far inside the fp32
    // and bf16 range) the head skips the running maximum: its table holds
    // bias - m, p = exp2(s sigma + table) is one FMA and an exp2, and P.V
    // accumulates across the key tiles in TMEM with no rescaling.  Otherwise
    // (V1, whose q.k is unbounded, or a wide span) sref is NaN and the online
    // softmax runs.  One warp per head (a head count above the warp count
    // takes further rounds).
    for (int hd = warp; hd < a.heads; hd += AW_THREADS / 32) {
        const float *tb = sbias + hd * LL;
        float mx = -INFINITY, mn = INFINITY;
        for (int e = lane; e < LL; e += 32) {
            const int dc = e % BS;
            if (dc < L) {
                mx = fmaxf(mx, tb[e]);
                mn = fminf(mn, tb[e]);
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        }
        float ref = __int_as_float(0x7fc00000);   // NaN: online softmax
        if (a.mode == 1) {
            const float sigma = AW_LOG2E / fmaxf(a.tau[hd], 0.01f);
            if (2.f * sigma + (mx - mn) <= 96.f) ref = sigma + mx;
        }
        __syncwarp();
        if (ref == ref)
            for (int e = lane; e < LL; e += 32) sbias[hd * LL + e] -= ref;
        if (lane == 0) sref[hd] = ref;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // the prologue read only the tables and tau: q, k, v and the output wait
    // for the kernels queued before this one (a no-op unless launched to
    // overlap them)
    griddep_launch_dependents();
    griddep_wait();

    if (warp == 0) {
        // ===================== loads =====================
        if (lane == 0) {
            bool ok = true;
            int64_t qi = 0;   // q tiles loaded so far (CTA order)
#pragma unroll 1
            for (int64_t lu = 0; ok && lu < my_units; ++lu) {
                const AwUnit un = aw_unit(g, (int64_t)blockIdx.x + lu * gridDim.x);
                const int ub = (int)(lu & 1);
                // the unit buffer, once both groups are done with unit lu - 2
                if (lu >= 2 && !(ok = aw_wait(BAR(AB_KVFREE + ub), ((lu >> 1) - 1) & 1, st.wait_ns, abort_flag)))
                    break;
                const uint32_t kv = base + F::O_KV + ub * 2 * KVB;
                const int row0 = (int)(un.win * N);
                mbar_arrive_expect_tx(BAR(AB_KVFULL + ub), 2 * KVB);
#pragma unroll 1
                for (int kt = 0; kt < NKT; ++kt) {
                    tma_load_2d(kv + kt * KT * 64, &tmap_kv, C + un.head * 32, row0 + kt * KT, BAR(AB_KVFULL + ub));
                    tma_load_2d(kv + KVB + kt * KT * 64, &tmap_kv, 2 * C + un.head * 32, row0 + kt * KT,
                                BAR(AB_KVFULL + ub));
                }
#pragma unroll 1
                for (int qt = 0; qt < QT; ++qt, ++qi) {
                    const int grp = (int)(qi & 1);
                    const int64_t gi = qi >> 1;   // the group's q tile count
                    // the group's q buffer, once its previous q tile's S MMAs are done
                    if (gi >= 1 && !(ok = aw_wait(BAR(AB_QFREE + grp), (gi - 1) & 1, st.wait_ns, abort_flag))) break;
                    mbar_arrive_expect_tx(BAR(AB_QFULL + grp), 128 * 64);
                    tma_load_2d(base + F::O_Q + grp * (128 * 64), &tmap_q, un.head * 32, row0 + qt * 128,
                                BAR(AB_QFULL + grp));
                }
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (warp == 2 || warp == 3) {
        // ===================== MMA issuer of group warp - 2 =====================
        const int grp = warp - 2;
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, KT), id_pv = idesc_bf16_bmn(128, 32);
            const uint32_t tg = tmem + 256 * grp;
            bool ok = true;
            int64_t blk = 0;                // the group's key-tile blocks so far
            uint32_t ph_p = 0, ph_pvc = 0;  // bit r: phase of AB_P / AB_PVC + r
            uint32_t pending = 0;           // bit x: P.V buffer x holds a result not yet read
#pragma unroll 1
            for (int64_t qi = grp; ok && qi < my_qtiles; qi += 2) {
                const int64_t lu = qi / QT, gi = qi >> 1;
                const int qt = (int)(qi - lu * QT);
                const int ub = (int)(lu & 1);
                if (!(ok = aw_wait(BAR(AB_QFULL + grp), gi & 1, st.wait_ns, abort_flag))) break;
                if (!(ok = aw_wait(BAR(AB_KVFULL + ub), (lu >> 1) & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                const uint64_t dq = desc_kmajor_sw64(base + F::O_Q + grp * (128 * 64));
                const uint64_t dk = desc_kmajor_sw64(base + F::O_KV + ub * 2 * KVB);
                const uint64_t dv = desc_mnmajor_sw64(base + F::O_KV + ub * 2 * KVB + KVB, 8192);
                auto issue_s = [&](int kt, int r) {
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tg + KT * r, aw_desc_add(dq, 32 * ks), aw_desc_add(dk, kt * KT * 64 + 32 * ks), id_s,
                                 ks);
                    mma_commit(BAR(AB_S + 8 * grp + r));
                };
                issue_s(0, (int)(blk & 1));
                issue_s(1, (int)((blk + 1) & 1));
                if (NKT == 2) mma_commit(BAR(AB_QFREE + grp));   // the last S read q
                // (the group's last q tile of the unit: its P.V MMAs release the
                // unit buffer)
                const bool last_of_unit = qt + 2 >= QT;
                // fixed reference: P.V of every key tile into one buffer (the q tile's),
                // accumulated; online softmax: one buffer per key tile, alternating
                const float ref = sref[aw_unit(g, (int64_t)blockIdx.x + lu * gridDim.x).head];
                const bool fast = ref == ref;
#pragma unroll 1
                for (int kt = 0; kt < NKT; ++kt, ++blk) {
                    const int r = (int)(blk & 1);
                    if (!(ok = aw_wait(BAR(AB_P + 8 * grp + r), (ph_p >> r) & 1u, st.wait_ns, abort_flag))) break;
                    ph_p ^= 1u << r;
                    const int x = fast ? (int)(gi & 1) : r;   // P.V buffer
                    if ((!fast || kt == 0) && ((pending >> x) & 1u)) {   // its last result was read
                        if (!(ok = aw_wait(BAR(AB_PVC + 8 * grp + x), (ph_pvc >> x) & 1u, st.wait_ns, abort_flag)))
                            break;
                        ph_pvc ^= 1u << x;
                        pending &= ~(1u << x);
                    }
                    tc_fence_after();
                    // P.V over the tile's 4M keys: A = P from S buffer r's first KT/2
                    // columns, B = the tile's v rows (N-major), D = P.V buffer x
#pragma unroll
                    for (int kk = 0; kk < KT / 16; ++kk)
                        mma_bf16_ts(tg + 2 * KT + 32 * x, tg + KT * r + 8 * kk,
                                    aw_desc_add(dv, kt * KT * 64 + kk * 1024), id_pv, (fast && kt > 0) || kk > 0);
                    if (!fast || kt == NKT - 1) {
                        mma_commit(BAR(AB_PV + 8 * grp + x));
                        pending |= 1u << x;
                    }
                    // S of key tile kt + 2 into the same buffer (after this P.V in
                    // issue order, so P has been read)
                    if (kt + 2 < NKT) {
                        issue_s(kt + 2, r);
                        if (kt + 2 == NKT - 1) mma_commit(BAR(AB_QFREE + grp));
                    }
                }
                if (!ok) break;
                if (last_of_unit) mma_commit(BAR(AB_KVFREE + ub));
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (warp >= AW_CWARP0) {
        // ===================== compute: one thread per query row =====================
        const int grp = (warp - AW_CWARP0) >> 2, quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t tg = tmem + 256 * grp + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        int64_t blk = 0;
        uint32_t ph_s = 0, ph_pv = 0;   // bit r: phase of AB_S / AB_PV + r
#pragma unroll 1
        for (int64_t qi = grp; qi < my_qtiles; qi += 2) {
            const int64_t lu = qi / QT;
            const int qt = (int)(qi - lu * QT);
            const AwUnit un = aw_unit(g, (int64_t)blockIdx.x + lu * gridDim.x);
            // this row's query; rows past the window's N (last q tile) do no work
            const int qn = qt * 128 + row;
            const bool active = qt * 128 + quarter * 32 < N;   // (warp-uniform)
            const bool row_ok = qn < N;
            const int qr = row_ok ? qn / M : 0, qc = row_ok ? qn - (qn / M) * M : 0;
            const float scale = a.mode == 1 ? AW_LOG2E / fmaxf(a.tau[un.head], 0.01f) : AW_LOG2E * rsqrtf(32.0f);
            // shift regions: only windows on the last window row or column are cut
            // (warp-uniform: a unit is one window)
            const bool masked = g.s > 0 && (un.wi == g.nh - 1 || un.wj == g.nw - 1);
            const bool rowcut = masked && un.wi == g.nh - 1, q_hi = qr >= M - g.s;
            uint32_t colbits = (1u << M) - 1u;
            if (masked && un.wj == g.nw - 1) {
                const uint32_t lo = (1u << (M - g.s)) - 1u;
                colbits = qc >= M - g.s ? ((1u << M) - 1u) & ~lo : lo;
            }
            const float *bq = sbias + un.head * LL + (qr + M - 1) * BS + (qc + M - 1);
            const float ref = sref[un.head];
            const int64_t wrow = un.win * N + qn;
            // o / l -> bf16 -> attn (window order, or token order) and the log2
            // normaliser m + log2(l)
            auto store_o = [&](const float (&o)[32], float l, float m) {
                if (!row_ok) return;
                const int64_t orow = a.o_token_order ? window_row_to_token(g, wrow) : wrow;
                const float inv = rcp_approx(l);
                uint4 *dst = reinterpret_cast<uint4 *>(a.attn + orow * (int64_t)C + un.head * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    dst[c] = make_uint4(pack_bf16x2(o[8 * c] * inv, o[8 * c + 1] * inv),
                                        pack_bf16x2(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                        pack_bf16x2(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                        pack_bf16x2(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
                if (a.lse) a.lse[wrow * a.heads + un.head] = m + log2f(l);
            };
            // logits of key tile kt (log2 units, the table's bias added) in s:
            // key (4kt + rr, kj) reads bias row qr - 4kt - rr + M - 1, column
            // qc - kj + M - 1; keys of another shift region get -inf
            auto logits = [&](float (&s)[KT], int kt) {
                const float *bt = bq - 4 * kt * BS;
                if (!masked) {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                        for (int kj = 0; kj < M; kj += 2)
                            aw_ffma2(s[rr * M + kj], s[rr * M + kj + 1], scale, bt[-(rr * BS + kj)],
                                     bt[-(rr * BS + kj + 1)]);
                } else {
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) {
                        const bool rok = !rowcut || ((4 * kt + rr >= M - g.s) == q_hi);
                        const uint32_t cb = rok ? colbits : 0u;
#pragma unroll
                        for (int kj = 0; kj < M; kj += 2) {
                            const int jj = rr * M + kj;
                            aw_ffma2(s[jj], s[jj + 1], scale, bt[-(rr * BS + kj)], bt[-(rr * BS + kj + 1)]);
                            if (!((cb >> kj) & 1u)) s[jj] = -INFINITY;
                            if (!((cb >> (kj + 1)) & 1u)) s[jj + 1] = -INFINITY;
                        }
                    }
                }
            };
            auto load_s = [&](float (&s)[KT], int r) {
#pragma unroll
                for (int c = 0; c < KT / 32; ++c)
                    tmem_ld32(tg + KT * r + 32 * c, *reinterpret_cast<float(*)[32]>(s + 32 * c));
                if (KT % 32)
                    tmem_ld16(tg + KT * r + 32 * (KT / 32), *reinterpret_cast<float(*)[16]>(s + 32 * (KT / 32)));
                tmem_wait_ld();
            };
            if (ref == ref) {
                // ---- fixed reference (the table holds bias - ref): p = exp2(logit),
                // P.V accumulated in TMEM buffer gi & 1 ----
                float l_run = 0.f;
#pragma unroll 1
                for (int kt = 0; kt < NKT; ++kt, ++blk) {
                    const int r = (int)(blk & 1);
                    if (!(ok = aw_warp_wait(BAR(AB_S + 8 * grp + r), (ph_s >> r) & 1u, st.wait_ns, abort_flag))) break;
                    ph_s ^= 1u << r;
                    tc_fence_after();
                    if (active) {
                        float s[KT];
                        load_s(s, r);
                        logits(s, kt);
                        l_run += aw_exp_store<KT, false>(s, 0.f, tg + KT * r);
                        tmem_wait_st();
                    }
                    aw_arrive(BAR(AB_P + 8 * grp + r), lane);
                }
                if (!ok) break;
                const int x = (int)((qi >> 1) & 1);
                if (!(ok = aw_warp_wait(BAR(AB_PV + 8 * grp + x), (ph_pv >> x) & 1u, st.wait_ns, abort_flag))) break;
                ph_pv ^= 1u << x;
                tc_fence_after();
                if (active) {
                    float o[32];
                    tmem_ld32(tg + 2 * KT + 32 * x, o);
                    tmem_wait_ld();
                    store_o(o, l_run, ref);
                }
                aw_arrive(BAR(AB_PVC + 8 * grp + x), lane);
                continue;
            }
            // ---- online softmax: running maximum, one P.V buffer per key tile ----
            float m_run = -INFINITY, l_run = 0.f, a_hold = 0.f;
            float o[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
            // the P.V of block b into o (o in the reference of the block before
            // b, moved to b's by the factor f)
            auto add_pv = [&](int64_t b, float f) -> bool {
                const int rp = (int)(b & 1);
                if (!aw_warp_wait(BAR(AB_PV + 8 * grp + rp), (ph_pv >> rp) & 1u, st.wait_ns, abort_flag)) return false;
                ph_pv ^= 1u << rp;
                tc_fence_after();
                if (active) {
                    float pv[32];
                    tmem_ld32(tg + 2 * KT + 32 * rp, pv);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = fmaf(o[e], f, pv[e]);
                }
                aw_arrive(BAR(AB_PVC + 8 * grp + rp), lane);
                return true;
            };
#pragma unroll 1
            for (int kt = 0; kt < NKT; ++kt, ++blk) {
                const int r = (int)(blk & 1);
                if (!(ok = aw_warp_wait(BAR(AB_S + 8 * grp + r), (ph_s >> r) & 1u, st.wait_ns, abort_flag))) break;
                ph_s ^= 1u << r;
                tc_fence_after();
                float alpha = 0.f;
                if (active) {
                    float s[KT];
                    load_s(s, r);
                    logits(s, kt);
                    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int jj = 0; jj < KT; jj += 2) mq[(jj >> 1) & 3] = aw_max3(mq[(jj >> 1) & 3], s[jj], s[jj + 1]);
                    const float m_new = fmaxf(m_run, fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])));
                    // no key seen yet: 0 as the reference (every p is then 0, and the
                    // factor 0 leaves o = 0 and l = 0 as they are)
                    const float m_use = m_new == -INFINITY ? 0.f : m_new;
                    alpha = ex2_approx(m_run - m_use);
                    const float sum = aw_exp_store<KT, true>(s, m_use, tg + KT * r);
                    l_run = l_run * alpha + sum;
                    m_run = m_new;
                    tmem_wait_st();
                }
                aw_arrive(BAR(AB_P + 8 * grp + r), lane);
                // the previous key tile's P.V (in the reference of the previous
                // maximum; o, holding the tiles before it, moves there by that tile's
                // factor)
                if (kt > 0 && !(ok = add_pv(blk - 1, a_hold))) break;
                a_hold = alpha;
            }
            if (!ok) break;
            if (!(ok = add_pv(blk - 1, a_hold))) break;
            if (active) store_o(o, l_run, m_run);
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

int aw_num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    }
    return n;
}

template <int M>
cudaError_t launch_window_t(const AttnArgs &a, DeviceStatus st, cudaStream_t stream)
{
    using F = WinCfg<M>;
    const size_t smem = (size_t)F::bytes(a.heads) + 1024;
    if (smem > 232448) return cudaErrorInvalidConfiguration;
    auto kern = attn_window_kernel<M>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tq, tkv;
    e = make_tensor_map_sw64(&tq, a.qkv, a.g.T, 3 * a.g.C, 128, false);
    if (e != cudaSuccess) return e;
    e = make_tensor_map_sw64(&tkv, a.qkv, a.g.T, 3 * a.g.C, F::KT, false);
    if (e != cudaSuccess) return e;
    const int64_t units = a.g.nwin * a.heads;
    const int grid = (int)(units < aw_num_sms() ? units : aw_num_sms());
    e = launch_maybe_overlapped(kern, dim3(grid), dim3(AW_THREADS), smem, stream, a.overlap, a, st, tq, tkv);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace

bool attn_window_supported(int M, int heads)
{
    if (!(M == 12 || M == 16 || M == 20 || M == 24)) return false;
    const int N = M * M, L = 2 * M - 1, BS = L + ((M - L) % 32 + 32) % 32;
    return heads <= 64 && 4 * N * 64 + 2 * 128 * 64 + 24 * 8 + 16 + 64 * 4 + heads * L * BS * 4 + 1024 <= 232448;
}

cudaError_t launch_attn_window(const AttnArgs &a, DeviceStatus st, cudaStream_t stream)
{
    switch (a.g.M) {
    case 12: return launch_window_t<12>(a, st, stream);
    case 16: return launch_window_t<16>(a, st, stream);
    case 20: return launch_window_t<20>(a, st, stream);
    case 24: return launch_window_t<24>(a, st, stream);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace swin
