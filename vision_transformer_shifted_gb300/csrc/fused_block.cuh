// The whole shifted-window attention block in one persistent kernel
// (sm_103a, tcgen05 + TMEM), for windows of at most 64 tokens (M = 7, 8) and
// C = 64, 96 or 128 channels (2, 3 or 4 heads of 32).
//
// Steps, per tile of two windows (pages "Boosting Swin Transformer Speed",
// Introduction / Training Optimization / Inference Optimization; "Swin
// Transformer V2" (neura.market), How It Works):
//   S1  the tile's two windows are gathered from x through the cyclic shift
//       by -s and the window partition: window A fills rows 0..63 of a
//       128-row tile, window B rows 64..127, token (ti, tj) of a window at
//       row 8*ti + tj; a window arrives as one 3-D TMA box (M image rows x 8
//       tokens x 32 channels) per 32 channels.  Windows that the shift wraps
//       around the image edge (last window row or column) are gathered with
//       cp.async instead
//   S2  [q|k] = X Wqk^T (128 x 2C) and v = X Wv^T (128 x C) on tcgen05 into
//       TMEM; the bias added (V2: q and k scaled to unit length) while they
//       are drained to shared memory as bf16
//   S3-S5 per head: S = q k^T, block-diagonal: two MMAs (128 x 64 x 32), one
//       per window, write the same 64 columns, each kept to its window's rows
//       by the MMA's output-lane mask; one thread per row applies the scale,
//       the relative bias and the shift mask (computed from the window's
//       coordinates) and the softmax (fp32, exp2); P (bf16) goes back into
//       TMEM over the S columns
//   S6  o_h = P v_h, again one lane-masked MMA pair (128 x 32 x 64), P read
//       from TMEM as the A operand, o_h written over the upper half of the
//       same S columns; scaled by 1/rowsum and staged as bf16
//   S7  y = o Wproj^T on tcgen05
//   S8  y + bproj staged in shared memory (token (ti, tj) at row M*ti + tj)
//       and written through the window reverse + roll(+s) map into
//       out[B, H, W, C]: one 3-D TMA store (M x M tokens x 32 channels) per
//       window and 32 channels, plain stores for wrapping windows
// Nothing but x, the weights and out touches HBM.
//
// Two tiles in flight.  The CTA's tiles alternate between two groups of four
// compute warps (group g takes the CTA's tiles j = g, g + 2, ...): while one
// group runs the softmax of its tile, the tensor cores serve the other's
// MMAs.  Warp w of a group owns TMEM lane quarter w % 4, and each of its
// threads one tile row, so a row's softmax needs no exchange between threads.
// Warp roles:
//   warp 0      producer: x gathers into X(g) (TMA; cp.async for wrapping
//               windows)
//   warp 1      tcgen05 issuer of every QKV MMA; owns TMEM
//   warps 2, 3  tcgen05 issuers of group 0's / group 1's S, P.V and
//               projection MMAs; they also issue the group's output stores
//   warps 4..7, 8..11  compute groups 0 and 1
// TMEM (512 columns): [0, 2C) q|k of the tile whose QKV ran last (the groups
// take turns), then 128 columns per group: v of its tile; then its two
// 64-column S buffers (heads alternate between them; P over the first 32
// columns, o_h over the last 32); then y.
// Shared memory: the weights once per CTA (64B-swizzled K-major), and per
// group X(g) (its tile's x; once the QKV MMAs have read it, the same bytes
// hold q), K(g) (k of each head) and V(g) (v of each head, the N-major B
// operand of P.V; then o, the projection's A operand; then the staged output
// rows).  C = 128 leaves room for one tile in flight only (the weights take
// 128 KB), so there the two groups split each tile's heads instead (group g:
// heads 2g, 2g + 1, with issuer warp 2 + g and its own S buffers in the
// second 128 TMEM columns of the pair; group 0 also drains v, and each group
// drains half of y).  k goes into X once the QKV MMAs have read x, and q is
// written back into TMEM as bf16 over its own fp32 columns, from where the S
// MMAs read it as their A operand.
// All hand-offs are mbarriers: "ready" barriers get one arrival per
// compute warp of the group, "done" barriers are tcgen05.commit targets.
// Every wait is bounded: a timeout sets the error word, and every role
// leaves at its next wait.
#pragma once
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

struct FusedArgs {
    const bf16 *x, *Wqkv, *bqkv, *table, *Wproj, *bproj;
    const float *tau;
    bf16 *out;
    int mode;
    Geom g;
    int *sched;         // [2] zero before the launch: next tile to hand out, CTAs done
    // The transformer block's LayerNorm and residual folded in: fold 0 = the
    // attention output alone; 1 = pre-norm (V1): attention of LN(x), out =
    // x + that; 2 = residual post-norm (V2): out = x + LN(attention of x).
    // (The kernel takes it as its FOLD parameter.)
    const bf16 *ln_g, *ln_b;
    int fold;
    // (host side) launched with programmatic stream serialization: the kernel's
    // prologue (weights, biases, tables) may run while the kernels queued
    // before it finish; everything after it waits for them
    int overlap;
};

// The folded variants (fold 1, 2), built in their own translation unit.
cudaError_t launch_fused_folded(const FusedArgs &a, DeviceStatus st, cudaStream_t stream);

namespace {

constexpr int PWARP = 0;      // producer
constexpr int QWARP = 1;      // QKV issuer, TMEM owner
constexpr int AWARP0 = 2;     // attention and projection issuers: warp 2 + group
constexpr int CWARP0 = 4;     // compute warps: 4 + 4 * group + quarter
constexpr int GWARPS = 4;     // compute warps per group
constexpr int FTHREADS = 12 * 32;
constexpr float FLOG2E = 1.4426950408889634f;

// G = 2: two tiles in flight (C = 64, 96): per group X(g) (x, then q), K(g)
// and V(g) in shared memory.  G = 1 (C = 128, whose resident weights leave
// shared memory for one tile only): the two compute groups split the tile's
// heads, q goes back into TMEM (bf16, over its own fp32 columns: the A
// operand of S), k into X once the QKV MMAs have read x, and there is no K.
template <int M, int C, int G>
struct FusedCfg {
    static constexpr int HEADS = C / 32;
    static constexpr int L = 2 * M - 1;
    static constexpr int KB = C / 32;          // 32-channel K blocks (64-byte swizzle)
    static constexpr int HT = 128 * 64;        // one [128 rows][32 channels] SW64 tile
    static constexpr bool SPLIT = G == 1;                 // one tile, heads split over the groups
    static constexpr int HPG = SPLIT ? HEADS / 2 : HEADS;  // heads per compute group
    static constexpr int TW = (SPLIT ? 2 : 1) * 4;         // warps arriving on a tile barrier
    // shared memory (bytes); SW64 tiles are 512-aligned
    static constexpr int WQK = 0;                       // [2C rows][C]
    static constexpr int WV = WQK + 2 * C * C * 2;      // [C rows][C]
    static constexpr int WP = WV + C * C * 2;           // [C rows][C]
    static constexpr int XT = WP + C * C * 2;           // X(g) = XT + g * KB * HT
    static constexpr int KT = XT + G * KB * HT;         // K(g) (G = 2)
    static constexpr int VT = KT + (SPLIT ? 0 : G * KB * HT);    // V(g)
    static constexpr int SMALL = VT + G * KB * HT;
    static constexpr int O_BQKV = 0;                          // [3C] f32
    static constexpr int O_BPROJ = O_BQKV + 3 * C * 4;        // [C] f32
    static constexpr int O_SCALE = O_BPROJ + C * 4;           // [4] f32
    // relative-bias table rows padded to LP floats: a warp's 32 rows span four
    // window rows ti, whose reads (LP ti + tj, tj < 8) then fall in four
    // distinct 8-bank groups (LP = 24 = -8 mod 32)
    static constexpr int LP = 24;
    static_assert(L <= LP, "bias row padding");
    static constexpr int O_REF = O_SCALE + 16;                // [4] f32: fixed softmax reference, or NaN
    static constexpr int O_BIAS = O_REF + 16;                 // [HEADS][L][LP] f32, times log2(e)
    static constexpr int O_LN = (O_BIAS + HEADS * L * LP * 4 + 15) / 16 * 16;   // [2][C] f32: LayerNorm gamma, beta
    static constexpr int O_CSUM = O_LN + 2 * C * 4;           // [3C] f32: column sums of the scaled Wqkv
    static constexpr int O_RING = O_CSUM + 3 * C * 4;         // [4] int: tile of the CTA's j-th tile (j mod 4)
    static constexpr int O_BARS = O_RING + 16;
    static constexpr int NBARS = 2 * 21 + 1;
    static constexpr int O_END = O_BARS + NBARS * 8 + 16;
    static constexpr int BYTES = SMALL + O_END;
    // TMEM columns
    static constexpr int T_QK = 0;                      // [0, 2C): q of head h at 32h, k at C + 32h
    static constexpr int T_R0 = 2 * C;                  // group g's 128 columns at T_R0 + 128 g
    static_assert(T_R0 + 256 <= 512, "TMEM budget");
    static_assert(G == 1 || G == 2, "one or two tiles in flight");
    static_assert(!SPLIT || HEADS % 2 == 0, "the groups split the heads evenly");
    static_assert(C <= 128, "v and y fit the group's 128 columns");
    static_assert(M <= 8, "two windows of 8-row-aligned window rows per 128-row tile");
    static_assert(BYTES + 1024 <= 232448, "shared memory budget");
};

// Barriers: group g's at 21 g + ..., and one shared by the groups.
enum {
    // (G = 1: the tile barriers -- X, XFREE, QKV, O, Y, RFREE, STAGE, VFREE --
    // are group 0's, and O, RFREE, STAGE and QKFREE take both groups' warps)
    BR_X = 0,       // x of the group's tile landed in X(g) (TMA bytes + producer arrival)
    BR_XFREE = 1,   // the group's last S MMA of its tile done: X(g) (q) may take the next x
    BR_QKV = 2,     // QKV MMAs of the group's tile done
    BR_QKR = 3,     // v and the q, k of head 0 drained to shared memory (compute warps)
    BR_S = 4,       // + r: S in buffer r done
    BR_P = 6,       // + r: P in buffer r (compute warps)
    BR_PV = 8,      // + r: P.V into buffer r done
    BR_OD = 10,     // + r: o_h of buffer r drained (compute warps)
    BR_O = 12,      // every o_h staged in V(g) (compute warps)
    BR_Y = 13,      // projection done
    BR_RFREE = 14,  // y drained from TMEM: the group's columns are free (compute warps)
    BR_STAGE = 15,  // output rows staged in V(g) (compute warps)
    BR_VFREE = 16,  // output stored: V(g) may take the next v (producer)
    BR_QKR1 = 17,   // + h - 1: q and k of head h = 1, 2, 3 drained (compute warps)
    BR_XREAD = 20,  // (pre-norm fold, G = 1) both groups have read the tile's x for their statistics
    BR_QKFREE = 42  // (shared) q and k of the last QKV drained from TMEM (compute warps)
};


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

// The same from every lane of a warp, with a warp-uniform result: the warp
// goes on to its warp-collective tcgen05 loads and stores only if every
// lane's wait ended.  (Polling from lane 0 alone, with a warp barrier
// after it, measured slower: 71.7 against 63.7 us on Swin-T stage 1.)
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
{
    const bool ok = wait_or_abort(bar, parity, limit_ns, abort);
    return __all_sync(0xffffffffu, ok);
}
// One arrival per warp on a ready barrier: every lane's prior shared-memory
// writes (made visible to the async proxy by the caller where an MMA reads
// them) and TMEM accesses happen before it.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// x0 += b0, x1 += b1 as one two-lane fp32 add (add.rn.f32x2).
__device__ __forceinline__ void fadd2(float &x0, float &x1, float b0, float b1)
{
    asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %3};\n\t"
        "add.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(b0), "f"(b1));
}

// x0 *= m, x1 *= m as one two-lane fp32 multiply (mul.rn.f32x2).
__device__ __forceinline__ void fmul2(float &x0, float &x1, float m)
{
    asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\t"
        "mul.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(m));
}

// x0 = x0 * m + b0, x1 = x1 * m + b1 as one two-lane fp32 fma (fma.rn.f32x2).
__device__ __forceinline__ void ffma2(float &x0, float &x1, float m, float b0, float b1)
{
    asm("{\n\t.reg .b64 p, q, r;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\t"
        "mov.b64 r, {%3, %4};\n\tfma.rn.f32x2 p, p, q, r;\n\tmov.b64 {%0, %1}, p;\n\t}"
        : "+f"(x0), "+f"(x1)
        : "f"(m), "f"(b0), "f"(b1));
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint4 pack8(const float *v)
{
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

// A shared-memory descriptor whose start address (bits 0..13, 16-byte
// units) is moved by `bytes`.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t bytes) { return d + (uint64_t)(bytes >> 4); }

// Where window `sl` (0: rows 0..63, 1: rows 64..127) of tile `tile` lies:
// kind 0 = none (odd window count), 1 = copied by TMA boxes, 2 = wraps around
// the image edge (cp.async / plain stores, and the only kind the shift mask
// cuts); its batch image, window row and column, and its first image row
// (b*H + i) and token column in the original frame.
struct WinInfo {
    int kind, b, wi, wj, img_row0, col0;
};

__device__ __forceinline__ WinInfo window_info(const Geom &g, int tile, int sl)
{
    WinInfo w;
    const int win = 2 * tile + sl;
    if (win >= (int)g.nwin) {
        w.kind = w.b = w.wi = w.wj = w.img_row0 = w.col0 = 0;
        return w;
    }
    const int per = g.nh * g.nw;
    w.b = win / per;
    const int rem = win - w.b * per;
    w.wi = rem / g.nw;
    w.wj = rem - w.wi * g.nw;
    w.kind = g.s > 0 && (w.wi == g.nh - 1 || w.wj == g.nw - 1) ? 2 : 1;
    w.img_row0 = w.b * g.H + w.wi * g.M + g.s;
    w.col0 = w.wj * g.M + g.s;
    return w;
}

// Token index (b*H*W + i*W + j) of in-window position (ti, tj), ti, tj < M.
__device__ __forceinline__ int window_token(const Geom &g, const WinInfo &w, int ti, int tj)
{
    int i = w.wi * g.M + g.s + ti;
    if (i >= g.H) i -= g.H;
    int j = w.wj * g.M + g.s + tj;
    if (j >= g.W) j -= g.W;
    return (w.b * g.H + i) * g.W + j;
}

template <int M, int C, int G, int FOLD>
__global__ void __launch_bounds__(FTHREADS, 1)
    fused_block_kernel(FusedArgs a, DeviceStatus st, const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_out)
// tmap_x: x as [B*H][W][C], boxes of 32 x 8 x M; tmap_out: out as [B*H][W][C],
// boxes of 32 x M x M
{
    using F = FusedCfg<M, C, G>;
    constexpr int HEADS = F::HEADS, L = F::L, KB = F::KB, HT = F::HT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    uint8_t *small = sm + F::SMALL;
    float *sbqkv = reinterpret_cast<float *>(small + F::O_BQKV);
    float *sbproj = reinterpret_cast<float *>(small + F::O_BPROJ);
    float *sscale = reinterpret_cast<float *>(small + F::O_SCALE);
    float *sref = reinterpret_cast<float *>(small + F::O_REF);
    float *sbias = reinterpret_cast<float *>(small + F::O_BIAS);
    float *sln = reinterpret_cast<float *>(small + F::O_LN);
    float *scsum = reinterpret_cast<float *>(small + F::O_CSUM);
    volatile int *sring = reinterpret_cast<volatile int *>(small + F::O_RING);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + F::O_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + F::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);

    const Geom g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);
    auto BAR = [&](int grp, int i) { return smem_u32(&bars[21 * grp + i]); };
    // q and k of head h drained (and, for h = 0, v before them)
    auto QKR = [&](int grp, int h) { return BAR(grp, h == 0 ? BR_QKR : BR_QKR1 + h - 1); };
    const uint32_t B_QKFREE = smem_u32(&bars[BR_QKFREE]);
    const int ntiles = (int)((g.nwin + 1) / 2);
    auto X = [&](int grp) { return base + F::XT + grp * KB * HT; };
    auto K = [&](int grp) { return F::SPLIT ? base + F::XT : base + F::KT + grp * KB * HT; };
    auto V = [&](int grp) { return base + F::VT + grp * KB * HT; };

    // ---- once per CTA: barriers and zeroed x tiles first, so that the
    // producer starts gathering at once; the other eleven warps meanwhile
    // bring in the weights and tables (their own barrier, 352 threads) and
    // allocate TMEM ---------------------------------------------------------
    if (tid == 0) {
        for (int grp = 0; grp < 2; ++grp) {
            const int b0 = 21 * grp;
            mbar_init(smem_u32(&bars[b0 + BR_X]), 2);
            mbar_init(smem_u32(&bars[b0 + BR_XREAD]), F::TW);
            mbar_init(smem_u32(&bars[b0 + BR_XFREE]), F::SPLIT ? 2 : 1);   // a commit per S issuer
            mbar_init(smem_u32(&bars[b0 + BR_QKV]), 1);
            mbar_init(smem_u32(&bars[b0 + BR_QKR]), GWARPS);
            for (int h = 1; h < 4; ++h) mbar_init(smem_u32(&bars[b0 + BR_QKR1 + h - 1]), GWARPS);
            for (int r = 0; r < 2; ++r) {
                mbar_init(smem_u32(&bars[b0 + BR_S + r]), 1);
                mbar_init(smem_u32(&bars[b0 + BR_P + r]), GWARPS);
                mbar_init(smem_u32(&bars[b0 + BR_PV + r]), 1);
                mbar_init(smem_u32(&bars[b0 + BR_OD + r]), GWARPS);
            }
            mbar_init(smem_u32(&bars[b0 + BR_O]), F::TW);
            mbar_init(smem_u32(&bars[b0 + BR_Y]), 1);
            mbar_init(smem_u32(&bars[b0 + BR_RFREE]), F::TW);
            mbar_init(smem_u32(&bars[b0 + BR_STAGE]), F::TW);
            mbar_init(smem_u32(&bars[b0 + BR_VFREE]), 1);
        }
        mbar_init(smem_u32(&bars[BR_QKFREE]), F::TW);
        *abort_flag = 0;
        mbar_init_fence();
    }
    // the x tiles start as zeros: rows that no window token fills (8*ti + tj
    // with ti or tj >= M, a missing second window) then only ever hold
    // finite values (zeros, other tokens, q of earlier tiles), so the v
    // rows of keys that do not exist -- multiplied by P = 0 -- stay finite
    for (int i = tid; i < G * KB * HT / 16; i += FTHREADS)
        reinterpret_cast<uint4 *>(sm + F::XT)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();   // (TMA writes and MMA reads of these bytes come after)
    __syncthreads();   // barriers, zeroed x tiles
    uint32_t tmem = 0;
    if (warp != PWARP) {
        const int stid = tid - 32;   // setup thread index (the producer warp excluded)
        constexpr int NS = FTHREADS - 32;
        auto setup_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(FTHREADS - 32) : "memory"); };
        {
            for (int q = stid; q < (2 * C) * (C / 8); q += NS) {     // Wq, Wk rows
                const int r = q / (C / 8), c16 = q % (C / 8);
                cp_async16(base + F::WQK + (c16 >> 2) * (2 * C * 64) + sw64_offset(r, c16 & 3),
                           a.Wqkv + (int64_t)r * C + c16 * 8, 16);
            }
            for (int q = stid; q < C * (C / 8); q += NS) {           // Wv rows
                const int r = q / (C / 8), c16 = q % (C / 8);
                cp_async16(base + F::WV + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3),
                           a.Wqkv + (int64_t)(2 * C + r) * C + c16 * 8, 16);
            }
            for (int q = stid; q < C * (C / 8); q += NS) {           // Wproj
                const int r = q / (C / 8), c16 = q % (C / 8);
                cp_async16(base + F::WP + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3),
                           a.Wproj + (int64_t)r * C + c16 * 8, 16);
            }
            cp_async_commit();
            for (int i = stid; i < HEADS * L * L; i += NS) {
                const int hd = i / (L * L), e = i % (L * L);
                sbias[(hd * L + e / L) * F::LP + e % L] = __bfloat162float(a.table[(int64_t)e * HEADS + hd]) * FLOG2E;
            }
            for (int i = stid; i < 3 * C; i += NS) sbqkv[i] = a.bqkv ? __bfloat162float(a.bqkv[i]) : 0.f;
            for (int i = stid; i < C; i += NS) sbproj[i] = a.bproj ? __bfloat162float(a.bproj[i]) : 0.f;
            if (FOLD)
                for (int i = stid; i < C; i += NS) {
                    sln[i] = __bfloat162float(a.ln_g[i]);
                    sln[C + i] = __bfloat162float(a.ln_b[i]);
                }
            if (stid < HEADS)
                sscale[stid] = a.mode == 1 ? FLOG2E / fmaxf(a.tau[stid], 0.01f) : FLOG2E * rsqrtf(32.0f);
            cp_async_wait<0>();
            fence_proxy_async_smem();
        }
        setup_sync();   // the weights and bias vectors are in shared memory
        if (FOLD == 1) {
            // Pre-norm: LN(x) = xh * gamma + beta with xh = (x - mean) * rstd, so
            // LN(x) Wqkv^T + bqkv = rstd (x W'^T - mean c) + b' with W' = Wqkv
            // diag(gamma), c its row sums (over the input channels) and b' =
            // Wqkv beta + bqkv: the MMAs take x as it is, and each row's rstd and
            // mean (each compute thread's, of its own row) enter as the q, k, v
            // columns are drained.
            // The bias first (fp32, the unscaled weights, one thread per output in
            // a fixed order), then every weight scaled by its column's gamma (bf16,
            // in place), then c from the scaled bf16 weights the MMAs use.
            auto wrow = [&](int n, int c16) -> uint8_t * {
                return n < 2 * C ? sm + F::WQK + (c16 >> 2) * (2 * C * 64) + sw64_offset(n, c16 & 3)
                                 : sm + F::WV + (c16 >> 2) * (C * 64) + sw64_offset(n - 2 * C, c16 & 3);
            };
            for (int n = stid; n < 3 * C; n += NS) {
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
                sbqkv[n] += acc;
            }
            setup_sync();   // (every bias read the unscaled weights)
    #pragma unroll 1
            for (int q = stid; q < 3 * C * (C / 8); q += NS) {
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
            fence_proxy_async_smem();   // read by the QKV MMAs
            setup_sync();
            for (int n = stid; n < 3 * C; n += NS) {
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
                scsum[n] = acc;
            }
            setup_sync();
        }
        // The value bias moves behind the softmax: a row's attention weights sum to
        // 1, so o = P (v + bv) = P v + bv, and (P v + bv) Wproj^T + bproj =
        // (P v) Wproj^T + (Wproj bv + bproj).  The projection bias used below is
        // that sum (fp32), and v is drained without a bias.  One thread per
        // output channel, in a fixed order (the result is the same on every CTA
        // and every call).
        if (stid >= C && stid < C + HEADS) {
            // V2: a head's logits (log2 units) lie in [-scale + min B, scale + max B]
            // (|cos| <= 1).  Where that span is at most 96, scale + max B serves
            // as the softmax reference instead of the row maximum: every weight is
            // then at least 2^-96 of it (no underflow to zero) and the normalised
            // result is the same.  V1 logits have no such bound: NaN, row maxima.
            const int hd = stid - C;
            float bmax = -INFINITY, bmin = INFINITY;
            for (int r = 0; r < L; ++r)
                for (int c = 0; c < L; ++c) {
                    const float v = sbias[(hd * L + r) * F::LP + c];
                    bmax = fmaxf(bmax, v);
                    bmin = fminf(bmin, v);
                }
            const float sc = sscale[hd];
            sref[hd] = a.mode == 1 && 2.f * sc + (bmax - bmin) <= 96.f ? sc + bmax : __int_as_float(0x7fffffff);
        }
        if ((a.bqkv || FOLD == 1) && stid < C) {
            float acc = 0.f;
            for (int c8 = 0; c8 < C / 8; ++c8) {
                const uint4 w8 =
                    *reinterpret_cast<const uint4 *>(sm + F::WP + (c8 >> 2) * (C * 64) + sw64_offset(stid, c8 & 3));
                const float *bv = sbqkv + 2 * C + 8 * c8;
                const float2 w01 = unpack_bf16x2(w8.x), w23 = unpack_bf16x2(w8.y), w45 = unpack_bf16x2(w8.z),
                             w67 = unpack_bf16x2(w8.w);
                acc = fmaf(w01.x, bv[0], acc);
                acc = fmaf(w01.y, bv[1], acc);
                acc = fmaf(w23.x, bv[2], acc);
                acc = fmaf(w23.y, bv[3], acc);
                acc = fmaf(w45.x, bv[4], acc);
                acc = fmaf(w45.y, bv[5], acc);
                acc = fmaf(w67.x, bv[6], acc);
                acc = fmaf(w67.y, bv[7], acc);
            }
            sbproj[stid] += acc;
        }
        if (warp == QWARP) {
            tmem_alloc(smem_u32(tmem_slot), 512);
            tmem_relinquish();
        }
        tc_fence_before();
        setup_sync();   // weights, tables, TMEM address
        tc_fence_after();
        tmem = *tmem_slot;
    }

    // Tiles are handed out at run time: the producer takes the next one from
    // a counter shared by the CTAs (windows on the shifted edges cost more, so
    // a fixed share per CTA left some CTAs running 20% longer than others)
    // and writes the CTA's j-th tile into ring slot j mod 4 before its first
    // arrival on BR_X; once the tiles run out it writes -1 into the next G
    // slots and completes their BR_X phases without loads.  Every other role
    // reads the slot after its wait on BR_X of tile j, and leaves at -1.  A
    // slot is written again four tiles later, after XFREE of tile j + 4 - G,
    // which every reader of tile j has passed by then.

    // The prologue above reads only the parameters; x, the tile counter and out
    // wait for the kernels queued before this one (a no-op unless launched to
    // overlap them), and the next such kernel may start its own prologue.
    griddep_launch_dependents();
    griddep_wait();
    if (warp == PWARP) {
        // ===================== producer warp: x gathers =====================
        const bool tma_thread = lane == 0;
        // x rows of tile `tile` into X(grp): TMA boxes (the TMA thread's arrival
        // on BR_X carries their bytes) and, for wrapping windows, cp.async
        // copies, a row per lane and pass.  BR_X's second arrival comes once
        // the cp.async copies have landed (x_landed); a tile without them gets
        // it at once.  Returns whether copies are pending.
        auto load_x = [&](int grp, int tile) -> bool {
            const uint32_t xb = X(grp), bx = BAR(grp, BR_X);
            const WinInfo w0 = window_info(g, tile, 0), w1 = window_info(g, tile, 1);
            if (tma_thread) {
                const uint32_t bytes = ((w0.kind == 1) + (w1.kind == 1)) * KB * (M * 8 * 64);
                mbar_arrive_expect_tx(bx, bytes);
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const WinInfo &w = sl ? w1 : w0;
                    if (w.kind != 1) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_3d(xb + kb * HT + sl * (64 * 64), &tmap_x, kb * 32, w.col0, w.img_row0, bx);
                }
            }
            if (w0.kind != 2 && w1.kind != 2) {
                if (tma_thread) mbar_arrive(bx);
                return false;
            }
#pragma unroll
            for (int sl = 0; sl < 2; ++sl) {
                const WinInfo &w = sl ? w1 : w0;
                if (w.kind != 2) continue;
                for (int t = lane; t < 64; t += 32) {
                    const int ti = t >> 3, tj = t & 7;
                    if (ti >= M || tj >= M) continue;
                    const bf16 *src = a.x + (int64_t)window_token(g, w, ti, tj) * C;
                    const int r = sl * 64 + t;
#pragma unroll
                    for (int c16 = 0; c16 < C / 8; ++c16)
                        cp_async16(xb + (c16 >> 2) * HT + sw64_offset(r, c16 & 3), src + c16 * 8, 16u);
                }
            }
            cp_async_commit();
            return true;
        };
        auto x_landed = [&](int grp) {
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(grp, BR_X));
        };
        bool ok = true;
        int ends = 0;   // end marks written
#pragma unroll 1
        for (int j = 0; ends < G; ++j) {
            const int grp = j % G, kg = j / G;
            // X(grp) takes tile j once the group's S MMAs of its previous tile have
            // read q (G = 1: k)
            if (j >= G && !(ok = warp_wait(BAR(grp, BR_XFREE), (kg - 1) & 1, st.wait_ns, abort_flag))) break;
            int tile = -1;
            if (ends == 0) {
                if (lane == 0) tile = atomicAdd(a.sched, 1);
                tile = __shfl_sync(0xffffffffu, tile, 0);
                if (tile >= ntiles) tile = -1;
            }
            if (tile < 0) {
                ++ends;
                if (lane == 0) {
                    sring[j & 3] = -1;
                    mbar_arrive(BAR(grp, BR_X));
                    mbar_arrive(BAR(grp, BR_X));
                }
                continue;
            }
            if (lane == 0) sring[j & 3] = tile;
            __syncwarp();
            if (load_x(grp, tile)) x_landed(grp);
        }
        cp_async_wait<0>();
        if (!ok) *abort_flag = 1;
    } else if (warp == QWARP) {
        // ============ QKV issuer: the CTA's tiles in order ============
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, 2 * C), id_c = idesc_bf16(128, C);
            const uint64_t d_wqk = desc_kmajor_sw64(base + F::WQK), d_wv = desc_kmajor_sw64(base + F::WV);
            bool ok = true;
#pragma unroll 1
            for (int j = 0;; ++j) {
                const int grp = j % G, kg = j / G;
                // tile j's x has landed, the q|k columns are free (tile j - 1's
                // drained) and the group's columns are free (y of its previous tile
                // drained)
                if (!(ok = wait_or_abort(BAR(grp, BR_X), kg & 1, st.wait_ns, abort_flag))) break;
                if (sring[j & 3] < 0) break;
                if (j > 0 && !(ok = wait_or_abort(B_QKFREE, (j - 1) & 1, st.wait_ns, abort_flag))) break;
                if (kg > 0 && !(ok = wait_or_abort(BAR(grp, BR_RFREE), (kg - 1) & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                const uint64_t dx = desc_kmajor_sw64(X(grp));
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_QK, desc_add(dx, kb * HT + 32 * ks),
                                 desc_add(d_wqk, kb * (2 * C * 64) + 32 * ks), id_qk, (kb | ks) != 0);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_R0 + 128 * grp, desc_add(dx, kb * HT + 32 * ks),
                                 desc_add(d_wv, kb * (C * 64) + 32 * ks), id_c, (kb | ks) != 0);
                mma_commit(BAR(grp, BR_QKV));
            }
            if (!ok) *abort_flag = 1;
        }
    } else if (warp < CWARP0) {
        // ============ issuer of group warp - 2: S, P.V, the projection ============
        // (G = 1: issuer g takes group g's heads of every tile; group 0's issuer
        // also the projection and the stores)
        const int grp = warp - AWARP0;
        const int tg = F::SPLIT ? 0 : grp;         // the tile's buffers and tile barriers
        const int h0 = F::SPLIT ? grp * F::HPG : 0;   // the group's first head
        if (lane == 0) {
            constexpr uint32_t id_s = idesc_bf16(128, 64), id_pv = idesc_bf16_bmn(128, 32), id_y = idesc_bf16(128, C);
            const uint64_t d_wp = desc_kmajor_sw64(base + F::WP);
            // output-lane masks: every row but window A's / window B's
            const uint32_t mask_a[4] = {0u, 0u, ~0u, ~0u}, mask_b[4] = {~0u, ~0u, 0u, 0u};
            const uint32_t t_r = tmem + F::T_R0 + 128 * grp, t_y = tmem + F::T_R0 + 128 * tg;
            const uint64_t dq = desc_kmajor_sw64(X(tg)), dk = desc_kmajor_sw64(K(tg));
            const uint64_t dv = desc_mnmajor_sw64(V(tg), 8192);
            // S of the group's head hl into buffer r: all 128 q rows against each
            // window's 64 keys, each MMA keeping only its window's rows (G = 1: q
            // from TMEM)
            auto issue_s = [&](int hl, int r) {
                const int hd = h0 + hl;
                const uint32_t d = t_r + 64 * r;
#pragma unroll
                for (int w = 0; w < 2; ++w)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks) {
                        const uint64_t bk = desc_add(dk, hd * HT + 4096 * w + 32 * ks);
                        if (F::SPLIT)
                            mma_bf16_ts_mask(d, tmem + F::T_QK + 32 * hd + 8 * ks, bk, id_s, ks, w ? mask_b : mask_a);
                        else
                            mma_bf16_mask(d, desc_add(dq, hd * HT + 32 * ks), bk, id_s, ks, w ? mask_b : mask_a);
                    }
                mma_commit(BAR(grp, BR_S + r));
            };
            // o_h = P v_h over each window's 64 keys, for its rows, into the upper
            // 32 columns of buffer r
            auto issue_pv = [&](int hl, int r) {
                const int hd = h0 + hl;
                const uint32_t pa = t_r + 64 * r, d = t_r + 64 * r + 32;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts_mask(d, pa + 8 * kk, desc_add(dv, hd * HT + 1024 * kk), id_pv, kk, mask_a);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts_mask(d, pa + 8 * kk, desc_add(dv, hd * HT + 4096 + 1024 * kk), id_pv, kk, mask_b);
                mma_commit(BAR(grp, BR_PV + r));
            };
            // phases: bit r of ph_p is BR_P + r's; od_n[r] counts the completions of
            // BR_OD + r so far (every o_h drain completes one; only those before
            // an S of head h + 2 are waited for here)
            uint32_t ph_p = 0;
            uint32_t od_n[2] = {0u, 0u};
            bool ok = true;
#pragma unroll 1
            for (int j = F::SPLIT ? 0 : grp; ok; j += G) {
                const int kg = j / G;
                if (!(ok = wait_or_abort(BAR(tg, BR_X), kg & 1, st.wait_ns, abort_flag))) break;
                const int p_tile = sring[j & 3];
                if (p_tile < 0) break;
                // S of the group's first two heads as soon as their q and k are
                // stored (v, drained first, has then left the TMEM columns S takes)
                if (!(ok = wait_or_abort(QKR(grp, 0), kg & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                issue_s(0, 0);
                if (F::HPG > 1) {
                    if (!(ok = wait_or_abort(QKR(grp, 1), kg & 1, st.wait_ns, abort_flag))) break;
                    tc_fence_after();
                    issue_s(1, 1);
                }
                if (F::HPG <= 2) mma_commit(BAR(tg, BR_XFREE));   // the group's last S has read q / k
#pragma unroll 1
                for (int hl = 0; hl < F::HPG; ++hl) {
                    const int r = hl & 1;
                    if (!(ok = wait_or_abort(BAR(grp, BR_P + r), (ph_p >> r) & 1u, st.wait_ns, abort_flag))) break;
                    ph_p ^= 1u << r;
                    // (G = 1: group 1's P.V reads the v that group 0 drains)
                    if (F::SPLIT && grp == 1 && hl == 0 &&
                        !(ok = wait_or_abort(QKR(0, 0), kg & 1, st.wait_ns, abort_flag)))
                        break;
                    tc_fence_after();
                    issue_pv(hl, r);
                    if (hl + 2 < F::HPG) {
                        // S of head hl + 2 into buffer r once o_hl has left it
                        if (!(ok = wait_or_abort(BAR(grp, BR_OD + r), od_n[r] & 1u, st.wait_ns, abort_flag))) break;
                        if (!(ok = wait_or_abort(QKR(grp, hl + 2), kg & 1, st.wait_ns, abort_flag))) break;
                        tc_fence_after();
                        issue_s(hl + 2, r);
                        if (hl + 2 == F::HPG - 1) mma_commit(BAR(tg, BR_XFREE));
                    }
                    ++od_n[r];
                }
                if (!ok) break;
                if (F::SPLIT && grp == 1) continue;   // (tg's issuer: the projection and the stores)
                // y = o Wproj^T into the tile's columns once every o_h is staged
                if (!(ok = wait_or_abort(BAR(tg, BR_O), kg & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                const uint64_t doa = desc_kmajor_sw64(V(tg));
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(t_y, desc_add(doa, kb * HT + 32 * ks), desc_add(d_wp, kb * (C * 64) + 32 * ks), id_y,
                                 (kb | ks) != 0);
                mma_commit(BAR(tg, BR_Y));
                // tile j's output rows (staged in V(tg) by the compute warps) -> out
                // through the window reverse + roll(+s) map; V(tg) may take the
                // next v once the stores have read them
                if (!(ok = wait_or_abort(BAR(tg, BR_STAGE), kg & 1, st.wait_ns, abort_flag))) break;
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const WinInfo w = window_info(g, p_tile, sl);
                    if (w.kind != 1) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_store_3d(&tmap_out, kb * 32, w.col0, w.img_row0, V(tg) + kb * HT + sl * (64 * 64));
                }
                bulk_commit();
                bulk_wait_read();
                mbar_arrive(BAR(tg, BR_VFREE));
            }
            bulk_wait_all();
            if (!ok) *abort_flag = 1;
        }
    } else {
        // ===================== compute warps =====================
        // (G = 1: group g takes heads [g HPG, (g + 1) HPG) of every tile, group 0
        // also v, and each group half of y)
        const int grp = (warp - CWARP0) / GWARPS, quarter = warp & 3;
        const int tg = F::SPLIT ? 0 : grp;            // the tile's buffers and tile barriers
        const int h0 = F::SPLIT ? grp * F::HPG : 0;   // the group's first head
        constexpr int KBG = F::SPLIT ? KB / 2 : KB;   // y's 32-column blocks per group
        const int kb0 = F::SPLIT ? grp * KBG : 0;
        const int row = quarter * 32 + lane;        // tile row = TMEM lane
        const int slot = row >> 6, t = row & 63;    // window slot; token (t >> 3, t & 7) of the row
        const int ti = t >> 3, tj = t & 7;
        const bool tok_row = ti < M && tj < M;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        const uint32_t t_r = t_lane + F::T_R0 + 128 * grp, t_y = t_lane + F::T_R0 + 128 * tg;
        uint8_t *xg = sm + F::XT + tg * KB * HT, *vg = sm + F::VT + tg * KB * HT;
        uint8_t *kgs = F::SPLIT ? xg : sm + F::KT + tg * KB * HT;
        // relative-bias row of this token; rows no token fills (their results
        // are never stored) read the nearest token row's entries: a valid row,
        // and the same addresses as a neighbour lane's
        const int bias_base = (min(ti, M - 1) + M - 1) * F::LP + (min(tj, M - 1) + M - 1);
        uint32_t ph_s = 0, ph_pv = 0;   // bit r: phase of BR_S + r / BR_PV + r
        // row sum of the head whose softmax last used S buffer r (each drain of
        // head h comes before the softmax of head h + 2)
        float l0 = 1.f, l1 = 1.f;
        bool ok = true;
#pragma unroll 1
        for (int j = F::SPLIT ? 0 : grp;; j += G) {
            const int kg = j / G;
            if (!(ok = warp_wait(BAR(tg, BR_X), kg & 1, st.wait_ns, abort_flag))) break;
            const int p_tile = sring[j & 3];
            if (p_tile < 0) break;
            const WinInfo win = window_info(g, p_tile, slot);
            // (pre-norm fold: the row's statistics come from x while the QKV MMAs
            // run on it)
            float2 rs = make_float2(1.f, 0.f);
            if (FOLD == 1) {
                // (pre-norm fold) this row's LayerNorm statistics, from its x in
                // X (read before the drains overwrite it, and while the QKV MMAs
                // read it too): fp32 mean, then mean square deviation.  Rows that hold no token get finite values
                // from whatever finite data the row holds; never stored.
                auto xchunk = [&](int c) {
                    return *reinterpret_cast<const uint4 *>(xg + (c >> 2) * HT + sw64_offset(row, c & 3));
                };
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < C / 8; ++c) {
                    const uint4 u = xchunk(c);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(wd[e]);
                        s4[2 * (e & 1)] += f.x;
                        s4[2 * (e & 1) + 1] += f.y;
                    }
                }
                const float mean = ((s4[0] + s4[1]) + (s4[2] + s4[3])) / (float)C;
                float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 0; c < C / 8; ++c) {
                    const uint4 u = xchunk(c);   // (read again: fewer live registers)
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(wd[e]);
                        const float d0 = f.x - mean, d1 = f.y - mean;
                        q4[2 * (e & 1)] = fmaf(d0, d0, q4[2 * (e & 1)]);
                        q4[2 * (e & 1) + 1] = fmaf(d1, d1, q4[2 * (e & 1) + 1]);
                    }
                }
                const float rstd = rsqrtf(((q4[0] + q4[1]) + (q4[2] + q4[3])) / (float)C + 1e-5f);
                rs = make_float2(rstd, -rstd * mean);
                // (G = 1: the other group writes k over these x rows)
                if (F::SPLIT) warp_arrive(BAR(tg, BR_XREAD), lane);
            }
            if (!(ok = warp_wait(BAR(tg, BR_QKV), kg & 1, st.wait_ns, abort_flag))) break;
            tc_fence_after();

            // ---- q and k of every head -> X(grp), K(grp) (bf16; V2: unit length),
            // then v -> V(grp) (the N-major B operand of P.V); two or three
            // 32-column TMEM loads in flight per wait ----
            // bias of the 32 channels from `bias`, V2 scaling, bf16, the row of a
            // [128][32] tile at dst
            // (pre-norm fold: v = rstd (acc - mean c) + bias = acc rs.x + (c rs.y +
            // bias), c the 32 column sums at csum)
            auto fold_in = [&](float (&v)[32], const float *bias, const float *csum) {
                const float4 *c4 = reinterpret_cast<const float4 *>(csum);
                const float4 *b4 = reinterpret_cast<const float4 *>(bias);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 cc = c4[e4], bb = bias ? b4[e4] : make_float4(0.f, 0.f, 0.f, 0.f);
                    float t0 = cc.x, t1 = cc.y, t2 = cc.z, t3 = cc.w;
                    ffma2(t0, t1, rs.y, bb.x, bb.y);
                    ffma2(t2, t3, rs.y, bb.z, bb.w);
                    ffma2(v[4 * e4], v[4 * e4 + 1], rs.x, t0, t1);
                    ffma2(v[4 * e4 + 2], v[4 * e4 + 3], rs.x, t2, t3);
                }
            };
            auto put = [&](float (&v)[32], const float *bias, const float *csum, uint8_t *dst, bool unit) {
                if (FOLD == 1) {
                    fold_in(v, bias, csum);
                } else if (bias) {
                    const float4 *b4 = reinterpret_cast<const float4 *>(bias);
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 bb = b4[e4];
                        fadd2(v[4 * e4], v[4 * e4 + 1], bb.x, bb.y);
                        fadd2(v[4 * e4 + 2], v[4 * e4 + 3], bb.z, bb.w);
                    }
                }
                if (unit) {
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
                    const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
                    for (int e = 0; e < 32; e += 2) fmul2(v[e], v[e + 1], inv);
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4 *>(dst + sw64_offset(row, c)) = pack8(v + 8 * c);
            };
            const bool v2 = a.mode == 1;
            // v first (no bias, see the projection bias), once the previous tile's
            // output rows have left V(grp): it frees the TMEM columns of the S
            // buffers.  Then q and k head by head (q with its bias, V2: unit
            // length; V1 drops the key bias: it adds q.bk / sqrt(d) to every logit
            // of a row, which the softmax cancels; V2 normalises k + bk, so keeps
            // it), each head's S MMA issued as soon as its q and k are stored.
            if (!F::SPLIT || grp == 0) {
                if (kg > 0 && !(ok = warp_wait(BAR(tg, BR_VFREE), (kg - 1) & 1, st.wait_ns, abort_flag))) break;
                if (FOLD == 1) {
                    // (head by head: the fold's column sums take registers)
#pragma unroll 1
                    for (int hd = 0; hd < HEADS; ++hd) {
                        float vh[32];
                        tmem_ld32(t_y + 32 * hd, vh);
                        tmem_wait_ld();
                        put(vh, nullptr, scsum + 2 * C + 32 * hd, vg + hd * HT, false);
                    }
                } else {
                    float vv[HEADS][32];
#pragma unroll
                    for (int hd = 0; hd < HEADS; ++hd) tmem_ld32(t_y + 32 * hd, vv[hd]);
                    tmem_wait_ld();
#pragma unroll
                    for (int hd = 0; hd < HEADS; ++hd) put(vv[hd], nullptr, nullptr, vg + hd * HT, false);
                }
            }
            if (FOLD == 1 && F::SPLIT && !(ok = warp_wait(BAR(tg, BR_XREAD), kg & 1, st.wait_ns, abort_flag))) break;
#pragma unroll 1
            for (int hl = 0; hl < F::HPG; ++hl) {
                const int hd = h0 + hl;
                float vq[32], vk[32];
                tmem_ld32(t_lane + F::T_QK + 32 * hd, vq);
                tmem_ld32(t_lane + F::T_QK + C + 32 * hd, vk);
                tmem_wait_ld();
                if (F::SPLIT) {
                    // (G = 1) q back into TMEM as bf16 pairs over its first 16 fp32
                    // columns (this thread's lane, already read): the A operand of S
                    if (FOLD == 1) {
                        fold_in(vq, sbqkv + 32 * hd, scsum + 32 * hd);
                    } else {
                        const float4 *b4 = reinterpret_cast<const float4 *>(sbqkv + 32 * hd);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 bb = b4[e4];
                            fadd2(vq[4 * e4], vq[4 * e4 + 1], bb.x, bb.y);
                            fadd2(vq[4 * e4 + 2], vq[4 * e4 + 3], bb.z, bb.w);
                        }
                    }
                    if (v2) {
                        float ss = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) ss = fmaf(vq[e], vq[e], ss);
                        const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
                        for (int e = 0; e < 32; e += 2) fmul2(vq[e], vq[e + 1], inv);
                    }
                    uint32_t qp[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) qp[e] = pack_bf16x2(vq[2 * e], vq[2 * e + 1]);
                    tmem_st16(t_lane + F::T_QK + 32 * hd, qp);
                    tmem_wait_st();
                } else {
                    put(vq, sbqkv + 32 * hd, scsum + 32 * hd, xg + hd * HT, v2);
                }
                put(vk, v2 ? sbqkv + C + 32 * hd : nullptr, scsum + C + 32 * hd, kgs + hd * HT, v2);
                fence_proxy_async_smem();   // read by the S (and P.V) MMAs
                warp_arrive(QKR(grp, hl), lane);
            }
            warp_arrive(B_QKFREE, lane);   // the q|k columns may take the next QKV

            // ---- the keys this row may attend to: its own shift region (key rows:
            // bit ki of rbits, key columns: bit kj of cbits).  Only windows on the
            // last window row or column are cut; a warp's rows lie in one window,
            // so `masked` is warp-uniform ----
            const bool masked = win.kind == 2;
            uint32_t rbits = (1u << M) - 1u, cbits = (1u << M) - 1u;
            if (masked) {
                const uint32_t lo = (1u << (M - g.s)) - 1u, hi = ((1u << M) - 1u) & ~lo;
                if (win.wi == g.nh - 1) rbits = ti >= M - g.s ? hi : lo;
                if (win.wj == g.nw - 1) cbits = tj >= M - g.s ? hi : lo;
            }
            // action i of a tile: the softmax of head a (a >= 0) or the o drain of
            // head -a - 1 (a < 0)
            // (the group's heads hl: after softmax 0 and 1, drain h and softmax
            // h + 2 while h + 2 < HPG, then the last two drains; three heads: S0
            // S1 D0 S2 D1 D2)
            auto head_action = [](int i) -> int {
                constexpr int NH = F::HPG;
                if (i < 2) return i;
                const int k = i - 2;
                if (k < 2 * (NH - 2)) return (k & 1) ? (k >> 1) + 2 : -(k >> 1) - 1;
                return -(NH - 2 + k - 2 * (NH - 2)) - 1;
            };
            // ---- softmax of head hd (buffer hd & 1) over the row's window keys ----
            auto softmax = [&](int hl) -> bool {
                const int r = hl & 1, hd = h0 + hl;
                if (!warp_wait(BAR(grp, BR_S + r), (ph_s >> r) & 1u, st.wait_ns, abort_flag)) return false;
                ph_s ^= 1u << r;
                tc_fence_after();
                float s[64];
                tmem_ld32(t_r + 64 * r, *reinterpret_cast<float(*)[32]>(s));
                tmem_ld32(t_r + 64 * r + 32, *reinterpret_cast<float(*)[32]>(s + 32));
                tmem_wait_ld();
                const float scale = sscale[hd];
                const float *bias = sbias + hd * L * F::LP + bias_base;
                // key column 8*ki + kj of the row's window: relative-bias entry
                // bias_base - (ki*LP + kj); columns with ki or kj >= M hold no key.
                // The row maximum and sum run in four partial chains (key row ki
                // feeds chain ki % 4), two keys per three-input max.
                if (masked) {
#pragma unroll
                    for (int ki = 0; ki < M; ++ki)
#pragma unroll
                        for (int kj = 0; kj < M; ++kj) {
                            const int jj = 8 * ki + kj;
                            const float v = fmaf(s[jj], scale, bias[-(ki * F::LP + kj)]);
                            s[jj] = ((rbits >> ki) & (cbits >> kj) & 1u) ? v : -INFINITY;
                        }
                } else {
#pragma unroll
                    for (int ki = 0; ki < M; ++ki) {
#pragma unroll
                        for (int kj = 0; kj + 1 < M; kj += 2)
                            ffma2(s[8 * ki + kj], s[8 * ki + kj + 1], scale, bias[-(ki * F::LP + kj)],
                                  bias[-(ki * F::LP + kj + 1)]);
                        if (M & 1) s[8 * ki + M - 1] = fmaf(s[8 * ki + M - 1], scale, bias[-(ki * F::LP + M - 1)]);
                    }
                }
                // the reference: the head's fixed one (warp-uniform), else the row
                // maximum (every row keeps a finite logit: a token always sees
                // itself, and a row no token fills still sees a nonempty region)
                float mx = sref[hd];
                if (mx != mx) {
                    float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int ki = 0; ki < M; ++ki) {
#pragma unroll
                        for (int kj = 0; kj + 1 < M; kj += 2)
                            mq[ki & 3] = fmax3(mq[ki & 3], s[8 * ki + kj], s[8 * ki + kj + 1]);
                        if (M & 1) mq[ki & 3] = fmaxf(mq[ki & 3], s[8 * ki + M - 1]);
                    }
                    mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                }
                // p = exp2(logit - max), two keys per packed subtract and sum (two
                // two-lane partial sums)
                float sq[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[32];
                const float nmx = -mx;
#pragma unroll
                for (int jj = 0; jj < 64; jj += 2) {
                    const int ki = jj >> 3;
                    const bool k0 = ki < M && (jj & 7) < M, k1 = ki < M && ((jj + 1) & 7) < M;
                    float p0 = 0.f, p1 = 0.f;
                    if (k0 && k1) {
                        float d0 = s[jj], d1 = s[jj + 1];
                        fadd2(d0, d1, nmx, nmx);
                        p0 = ex2_approx(d0);
                        p1 = ex2_approx(d1);
                        fadd2(sq[2 * (ki & 1)], sq[2 * (ki & 1) + 1], p0, p1);
                    } else if (k0) {
                        p0 = ex2_approx(s[jj] - mx);
                        sq[2 * (ki & 1)] += p0;
                    }
                    pk[jj / 2] = pack_bf16x2(p0, p1);
                }
                const float sum = (sq[0] + sq[1]) + (sq[2] + sq[3]);
                if (r) l1 = sum;
                else l0 = sum;
                // P (bf16, two keys per 32-bit column) over the first 32 columns
                tmem_st16(t_r + 64 * r, *reinterpret_cast<uint32_t(*)[16]>(pk));
                tmem_st16(t_r + 64 * r + 16, *reinterpret_cast<uint32_t(*)[16]>(pk + 16));
                tmem_wait_st();
                warp_arrive(BAR(grp, BR_P + r), lane);
                return true;
            };
            // ---- o_h / rowsum -> bf16 -> head hd's tile of V(grp) (the
            // projection's A operand), once P.V has read v_h ----
            auto drain_o = [&](int hl) -> bool {
                const int r = hl & 1, hd = h0 + hl;
                if (!warp_wait(BAR(grp, BR_PV + r), (ph_pv >> r) & 1u, st.wait_ns, abort_flag)) return false;
                ph_pv ^= 1u << r;
                tc_fence_after();
                float o[32];
                tmem_ld32(t_r + 64 * r + 32, o);
                tmem_wait_ld();
                const float inv = rcp_approx(r ? l1 : l0);
#pragma unroll
                for (int e = 0; e < 32; e += 2) fmul2(o[e], o[e + 1], inv);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(vg + hd * HT + sw64_offset(row, c)) = pack8(o + 8 * c);
                warp_arrive(BAR(grp, BR_OD + r), lane);
                return true;
            };
            // heads 0 and 1 first (both S buffers), then each o_h drain frees its
            // buffer for the S of head h + 2: for three heads softmax 0, 1, drain
            // 0, softmax 2, drain 1, 2 (one rolled loop: one copy of each body,
            // which keeps the kernel's code within the instruction caches)
#pragma unroll 1
            for (int i = 0; i < 2 * F::HPG; ++i) {
                const int hl = head_action(i);
                if (!(ok = hl >= 0 ? softmax(hl) : drain_o(-hl - 1))) break;
            }
            if (!ok) break;
            fence_proxy_async_smem();   // o is read by the projection MMA
            warp_arrive(BAR(tg, BR_O), lane);

            // ---- y + bproj -> bf16 rows in V(grp), token (ti, tj) of a window at
            // row M*ti + tj of its half (one dense box per window for the TMA
            // store through the window reverse + roll(+s) map); the rows of
            // windows that wrap go straight to out ----
            // (block fold) the residual, this row's token of x (its channels
            // 32 kb0 ...): into L1 while the projection runs, then read block
            // by block
            const bool resid = FOLD != 0 && tok_row && win.kind != 0;
            const uint4 *xsrc =
                resid ? reinterpret_cast<const uint4 *>(a.x + (int64_t)window_token(g, win, ti, tj) * C + 32 * kb0)
                      : nullptr;
            if (resid) {
#pragma unroll
                for (int q = 0; q < (FOLD ? KBG * 4 : 0); q += 4) prefetch_l1(xsrc + q);
            }
            if (!(ok = warp_wait(BAR(tg, BR_Y), kg & 1, st.wait_ns, abort_flag))) break;
            tc_fence_after();
            {
                // (post-norm fold) the row's LayerNorm statistics, over all C
                // channels of y + bproj (this thread's): fp32 mean, then mean
                // square deviation
                constexpr bool post = !F::SPLIT && FOLD == 2;
                float nm = 0.f, rstd = 1.f;
                // y's 32-column block kb0 + kb: bias, (fold) LayerNorm and
                // residual, bf16 out
                auto finish = [&](float (&v)[32], int kb) {
                    const float4 *bp = reinterpret_cast<const float4 *>(sbproj + 32 * (kb0 + kb));
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 bb = bp[e4];
                        fadd2(v[4 * e4], v[4 * e4 + 1], bb.x, bb.y);
                        fadd2(v[4 * e4 + 2], v[4 * e4 + 3], bb.z, bb.w);
                    }
                    if (post) {
                        const float4 *g4 = reinterpret_cast<const float4 *>(sln + 32 * kb), *b4 = g4 + C / 4;
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 gg = g4[e4], bb = b4[e4];
                            float *w = v + 4 * e4;
                            fadd2(w[0], w[1], nm, nm);
                            fadd2(w[2], w[3], nm, nm);
                            fmul2(w[0], w[1], rstd);
                            fmul2(w[2], w[3], rstd);
                            w[0] = fmaf(w[0], gg.x, bb.x);
                            w[1] = fmaf(w[1], gg.y, bb.y);
                            w[2] = fmaf(w[2], gg.z, bb.z);
                            w[3] = fmaf(w[3], gg.w, bb.w);
                        }
                    }
                    if (resid) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint4 u = xsrc[4 * kb + q];
                            const float2 f0 = unpack_bf16x2(u.x), f1 = unpack_bf16x2(u.y), f2 = unpack_bf16x2(u.z),
                                         f3 = unpack_bf16x2(u.w);
                            float *w = v + 8 * q;
                            fadd2(w[0], w[1], f0.x, f0.y);
                            fadd2(w[2], w[3], f1.x, f1.y);
                            fadd2(w[4], w[5], f2.x, f2.y);
                            fadd2(w[6], w[7], f3.x, f3.y);
                        }
                    }
                    if (win.kind == 2) {   // (warp-uniform)
                        if (tok_row) {
                            uint4 *dst =
                                reinterpret_cast<uint4 *>(a.out + (int64_t)window_token(g, win, ti, tj) * C) + 4 * (kb0 + kb);
#pragma unroll
                            for (int c = 0; c < 4; ++c) dst[c] = pack8(v + 8 * c);
                        }
                    } else if (win.kind == 1 && tok_row) {
                        const int srow = slot * 64 + ti * M + tj;
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4 *>(vg + (kb0 + kb) * HT + sw64_offset(srow, c)) = pack8(v + 8 * c);
                    }
                };
                if (FOLD == 0) {
                    // all of y's blocks in one TMEM round trip
                    float y[KBG][32];
#pragma unroll
                    for (int kb = 0; kb < KBG; ++kb) tmem_ld32(t_y + 32 * (kb0 + kb), y[kb]);
                    tmem_wait_ld();
                    warp_arrive(BAR(tg, BR_RFREE), lane);   // the tile's TMEM columns are free
#pragma unroll
                    for (int kb = 0; kb < KBG; ++kb) finish(y[kb], kb);
                } else {
                    if (post) {
                        float y[KBG][32];
#pragma unroll
                        for (int kb = 0; kb < KBG; ++kb) tmem_ld32(t_y + 32 * kb, y[kb]);
                        tmem_wait_ld();
                        float sum = 0.f;
#pragma unroll
                        for (int kb = 0; kb < KBG; ++kb)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                y[kb][e] += sbproj[32 * kb + e];
                                sum += y[kb][e];
                            }
                        const float mean = sum / (float)C;
                        float sq = 0.f;
#pragma unroll
                        for (int kb = 0; kb < KBG; ++kb)
#pragma unroll
                            for (int e = 0; e < 32; ++e) {
                                const float d = y[kb][e] - mean;
                                sq = fmaf(d, d, sq);
                            }
                        nm = -mean;
                        rstd = rsqrtf(sq / (float)C + 1e-5f);
                    }
                    // one block at a time (fewer live registers)
#pragma unroll
                    for (int kb = 0; kb < KBG; ++kb) {
                        float v[32];
                        tmem_ld32(t_y + 32 * (kb0 + kb), v);
                        tmem_wait_ld();
                        if (kb == KBG - 1) warp_arrive(BAR(tg, BR_RFREE), lane);   // the tile's TMEM columns are free
                        finish(v, kb);
                    }
                }
            }
            fence_proxy_async_smem();   // the TMA stores read these rows
            warp_arrive(BAR(tg, BR_STAGE), lane);
        }
        if (!ok) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(st.err, ERR_TIMEOUT);
    if (tid == 0) {
        // every producer of this launch is past its last take from the counter
        // once the last CTA gets here: it zeroes both for the next launch
        __threadfence();
        if (atomicAdd(a.sched + 1, 1) == (int)gridDim.x - 1) {
            atomicExch(a.sched, 0);
            atomicExch(a.sched + 1, 0);
        }
    }
    if (warp == QWARP) {
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

template <int M, int C, int G, int FOLD>
cudaError_t launch_fused_t(const FusedArgs &a, DeviceStatus st, cudaStream_t stream)
{
    using F = FusedCfg<M, C, G>;
    const size_t smem = F::BYTES + 1024;
    auto kern = fused_block_kernel<M, C, G, FOLD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tx, to;
    e = make_tensor_map_sw64_3d(&tx, a.x, (int64_t)a.g.B * a.g.H, a.g.W, C, 8, M);
    if (e != cudaSuccess) return e;
    e = make_tensor_map_sw64_3d(&to, a.out, (int64_t)a.g.B * a.g.H, a.g.W, C, M, M);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.g.nwin + 1) / 2;
    const int grid = (int)(ntiles < num_sms() ? ntiles : num_sms());
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(FTHREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = a.overlap ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, st, tx, to);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace
} // namespace swin
