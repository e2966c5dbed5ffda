// The whole shifted-window attention block in one persistent kernel
// (sm_103a, tcgen05 + TMEM), for windows of at most 64 tokens (M = 7, 8) and
// C = 64 or 96 channels (2 or 3 heads of 32).
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
//   S2  [q|k|v] = X Wqkv^T (128 x 3C) on tcgen05 into TMEM; bias added when
//       draining to shared memory; V2 normalises q and k to unit length in
//       fp32 while draining.  The next tile's QKV runs while this tile's
//       heads are computed: it has TMEM columns of its own
//   S3-S5 per head: S = q k^T, block-diagonal: two MMAs (128 x 64 x 32)
//       write the same 64 columns, one for each window's rows (the other
//       window's rows masked by the MMA's output-lane mask), alternating
//       between two S buffers so that the next head's logits are ready while
//       this head's softmax runs; softmax of each row over its window's keys
//       with the relative bias and the shift mask (fp32, exp2); P (bf16) back
//       into TMEM over the S columns
//   S6  o_h = P v_h, again one lane-masked MMA pair (128 x 32 x 64), with P
//       read from TMEM as the A operand (so P never touches shared memory)
//   S7  y = (o / rowsum) Wproj^T on tcgen05 (into the o columns), o staged
//       as bf16 in the tile's x buffer
//   S8  y + bproj staged in shared memory (token (ti, tj) at row M*ti + tj)
//       and written through the window reverse + roll(+s) map into
//       out[B, H, W, C]: one 3-D TMA store (M x M tokens x 32 channels) per
//       window and 32 channels, plain stores for wrapping windows
// Nothing but x, the weights and out touches HBM.
//
// Warp roles.  Warps 4..11 compute: warp w serves TMEM lane quarter w % 4 =
// tile rows 32(w%4)..+31 and column half w / 4 - 1 (every drain and the
// softmax split their columns between the two halves).  Three warps issue the
// tcgen05 MMAs (lane 0 each; an MMA costs its issuing thread some 80 cycles
// whatever its size, so the small attention MMAs are spread over two
// issuers): warps 0 and 1 the S and P.V halves of the first and second
// window's rows, warp 2 the next tile's QKV and the projection.  Warp 3
// produces and retires tiles: the row -> token map and the attention masks
// of a tile, its x gather into one of two x buffers (freed as soon as the
// tile's QKV has read it), and the output store.  All hand-offs are mbarriers: "ready" barriers get one arrival per
// warp, "done" barriers are tcgen05.commit targets.  Every barrier that
// serves alternating buffers is split per buffer, so no barrier can run two
// phases ahead of a waiter by construction.
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int NCWARPS = 8;                       // compute warps
constexpr int NCOMPUTE = NCWARPS * 32;
// (the issuers and the producer take the lowest warp indices: a warp
// scheduler that prefers older warps then serves them first; they wait by
// suspending on mbarriers, so they take no issue slots while idle)
constexpr int ATT_WARP0 = 0;                     // warps 0, 1: S and P.V of one window's rows each
constexpr int QKV_WARP = 2;                      // warp 2: QKV and the projection
constexpr int PWARP = 3;                         // warp 3: producer
constexpr int CWARP0 = 4;                        // warps 4..11: compute
constexpr int NPROD = 32;
constexpr int FTHREADS = NCOMPUTE + 3 * 32 + NPROD;   // 384
// (384 threads cap registers at 168 per thread, so that three warps of one
// SM sub-partition fit its 16 K registers)
constexpr int FBOUND_THREADS = 384;
constexpr float FLOG2E = 1.4426950408889634f;

template <int M, int C>
struct FusedCfg {
    static constexpr int HEADS = C / 32;
    static constexpr int L = 2 * M - 1;
    static constexpr int KB = C / 32;          // 32-channel K blocks (64-byte swizzle)
    // shared memory (bytes); SW64 tiles are 512-aligned, SW128 tiles 1024-aligned
    static constexpr int WQK = 0;                       // [2C rows][C]   SW64
    static constexpr int WV = WQK + 2 * C * C * 2;      // [C rows][C]    SW64
    static constexpr int WP = WV + C * C * 2;           // [C rows][C]    SW64
    // x buffers: tile k's x in X(k % 2), free again as soon as its QKV has
    // read it (the tile two ahead is gathered into it while this one runs)
    static constexpr int XSZ = 128 * C * 2;
    static constexpr int X0 = WP + C * C * 2;
    static constexpr int X1 = X0 + XSZ;
    static constexpr int QA = X1 + XSZ;                 // HEADS x [128][32] SW64 (q of each head)
    static constexpr int KA = QA + HEADS * 128 * 64;    // HEADS x [128][32] SW64 (k of each head)
    // v of each head (an N-major B operand); once the last P.V has read it,
    // the same bytes hold o (the projection's A operand, x tile layout) and
    // then the output rows y + bproj
    static constexpr int VA = KA + HEADS * 128 * 64;    // HEADS x [128 keys][32] SW64
    static constexpr int SMALL = VA + HEADS * 128 * 64;
    // small arrays after SMALL (byte offsets)
    static constexpr int O_BQKV = 0;                          // [3C] f32
    static constexpr int O_BPROJ = O_BQKV + 3 * C * 4;        // [C] f32
    static constexpr int O_SCALE = O_BPROJ + C * 4;           // [4] f32
    static constexpr int O_MAX = O_SCALE + 16;                // [2 heads parity][2 halves][128] f32
    static constexpr int O_PART = O_MAX + 2 * 2 * 128 * 4;    // [HEADS][2][128] f32
    // per-tile metadata, three slots (tile k in slot k % 3): the producer fills
    // tile k + 2's while the compute warps read tile k + 1's and it copies out
    // tile k's
    static constexpr int O_TOK = O_PART + HEADS * 2 * 128 * 4; // [3 slots][128] int
    static constexpr int O_ALLOW = O_TOK + 3 * 128 * 4;       // [3 slots][lo, hi][128] u32
    // [3 slots][2 windows] int4 {copy: 0 none, 1 TMA, 2 wraps; first token column;
    // first image row (b*H + i); unused}
    static constexpr int O_WIN = O_ALLOW + 3 * 2 * 128 * 4;
    static constexpr int O_BIAS = O_WIN + 3 * 2 * 16;         // [HEADS][L*L] f32, times log2(e)
    static constexpr int O_BARS = (O_BIAS + HEADS * L * L * 4 + 7) / 8 * 8;
    static constexpr int NBARS = 20;   // 0..19
    static constexpr int O_END = O_BARS + NBARS * 8 + 16;
    static constexpr int BYTES = SMALL + O_END;
    // TMEM columns: q|k|v of a tile (the next tile's while this one's heads
    // run), two 64-column S buffers, o (then y)
    static constexpr int T_QKV = 0;                     // 3C: q of head h at 32h, k at C + 32h, v at 2C + 32h
    static constexpr int T_SA = 3 * C;                  // S of even heads
    static constexpr int T_SB = T_SA + 64;              // S of odd heads
    static constexpr int T_O = T_SB + 64;               // C: o, then y
    static_assert(T_O + C <= 512, "TMEM budget");
    static_assert(M <= 8, "two windows of 8-row-aligned window rows per 128-row tile");
    // keys (and tile rows) of one window: bit 8*ki + kj for ki, kj < M
    static constexpr uint64_t FULL = M == 8 ? ~0ull : [] {
        uint64_t m = 0;
        for (int i = 0; i < M; ++i) m |= ((1ull << M) - 1ull) << (8 * i);
        return m;
    }();
    static_assert(BYTES + 1024 <= 232448, "shared memory budget");
};

struct FusedArgs {
    const bf16 *x, *Wqkv, *bqkv, *table, *Wproj, *bproj;
    const float *tau;
    bf16 *out;
    int mode;
    Geom g;
    int64_t tile_mul;   // tile visiting order: j * tile_mul mod ntiles (coprime to ntiles) ...
    int perm_step;      // ... and gridDim.x * tile_mul mod ntiles
};

// Barrier among `count` threads (named barrier `id`); returns the OR of `v`
// over them, so that a failure seen by one thread is seen by all.
template <int ID, int COUNT>
__device__ __forceinline__ bool named_sync_or(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(ID), "n"(COUNT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool compute_sync_or(bool v) { return named_sync_or<1, NCOMPUTE>(v); }
// The two compute warps of TMEM lane quarter q (the two halves of the same
// 32 rows) only: named barrier 3 + q, 64 threads.
__device__ __forceinline__ bool pair_sync_or(int q, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred t, %2, 64, p;\n\t"
        "selp.u32 %0, 1, 0, t;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(3 + q)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool producer_sync_or(bool v) { return named_sync_or<2, NPROD>(v); }

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
// writes (made visible to the async proxy by the caller where an MMA reads
// them) and TMEM loads happen before it.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

__device__ __forceinline__ uint4 pack8(const float *v, const float4 b0, const float4 b1)
{
    return make_uint4(pack_bf16x2(v[0] + b0.x, v[1] + b0.y), pack_bf16x2(v[2] + b0.z, v[3] + b0.w),
                      pack_bf16x2(v[4] + b1.x, v[5] + b1.y), pack_bf16x2(v[6] + b1.z, v[7] + b1.w));
}

__device__ __forceinline__ uint4 pack8(const float *v)
{
    return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7]));
}

template <int M, int C>
__global__ void __launch_bounds__(FBOUND_THREADS, 1)
    fused_block_kernel(FusedArgs a, DeviceStatus st, const __grid_constant__ CUtensorMap tmap_x,
                       const __grid_constant__ CUtensorMap tmap_out)
// tmap_x: x as [B*H][W][C], boxes of 32 x 8 x M; tmap_out: out as [B*H][W][C],
// boxes of 32 x M x M
{
    using F = FusedCfg<M, C>;
    constexpr int HEADS = F::HEADS, L = F::L, KB = F::KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    uint8_t *small = sm + F::SMALL;
    float *sbqkv = reinterpret_cast<float *>(small + F::O_BQKV);
    float *sbproj = reinterpret_cast<float *>(small + F::O_BPROJ);
    float *sscale = reinterpret_cast<float *>(small + F::O_SCALE);
    float *smax = reinterpret_cast<float *>(small + F::O_MAX);
    float *spart = reinterpret_cast<float *>(small + F::O_PART);
    int *stok = reinterpret_cast<int *>(small + F::O_TOK);
    uint32_t *sallow = reinterpret_cast<uint32_t *>(small + F::O_ALLOW);
    int4 *swin = reinterpret_cast<int4 *>(small + F::O_WIN);
    float *sbias = reinterpret_cast<float *>(small + F::O_BIAS);
    uint64_t *bars = reinterpret_cast<uint64_t *>(small + F::O_BARS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + F::NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);

    const Geom g = a.g;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);
    // done barriers (tcgen05.commit): the QKV issuer's (count 1) ...
    const uint32_t B_QKV = smem_u32(&bars[0]), B_Y = smem_u32(&bars[1]);
    auto B_XFREE = [&](int b) { return smem_u32(&bars[2 + b]); };       // QKV has read X(b)
    // ... and both attention issuers' (count 2)
    auto B_S = [&](int r) { return smem_u32(&bars[4 + r]); };           // S buffer r written
    const uint32_t B_O1 = smem_u32(&bars[6]);                           // P.V of every head but the last
    const uint32_t B_O = smem_u32(&bars[7]);                            // every P.V
    auto B_PVW = [&](int w) { return smem_u32(&bars[8 + w]); };         // issuer w's last P.V (count 1)
    // ready barriers (one arrival per compute warp)
    const uint32_t R_Q0 = smem_u32(&bars[10]), R_QK = smem_u32(&bars[11]), R_V = smem_u32(&bars[12]);
    auto R_P = [&](int r) { return smem_u32(&bars[13 + r]); };          // P in S buffer r
    const uint32_t R_O = smem_u32(&bars[15]);                           // o in the v tiles
    const uint32_t R_STAGE = smem_u32(&bars[16]);                       // output rows staged (v tiles)
    // producer barriers
    auto R_X = [&](int b) { return smem_u32(&bars[17 + b]); };          // x tile in X(b) (count 2)
    const uint32_t R_VFREE = smem_u32(&bars[19]);                       // output stored: v tiles free
    const int64_t ntiles = (g.nwin + 1) / 2;
    auto xbuf = [&](int buf) { return buf ? F::X1 : F::X0; };
    auto t_s = [&](int r) { return r ? F::T_SB : F::T_SA; };

    // ---- once per CTA: weights, biases, tables, barriers, TMEM ---------------
    if (warp >= CWARP0) {
        const int ct = tid - CWARP0 * 32;   // compute thread index
        for (int q = ct; q < (2 * C) * (C / 8); q += NCOMPUTE) {     // Wq, Wk rows
            const int r = q / (C / 8), c16 = q % (C / 8);
            cp_async16(base + F::WQK + (c16 >> 2) * (2 * C * 64) + sw64_offset(r, c16 & 3),
                       a.Wqkv + (int64_t)r * C + c16 * 8, 16);
        }
        for (int q = ct; q < C * (C / 8); q += NCOMPUTE) {           // Wv rows
            const int r = q / (C / 8), c16 = q % (C / 8);
            cp_async16(base + F::WV + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3),
                       a.Wqkv + (int64_t)(2 * C + r) * C + c16 * 8, 16);
        }
        for (int q = ct; q < C * (C / 8); q += NCOMPUTE) {           // Wproj
            const int r = q / (C / 8), c16 = q % (C / 8);
            cp_async16(base + F::WP + (c16 >> 2) * (C * 64) + sw64_offset(r, c16 & 3),
                       a.Wproj + (int64_t)r * C + c16 * 8, 16);
        }
        cp_async_commit();
        for (int i = ct; i < HEADS * L * L; i += NCOMPUTE) {
            const int hd = i / (L * L), e = i % (L * L);
            sbias[i] = __bfloat162float(a.table[(int64_t)e * HEADS + hd]) * FLOG2E;
        }
        for (int i = ct; i < 3 * C; i += NCOMPUTE) sbqkv[i] = a.bqkv ? __bfloat162float(a.bqkv[i]) : 0.f;
        for (int i = ct; i < C; i += NCOMPUTE) sbproj[i] = a.bproj ? __bfloat162float(a.bproj[i]) : 0.f;
        if (ct < HEADS)
            sscale[ct] = a.mode == 1 ? FLOG2E / fmaxf(a.tau[ct], 0.01f) : FLOG2E * rsqrtf(32.0f);
        // rows that no window token fills (8*ti + tj with ti or tj >= M, a
        // missing second window) start as zeros and only ever hold finite
        // values after that (o = 0, y = bproj), so their masked products are 0
        for (int i = ct; i < 2 * F::XSZ / 16; i += NCOMPUTE)
            reinterpret_cast<uint4 *>(sm + F::X0)[i] = make_uint4(0u, 0u, 0u, 0u);
        cp_async_wait<0>();
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);          // B_QKV, B_Y, B_XFREE
        for (int i = 4; i < 8; ++i) mbar_init(smem_u32(&bars[i]), 2);          // B_S, B_O1, B_O
        for (int i = 8; i < 10; ++i) mbar_init(smem_u32(&bars[i]), 1);         // B_PVW
        for (int i = 10; i < 17; ++i) mbar_init(smem_u32(&bars[i]), NCWARPS);  // R_*
        for (int i = 17; i < 19; ++i) mbar_init(smem_u32(&bars[i]), 2);        // R_X
        mbar_init(smem_u32(&bars[19]), 1);                                      // R_VFREE
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == QKV_WARP) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    const int p = tid - PWARP * 32;    // producer thread index (producer warp)
    // row -> token map (-1 for rows no token fills), the keys each row may
    // attend to (bit 8*ki + kj = key (ki, kj) of its window: the whole
    // window, or its own shift region; none for an empty row) and how each
    // window is copied, for tile `tile` into metadata slot `ms`.  (32-bit
    // arithmetic: the fused path takes grids of fewer than 2^31 tokens.)
    // Whole producer warp; lane handles rows lane + 32 i.
    auto meta = [&](int tile, int ms) {
        int bi[2], wi[2], wj[2];
        bool wvalid[2], masked[2];
        uint32_t rset[2][3], cset[2][3];   // keys' row (ki) / column (kj) sets per shift band
#pragma unroll
        for (int sl = 0; sl < 2; ++sl) {
            const int win = 2 * tile + sl;
            wvalid[sl] = win < (int)g.nwin;
            bi[sl] = wi[sl] = wj[sl] = 0;
            if (wvalid[sl]) {
                const int per = g.nh * g.nw;
                bi[sl] = win / per;
                const int rem = win - bi[sl] * per;
                wi[sl] = rem / g.nw;
                wj[sl] = rem - wi[sl] * g.nw;
            }
            masked[sl] = wvalid[sl] && g.s > 0 && (wi[sl] == g.nh - 1 || wj[sl] == g.nw - 1);
#pragma unroll
            for (int bnd = 0; bnd < 3; ++bnd) rset[sl][bnd] = cset[sl][bnd] = 0;
            if (masked[sl]) {
#pragma unroll
                for (int q = 0; q < M; ++q) {
                    const int rb = shift_band(wi[sl] * M + q, g.H, M, g.s), cb = shift_band(wj[sl] * M + q, g.W, M, g.s);
#pragma unroll
                    for (int bnd = 0; bnd < 3; ++bnd) {
                        rset[sl][bnd] |= (rb == bnd ? 1u : 0u) << q;
                        cset[sl][bnd] |= (cb == bnd ? 1u : 0u) << q;
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = p + 32 * i, sl = i >> 1, tp = r & 63, ti = tp >> 3, tj = tp & 7;
            // first shifted-frame position of the window in the original frame
            const int i0 = wi[sl] * M + g.s, j0 = wj[sl] * M + g.s;
            int tok = -1;
            uint64_t allow = 0;
            if (wvalid[sl] && ti < M && tj < M) {
                int ii = i0 + ti, jj = j0 + tj;
                if (ii >= g.H) ii -= g.H;
                if (jj >= g.W) jj -= g.W;
                tok = (bi[sl] * g.H + ii) * g.W + jj;
                if (masked[sl]) {
                    // same region = same row band and same column band
                    const int rb = shift_band(wi[sl] * M + ti, g.H, M, g.s);
                    const int cb = shift_band(wj[sl] * M + tj, g.W, M, g.s);
                    const uint32_t rs = rb == 0 ? rset[sl][0] : (rb == 1 ? rset[sl][1] : rset[sl][2]);
                    const uint64_t cs = cb == 0 ? cset[sl][0] : (cb == 1 ? cset[sl][1] : cset[sl][2]);
#pragma unroll
                    for (int ki = 0; ki < M; ++ki) allow |= (rs >> ki) & 1u ? cs << (8 * ki) : 0ull;
                } else {
                    allow = F::FULL;
                }
            }
            stok[ms * 128 + r] = tok;
            sallow[(ms * 2 + 0) * 128 + r] = (uint32_t)allow;
            sallow[(ms * 2 + 1) * 128 + r] = (uint32_t)(allow >> 32);
            // a window is one box of x unless the shift wraps it around the
            // bottom or right edge (last window row or column)
            if (tp == 0)
                swin[ms * 2 + sl] = make_int4(wvalid[sl] ? (masked[sl] ? 2 : 1) : 0, j0, bi[sl] * g.H + i0, 0);
        }
    };
    // Tiles are visited in a permuted order: the CTA's j-th tile is
    // (blockIdx.x + j*gridDim.x) * tile_mul mod ntiles, tile_mul coprime to
    // ntiles, so that every CTA gets its share of the windows on the shifted
    // edges (those cost the producer more).  perm holds the permuted index of
    // the next tile whose metadata is due; perm_step = gridDim.x * tile_mul
    // mod ntiles.
    const int nt = (int)ntiles;
    int perm = (int)(((unsigned long long)blockIdx.x * (unsigned long long)a.tile_mul) % (unsigned long long)nt);
    auto next_meta = [&](int ms) {
        meta(perm, ms);
        perm += a.perm_step;
        if (perm >= nt) perm -= nt;
    };
    if (warp == PWARP) {
        // the first three tiles' metadata, ordered before every reader by the
        // barrier below
        for (int j = 0; j < 3; ++j)
            if (blockIdx.x + (int64_t)j * gridDim.x < ntiles) next_meta(j);
    }
    tc_fence_before();
    __syncthreads();   // weights, tables, metadata of tiles 0..2, barriers, TMEM address
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == PWARP) {
        // ===================== producer warp =====================
        const bool tma_thread = p == 0;   // issues every TMA copy
        // x rows of the tile whose metadata is in slot `ms` into X(b): TMA
        // boxes and, for wrapping windows, this warp's cp.async copies (one
        // commit group); R_X(b) gets two arrivals, the TMA thread's here (with
        // the transaction bytes) and x_landed's once the cp.async copies have
        // landed
        auto load_x = [&](int b, int ms) {
            const uint32_t xb = base + xbuf(b);
            if (tma_thread) {
                const int4 w0 = swin[ms * 2], w1 = swin[ms * 2 + 1];
                const uint32_t bytes = ((w0.x == 1) + (w1.x == 1)) * KB * (M * 8 * 64);
                mbar_arrive_expect_tx(R_X(b), bytes);
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int4 w = sl ? w1 : w0;
                    if (w.x != 1) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_load_3d(xb + kb * (128 * 64) + sl * (64 * 64), &tmap_x, kb * 32, w.y, w.z, R_X(b));
                }
            }
            {
                // wrapping windows: a row per lane, its C/8 chunks
                for (int sl = 0; sl < 2; ++sl) {
                    if (swin[ms * 2 + sl].x != 2) continue;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int r = sl * 64 + lane + 32 * i;
                        const int tk = stok[ms * 128 + r];
                        if (tk < 0) continue;
                        const bf16 *src = a.x + (int64_t)tk * C;
#pragma unroll
                        for (int c16 = 0; c16 < C / 8; ++c16)
                            cp_async16(xb + (c16 >> 2) * (128 * 64) + sw64_offset(r, c16 & 3), src + c16 * 8, 16u);
                    }
                }
                cp_async_commit();
            }
        };
        auto x_landed = [&](int b) {
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(R_X(b));
        };
        bool failed = false;
        load_x(0, 0);
        x_landed(0);
        if (blockIdx.x + (int64_t)gridDim.x < ntiles) {
            load_x(1, 1);
            x_landed(1);
        }
        int k = 0;
#pragma unroll 1
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
            const int b = k & 1, ms = k % 3;
            // X(b) takes the tile two ahead as soon as this tile's QKV has read it
            if (!wait_or_abort(B_XFREE(b), (k >> 1) & 1, st.wait_ns, abort_flag)) failed = true;
            if (producer_sync_or(failed)) { failed = true; break; }
            const bool load2 = tile + 2 * (int64_t)gridDim.x < ntiles;
            if (load2) load_x(b, (k + 2) % 3);   // (its cp.async copies are waited for below)
            // this tile's output rows (in the v tiles) -> out through the window
            // reverse + roll(+s) map
            if (!wait_or_abort(R_STAGE, k & 1, st.wait_ns, abort_flag)) failed = true;
            if (producer_sync_or(failed)) { failed = true; break; }
            const uint32_t ya = base + F::VA;
            if (tma_thread) {
#pragma unroll
                for (int sl = 0; sl < 2; ++sl) {
                    const int4 w = swin[ms * 2 + sl];
                    if (w.x != 1) continue;
#pragma unroll
                    for (int kb = 0; kb < KB; ++kb)
                        tma_store_3d(&tmap_out, kb * 32, w.y, w.z, ya + kb * (128 * 64) + sl * (64 * 64));
                }
                bulk_commit();
                bulk_wait_read();   // the v tiles may be refilled once the stores have read them
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(R_VFREE);
            producer_sync_or(false);   // every read of slot ms is done
            // slot ms takes the tile three ahead
            if (tile + 3 * (int64_t)gridDim.x < ntiles) next_meta(ms);
            if (load2) x_landed(b);
        }
        cp_async_wait<0>();
        if (tma_thread) bulk_wait_all();
        if (failed) *abort_flag = 1;
    } else if (warp >= ATT_WARP0 && warp < ATT_WARP0 + 2) {
        // ============ attention issuers: S and P.V for one window's rows ============
        if (lane == 0) {
            const int w = warp - ATT_WARP0;   // 0: rows 0..63 (first window), 1: rows 64..127
            // output-lane mask: every row but this window's
            const uint32_t mask[4] = {w ? ~0u : 0u, w ? ~0u : 0u, w ? 0u : ~0u, w ? 0u : ~0u};
            const uint32_t id_s = idesc_bf16(128, 64), id_pv = idesc_bf16_bmn(128, 32);
            uint32_t ph_pvw = 0, ph_rp = 0;   // ph_rp bit r: phase of R_P(r)
            // S of head hd for this window's rows: all 128 q rows against this
            // window's 64 keys
            auto issue_s = [&](int hd) {
                const uint32_t d = tmem + t_s(hd & 1);
                const uint32_t qa = base + F::QA + hd * 8192, ka = base + F::KA + hd * 8192 + w * 4096;
#pragma unroll
                for (int ks = 0; ks < 2; ++ks)
                    mma_bf16_mask(d, desc_kmajor_sw64(qa + 32 * ks), desc_kmajor_sw64(ka + 32 * ks), id_s, ks, mask);
                mma_commit(B_S(hd & 1));
            };
            // o_h += P v_h over this window's 64 keys, for its rows
            auto issue_pv = [&](int hd) {
                const uint32_t pa = tmem + t_s(hd & 1), va = base + F::VA + hd * 8192 + w * 4096;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts_mask(tmem + F::T_O + 32 * hd, pa + 8 * kk, desc_mnmajor_sw64(va + 1024 * kk, 8192),
                                     id_pv, kk, mask);
                mma_commit(B_PVW(w));
                if (hd == HEADS - 2) mma_commit(B_O1);
                if (hd == HEADS - 1) mma_commit(B_O);
            };
            bool ok = true;
            int k = 0;
#pragma unroll 1
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
                // S of head 0 once its q and k are drained, of head 1 once every
                // head's are; P.V of head h once its P is in TMEM (head 0: and
                // every v drained); S of head h + 2 once this issuer's P.V h has
                // read P out of that buffer
                if (!(ok = wait_or_abort(R_Q0, k & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                issue_s(0);
                if (HEADS > 1) {
                    if (!(ok = wait_or_abort(R_QK, k & 1, st.wait_ns, abort_flag))) break;
                    tc_fence_after();
                    issue_s(1);
                }
#pragma unroll 1
                for (int hd = 0; hd < HEADS; ++hd) {
                    const int r = hd & 1;
                    if (!(ok = wait_or_abort(R_P(r), (ph_rp >> r) & 1u, st.wait_ns, abort_flag))) break;
                    ph_rp ^= 1u << r;
                    if (hd == 0 && !(ok = wait_or_abort(R_V, k & 1, st.wait_ns, abort_flag))) break;
                    tc_fence_after();
                    issue_pv(hd);
                    if (!(ok = wait_or_abort(B_PVW(w), ph_pvw, st.wait_ns, abort_flag))) break;
                    ph_pvw ^= 1;
                    if (hd + 2 < HEADS) issue_s(hd + 2);
                }
                if (!ok) break;
            }
        }
    } else if (warp == QKV_WARP) {
        // ============ QKV issuer: the next tile's QKV, this tile's projection ============
        if (lane == 0) {
            const uint32_t id_qk = idesc_bf16(128, 2 * C), id_v = idesc_bf16(128, C), id_y = idesc_bf16(128, C);
            auto issue_qkv = [&](int buf) {
                const uint32_t xb = base + xbuf(buf);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_QKV, desc_kmajor_sw64(xb + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(base + F::WQK + kb * (2 * C * 64) + 32 * ks), id_qk, (kb | ks) != 0);
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_QKV + 2 * C, desc_kmajor_sw64(xb + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(base + F::WV + kb * (C * 64) + 32 * ks), id_v, (kb | ks) != 0);
                mma_commit(B_QKV);
                mma_commit(B_XFREE(buf));
            };
            bool ok = wait_or_abort(R_X(0), 0, st.wait_ns, abort_flag);
            if (ok) {
                tc_fence_after();
                issue_qkv(0);
            }
            int k = 0;
#pragma unroll 1
            for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++k) {
                const int buf = k & 1;
                // the next tile's QKV once this tile's q, k and v have left TMEM
                // and the next x has landed
                if (tile + gridDim.x < ntiles) {
                    if (!(ok = wait_or_abort(R_V, k & 1, st.wait_ns, abort_flag))) break;
                    if (!(ok = wait_or_abort(R_X(buf ^ 1), ((k + 1) >> 1) & 1, st.wait_ns, abort_flag))) break;
                    tc_fence_after();
                    issue_qkv(buf ^ 1);
                }
                // the projection once o is in the v tiles
                if (!(ok = wait_or_abort(R_O, k & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                const uint32_t oa = base + F::VA;
#pragma unroll
                for (int kb = 0; kb < KB; ++kb)
#pragma unroll
                    for (int ks = 0; ks < 2; ++ks)
                        mma_bf16(tmem + F::T_O, desc_kmajor_sw64(oa + kb * (128 * 64) + 32 * ks),
                                 desc_kmajor_sw64(base + F::WP + kb * (C * 64) + 32 * ks), id_y, (kb | ks) != 0);
                mma_commit(B_Y);
            }
        }
    } else {
        // ===================== compute warps =====================
        const int quarter = warp & 3, half = (warp >> 2) - 1;
        const int row = quarter * 32 + lane;       // tile row = TMEM lane
        const int slot = row >> 6, t = row & 63;   // window slot; token (t >> 3, t & 7) of the row
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        // relative-bias row of this token (empty rows read a valid row, then are masked)
        const int ti = t >> 3, tj = t & 7;
        const int bias_base = ti < M && tj < M ? (ti + M - 1) * L + (tj + M - 1) : (M - 1) * L + (M - 1);
        uint32_t ph_s = 0;   // bit r: phase of B_S(r)
        bool failed = false;
        int k = 0;
#pragma unroll 1
        for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
            // this tile's QKV is done.  (Its metadata -- masks -- was written
            // before the CTA-wide barrier for tiles 0..2, and three tiles ahead
            // before the producer's R_VFREE arrival, which is waited below
            // before the masks are read, for the others.)
            if (!wait_or_abort(B_QKV, k & 1, st.wait_ns, abort_flag)) failed = true;
            tc_fence_after();

            // q (half 0) or k (half 1) of every head to shared memory
#pragma unroll 1
            for (int hd = 0; hd < HEADS; ++hd) {
                const int col = half == 0 ? hd * 32 : C + hd * 32;
                float v[32];
                tmem_ld32(t_lane + F::T_QKV + col, v);
                tmem_wait_ld();
                const float4 *b4 = reinterpret_cast<const float4 *>(sbqkv + col);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 bb = b4[e4];
                    v[4 * e4] += bb.x;
                    v[4 * e4 + 1] += bb.y;
                    v[4 * e4 + 2] += bb.z;
                    v[4 * e4 + 3] += bb.w;
                }
                if (a.mode == 1) {
                    float ss = 0.f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss = fmaf(v[e], v[e], ss);
                    const float inv = 1.0f / fmaxf(sqrtf(ss), 1e-12f);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= inv;
                }
                uint8_t *dst = sm + (half == 0 ? F::QA : F::KA) + hd * 8192;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(dst + sw64_offset(row, c)) = pack8(v + 8 * c);
                if (hd == 0 || hd == HEADS - 1) {
                    fence_proxy_async_smem();
                    warp_arrive(hd == 0 ? R_Q0 : R_QK, lane);
                }
            }
            // v drain: this half's C/2 channels of the row's token -> key row
            // `row` of each head's v tile (the N-major B operand of P.V), once
            // the previous tile's output rows have left those bytes
            if (k > 0 && !wait_or_abort(R_VFREE, (k - 1) & 1, st.wait_ns, abort_flag)) failed = true;
            {
                constexpr int HC = C / 2;
#pragma unroll
                for (int c0 = 0; c0 < HC; c0 += 16) {
                    float v[16];
                    tmem_ld16(t_lane + F::T_QKV + 2 * C + half * HC + c0, v);
                    tmem_wait_ld();
                    const float4 *b4 = reinterpret_cast<const float4 *>(sbqkv + 2 * C + half * HC + c0);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int ch = (half * HC + c0) / 8 + c;   // 8-channel chunk of v
                        *reinterpret_cast<uint4 *>(sm + F::VA + (ch >> 2) * 8192 + sw64_offset(row, ch & 3)) =
                            pack8(v + 8 * c, b4[2 * c], b4[2 * c + 1]);
                    }
                }
            }
            fence_proxy_async_smem();
            warp_arrive(R_V, lane);

            const int ms = k % 3;
            const uint32_t allow_lo = sallow[(ms * 2 + 0) * 128 + row];
            const uint32_t allow_hi = sallow[(ms * 2 + 1) * 128 + row];
            const bool row_ok = (allow_lo | allow_hi) != 0;   // a real token always sees itself
            const uint32_t allow = half == 0 ? allow_lo : allow_hi;

#pragma unroll 1
            for (int hd = 0; hd < HEADS; ++hd) {
                const int r = hd & 1;
                if (!wait_or_abort(B_S(r), (ph_s >> r) & 1u, st.wait_ns, abort_flag)) failed = true;
                ph_s ^= 1u << r;
                tc_fence_after();

                // ---- softmax over this row's own window, keys 32*half .. +31 -------
                float s[32];
                tmem_ld32(t_lane + t_s(r) + 32 * half, s);
                tmem_wait_ld();
                const float scale = sscale[hd];
                const float *bias = sbias + hd * L * L + bias_base;
                float mx = -INFINITY;
                // key column j = 8*ki + kj of the row's window: relative-bias row
                // bias_base - (ki*L + kj); j is a compile-time constant in each
                // unrolled loop, and columns with ki or kj >= M hold no key
                if (half == 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if ((j >> 3) < M && (j & 7) < M) {
                            const float v = fmaf(s[j], scale, bias[-((j >> 3) * L + (j & 7))]);
                            s[j] = (allow >> j) & 1u ? v : -INFINITY;
                        } else {
                            s[j] = -INFINITY;
                        }
                        mx = fmaxf(mx, s[j]);
                    }
                } else {
#pragma unroll
                    for (int j = 32; j < 64; ++j) {
                        if ((j >> 3) < M && (j & 7) < M) {
                            const float v = fmaf(s[j - 32], scale, bias[-((j >> 3) * L + (j & 7))]);
                            s[j - 32] = (allow >> (j - 32)) & 1u ? v : -INFINITY;
                        } else {
                            s[j - 32] = -INFINITY;
                        }
                        mx = fmaxf(mx, s[j - 32]);
                    }
                }
                float *mxb = smax + r * 256;
                mxb[half * 128 + row] = mx;
                // only the other half of the same rows is waited for; a failure
                // stays local to the pair until the compute-wide barrier after
                // the heads (every wait returns at once after an abort)
                if (pair_sync_or(quarter, failed)) failed = true;
                mx = row_ok ? fmaxf(mxb[row], mxb[128 + row]) : 0.f;   // padding rows: all -inf -> p = 0
                float sum = 0.f;
                uint32_t pk[16];
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const float p0 = ex2_approx(s[jj] - mx), p1 = ex2_approx(s[jj + 1] - mx);
                    sum += p0 + p1;
                    pk[jj / 2] = pack_bf16x2(p0, p1);
                }
                spart[(hd * 2 + half) * 128 + row] = sum;
                // P (bf16, two keys per 32-bit column) over the first 32 columns of
                // this S buffer, the A operand of the P.V MMA pair
                tmem_st16(t_lane + t_s(r) + 16 * half, pk);
                tmem_wait_st();
                warp_arrive(R_P(r), lane);
            }
            // (a failure above is not uniform across threads yet: the barriers
            // below make every compute thread leave together; waits return at
            // once after an abort)
            // ---- o / rowsum -> bf16 -> the v tiles (A operand of the projection):
            // every head but the last as soon as its P.V is done, then the last ----
            auto drain_o = [&](int hd) {
                float o[16];
                tmem_ld16(t_lane + F::T_O + 32 * hd + 16 * half, o);
                tmem_wait_ld();
                const float l = spart[(hd * 2) * 128 + row] + spart[(hd * 2 + 1) * 128 + row];
                const float inv = row_ok ? rcp_approx(l) : 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] *= inv;
                uint8_t *dst = sm + F::VA + hd * (128 * 64);
#pragma unroll
                for (int c = 0; c < 2; ++c)
                    *reinterpret_cast<uint4 *>(dst + sw64_offset(row, 2 * half + c)) = pack8(o + 8 * c);
            };
            if (!wait_or_abort(B_O1, k & 1, st.wait_ns, abort_flag)) failed = true;
            if (compute_sync_or(failed)) { failed = true; break; }   // also orders spart
            tc_fence_after();
#pragma unroll 1
            for (int hd = 0; hd < HEADS - 1; ++hd) drain_o(hd);
            if (!wait_or_abort(B_O, k & 1, st.wait_ns, abort_flag)) failed = true;
            if (compute_sync_or(failed)) { failed = true; break; }
            tc_fence_after();
            drain_o(HEADS - 1);
            fence_proxy_async_smem();
            warp_arrive(R_O, lane);
            if (!wait_or_abort(B_Y, k & 1, st.wait_ns, abort_flag)) failed = true;
            tc_fence_after();

            // ---- y + bproj -> bf16 rows in the v tiles, token (ti, tj) of a window at
            // row M*ti + tj of its half (one dense box per window for the TMA
            // store through the window reverse + roll(+s) map) ----
            {
                constexpr int HC = C / 2;
                uint8_t *stage = sm + F::VA;
                const bool tok_row = ti < M && tj < M;
                const int srow = slot * 64 + ti * M + tj;
                // rows of a window that the shift wraps around the image edge are
                // stored straight to out (the TMA store takes the others)
                const int ytok = swin[ms * 2 + slot].x == 2 ? stok[ms * 128 + row] : -1;
#pragma unroll
                for (int c0 = 0; c0 < HC; c0 += 16) {
                    float y[16];
                    tmem_ld16(t_lane + F::T_O + half * HC + c0, y);
                    tmem_wait_ld();
                    const float4 *bp = reinterpret_cast<const float4 *>(sbproj + half * HC + c0);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int chunk = (half * HC + c0) / 8 + c;
                        const uint4 pk8 = pack8(y + 8 * c, bp[2 * c], bp[2 * c + 1]);
                        if (ytok >= 0)
                            *reinterpret_cast<uint4 *>(a.out + (int64_t)ytok * C + chunk * 8) = pk8;
                        else if (tok_row)
                            *reinterpret_cast<uint4 *>(stage + (chunk >> 2) * (128 * 64) + sw64_offset(srow, chunk & 3)) = pk8;
                    }
                }
            }
            fence_proxy_async_smem();   // the TMA stores read these rows
            warp_arrive(R_STAGE, lane);
        }
        if (failed) *abort_flag = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(st.err, ERR_TIMEOUT);
    if (warp == QKV_WARP) {
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

// Smallest v >= start (and >= 1) with gcd(v, n) == 1.
int64_t coprime_near(int64_t n, int64_t start)
{
    auto gcd = [](int64_t x, int64_t y) {
        while (y) {
            const int64_t t = x % y;
            x = y;
            y = t;
        }
        return x;
    };
    if (n <= 1) return 1;
    for (int64_t v = start < 1 ? 1 : start;; ++v)
        if (gcd(v, n) == 1) return v % n ? v : 1;
}

template <int M, int C>
cudaError_t launch_fused_t(const FusedArgs &a, DeviceStatus st, cudaStream_t stream)
{
    using F = FusedCfg<M, C>;
    const size_t smem = F::BYTES + 1024;
    auto kern = fused_block_kernel<M, C>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tx, to;
    e = make_tensor_map_sw64_3d(&tx, a.x, (int64_t)a.g.B * a.g.H, a.g.W, C, 8, M);
    if (e != cudaSuccess) return e;
    e = make_tensor_map_sw64_3d(&to, a.out, (int64_t)a.g.B * a.g.H, a.g.W, C, M, M);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.g.nwin + 1) / 2;
    const int grid = (int)(ntiles < num_sms() ? ntiles : num_sms());
    FusedArgs b = a;
    b.tile_mul = coprime_near(ntiles, (ntiles * 5) / 8 + 1);
    b.perm_step = (int)(((unsigned long long)grid * (unsigned long long)b.tile_mul) % (unsigned long long)ntiles);
    kern<<<grid, FTHREADS, smem, stream>>>(b, st, tx, to);
    return cudaGetLastError();
}

} // namespace

bool fused_supported(int M, int C, int heads)
{
    return (M == 7 || M == 8) && (C == 64 || C == 96) && C == heads * 32;
}

cudaError_t launch_fused(const bf16 *x, const bf16 *Wqkv, const bf16 *bqkv, const bf16 *table, const float *tau,
                         const bf16 *Wproj, const bf16 *bproj, bf16 *out, int mode, const Geom &g, DeviceStatus st,
                         cudaStream_t stream)
{
    FusedArgs a{x, Wqkv, bqkv, table, Wproj, bproj, tau, out, mode, g, 1, 0};
    if (g.M == 7 && g.C == 96) return launch_fused_t<7, 96>(a, st, stream);
    if (g.M == 8 && g.C == 96) return launch_fused_t<8, 96>(a, st, stream);
    if (g.M == 7 && g.C == 64) return launch_fused_t<7, 64>(a, st, stream);
    if (g.M == 8 && g.C == 64) return launch_fused_t<8, 64>(a, st, stream);
    return cudaErrorInvalidValue;
}

} // namespace swin
