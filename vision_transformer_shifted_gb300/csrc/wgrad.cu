// Weight and bias gradients of the attention block's two projections on
// tcgen05:
//   dW[o][i] = sum over tokens t of G[t][o] * X[t][i],  db[o] = sum_t G[t][o]
// (dWproj = dy^T attn, dWqkv = dqkv^T x; G [T, n_out], X [T, n_in], both
// bf16 row-major, dW fp32 [n_out, n_in]).  The pages' training path runs the
// block's backward ("Boosting Swin Transformer Speed", Training Optimization);
// the sums over the 200 K tokens of a batch are plain long-K reductions, and
// the order of the tokens does not matter to them, so G and X are read as
// they are (no gather).
//
// As an MMA: D[m][n] = sum_k A[m][k] B[n][k] with m = o, n = i, k = t; both
// operands arrive MN-major (A[m][k] = G[k][m]: the 32 o of a row of G are
// contiguous), as 2-D TMA boxes of 32 columns x 64 tokens (64-byte swizzle)
// and are used as they land.  A CTA holds MT x 128 rows of o times NT columns
// of i in TMEM (MT accumulators of 128 x (NT + 32), at most 512 columns) and
// sums the tokens of its share of the batch (split-K).  The last 32 columns
// of every accumulator multiply G by a constant tile of ones (written once
// into every stage, never loaded), so that column NT is db.  Each CTA writes
// its fp32 partial block to a workspace, and two small kernels add the
// partials in a fixed order (the result does not depend on scheduling).
#include "common.cuh"
#include "ptx.cuh"

namespace swin {

namespace {

constexpr int WG_BK = 64;                  // tokens per stage
constexpr int WG_STAGES = 3;
constexpr int WG_THREADS = 6 * 32;         // producer, MMA issuer, four drain warps
constexpr int WG_BOX = WG_BK * 64;         // one 32-column box: 64 rows of 64 bytes

struct WgPlan {
    int MT, NT;           // m tiles of 128 per CTA, columns of i per CTA
    int tiles_m, tiles_n; // CTA blocks over o and i
    int splits;           // token ranges (split-K)
    int chunks;           // BK-token chunks of the whole batch
    int stage_bytes;
};

struct WgArgs {
    int n_out, n_in;
    int64_t T;
    float *partial;       // [splits][n_tot]: dW (n_out x n_in), then db (n_out), then padding
    int64_t n_tot;
};

__device__ __forceinline__ bool wg_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns, volatile int *abort)
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

__global__ void __launch_bounds__(WG_THREADS, 1)
    wgrad_kernel(WgArgs a, WgPlan pl, DeviceStatus st, const __grid_constant__ CUtensorMap tmap_g,
                 const __grid_constant__ CUtensorMap tmap_x)
// tmap_g: G [T, n_out], tmap_x: X [T, n_in]; boxes of 32 columns x 64 rows, SW64
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = smem_align(smem_raw, 1024);
    const int MT = pl.MT, NT = pl.NT, SB = pl.stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + WG_STAGES * SB);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * WG_STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t base = smem_u32(sm);
    auto FULL = [&](int s) { return smem_u32(&bars[s]); };
    auto EMPTY = [&](int s) { return smem_u32(&bars[WG_STAGES + s]); };
    const uint32_t DONE = smem_u32(&bars[2 * WG_STAGES]);
    // this CTA's block of dW and token chunks
    const int blk = blockIdx.x % (pl.tiles_m * pl.tiles_n), split = blockIdx.x / (pl.tiles_m * pl.tiles_n);
    const int o0 = (blk / pl.tiles_n) * MT * 128, i0 = (blk % pl.tiles_n) * NT;
    const int per = (pl.chunks + pl.splits - 1) / pl.splits;
    const int c_begin = split * per, c_end = min(pl.chunks, c_begin + per);
    const int nch = c_end > c_begin ? c_end - c_begin : 0;
    const int a_bytes = MT * 4 * WG_BOX;   // A of a stage: MT x 4 groups of 32 o
    const int NB = NT + 32;                // B columns: NT of X, then 32 of ones

    // the ones group of every stage (bf16 1.0 = 0x3F80)
    for (int s = 0; s < WG_STAGES; ++s)
        for (int q = tid; q < WG_BOX / 16; q += WG_THREADS)
            reinterpret_cast<uint4 *>(sm + s * SB + a_bytes + (NT / 32) * WG_BOX)[q] =
                make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    fence_proxy_async_smem();
    if (tid == 0) {
        for (int s = 0; s < WG_STAGES; ++s) {
            mbar_init(FULL(s), 1);
            mbar_init(EMPTY(s), 1);
        }
        mbar_init(DONE, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // (the prologue touched no global memory: G and X are read, and the partial
    // sums written, only after the kernels queued before this one complete; a
    // no-op unless launched to overlap them)
    griddep_launch_dependents();
    griddep_wait();
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
#pragma unroll 1
            for (int j = 0; j < nch; ++j) {
                const int s = j % WG_STAGES;
                if (j >= WG_STAGES && !(ok = wg_wait(EMPTY(s), ((j / WG_STAGES) - 1) & 1, st.wait_ns, abort_flag)))
                    break;
                const uint32_t sa = base + s * SB, sb = sa + a_bytes;
                const int t0 = (c_begin + j) * WG_BK;
                mbar_arrive_expect_tx(FULL(s), (uint32_t)(a_bytes + (NT / 32) * WG_BOX));
                for (int g4 = 0; g4 < MT * 4; ++g4)   // (columns past n_out arrive as zeros)
                    tma_load_2d(sa + g4 * WG_BOX, &tmap_g, o0 + 32 * g4, t0, FULL(s));
                for (int g4 = 0; g4 < NT / 32; ++g4) tma_load_2d(sb + g4 * WG_BOX, &tmap_x, i0 + 32 * g4, t0, FULL(s));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = idesc_bf16_amn_bmn(128, NB);
#pragma unroll 1
            for (int j = 0; j < nch; ++j) {
                const int s = j % WG_STAGES;
                if (!(ok = wg_wait(FULL(s), (j / WG_STAGES) & 1, st.wait_ns, abort_flag))) break;
                tc_fence_after();
                const uint32_t sa = base + s * SB, sb = sa + a_bytes;
                // A: m tile mt = groups 4 mt .. 4 mt + 3, 32 o each at a stride of one
                // box; 16 tokens a K step (1024 bytes of each box)
                for (int ks = 0; ks < WG_BK / 16; ++ks) {
                    const uint64_t db = desc_mnmajor_sw64(sb + ks * 1024, WG_BOX);
                    for (int mt = 0; mt < MT; ++mt)
                        mma_bf16(tmem + mt * NB, desc_mnmajor_sw64(sa + mt * 4 * WG_BOX + ks * 1024, WG_BOX), db, id,
                                 (j | ks) != 0);
                }
                mma_commit(EMPTY(s));
            }
            mma_commit(DONE);
        }
    } else {
        // drain: warp w serves TMEM lanes 32 (w % 4) .. + 31 = o rows of every m tile
        const int quarter = warp & 3;
        const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
        ok = wg_wait(DONE, 0, st.wait_ns, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        if (ok) {
            for (int mt = 0; mt < MT; ++mt) {
                const int o = o0 + mt * 128 + quarter * 32 + lane;
                float *prow = a.partial + (int64_t)split * a.n_tot + (int64_t)o * a.n_in + i0;
                for (int c = 0; c < NT; c += 32) {
                    float v[32];
                    tmem_ld32(t_lane + mt * NB + c, v);
                    tmem_wait_ld();
                    if (o < a.n_out) {
                        float4 *dst = reinterpret_cast<float4 *>(prow + c);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = nch ? make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3])
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                if (i0 == 0) {   // db from the first block of i
                    float v[8];
                    tmem_ld8(t_lane + mt * NB + NT, v);
                    tmem_wait_ld();
                    if (o < a.n_out)
                        a.partial[(int64_t)split * a.n_tot + (int64_t)a.n_out * a.n_in + o] = nch ? v[0] : 0.f;
                }
            }
        }
    }
    if (!ok) *abort_flag = 1;
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && *abort_flag) atomicOr(st.err, ERR_TIMEOUT);
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, 512);
    }
}

// Level 1: part1[y][e] = sum of partial[s][e] over s = y, y + RS, ... (in order).
__global__ void wgrad_reduce1_kernel(const float *partial, int splits, int RS, int64_t n_tot, float *part1)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y;
    if (i4 * 4 >= n_tot) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = y; s < splits; s += RS) {
        const float4 v = reinterpret_cast<const float4 *>(partial + (int64_t)s * n_tot)[i4];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    reinterpret_cast<float4 *>(part1 + (int64_t)y * n_tot)[i4] = acc;
}

// Level 2: the RS level-1 sums in order, into dW (the first n_w entries) and db.
__global__ void wgrad_reduce2_kernel(const float *part1, int RS, int64_t n_w, int n_b, float *dW, float *db)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= n_w + n_b) return;
    const int64_t n_tot = ((n_w + n_b + 3) / 4) * 4;
    float acc = 0.f;
    for (int y = 0; y < RS; ++y) acc += part1[(int64_t)y * n_tot + e];
    if (e < n_w)
        dW[e] = acc;
    else if (db)
        db[e - n_w] = acc;
}

int wg_num_sms()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    }
    return n;
}

bool wg_plan(int n_out, int n_in, int64_t T, WgPlan &p)
{
    if (n_out <= 0 || n_in <= 0 || n_in % 32 || T <= 0) return false;
    int NT = 0;
    for (int nt = 224; nt >= 32; nt -= 32)
        if (n_in % nt == 0) {
            NT = nt;
            break;
        }
    if (!NT) return false;
    const int mtiles = (n_out + 127) / 128;
    p.NT = NT;
    p.MT = 512 / (NT + 32) < mtiles ? 512 / (NT + 32) : mtiles;
    // (shared memory: three stages of MT x 4 + NT / 32 + 1 boxes of 4 KB)
    while (p.MT > 1 && WG_STAGES * (p.MT * 4 + NT / 32 + 1) * WG_BOX > 200 * 1024) --p.MT;
    p.tiles_m = (mtiles + p.MT - 1) / p.MT;
    p.tiles_n = n_in / NT;
    p.chunks = (int)((T + WG_BK - 1) / WG_BK);
    const int blocks = p.tiles_m * p.tiles_n, sms = wg_num_sms();
    p.splits = sms / blocks > 1 ? sms / blocks : 1;
    if (p.splits > p.chunks) p.splits = p.chunks;
    p.stage_bytes = (p.MT * 4 + NT / 32 + 1) * WG_BOX;
    return true;
}

} // namespace

static int64_t wg_ntot(int n_out, int n_in) { return (((int64_t)n_out * n_in + n_out + 3) / 4) * 4; }
static int wg_rs(const WgPlan &p) { return p.splits < 16 ? p.splits : 16; }

size_t wgrad_workspace_bytes(int n_out, int n_in, int64_t T)
{
    WgPlan p;
    if (!wg_plan(n_out, n_in, T, p)) return 0;
    return (size_t)(p.splits + wg_rs(p)) * wg_ntot(n_out, n_in) * sizeof(float);
}

cudaError_t launch_wgrad(const bf16 *G, int n_out, const bf16 *X, int n_in, int64_t T, float *dW, float *db,
                         float *workspace, DeviceStatus st, cudaStream_t stream, int overlap)
{
    WgPlan p;
    if (!wg_plan(n_out, n_in, T, p) || T >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
    CUtensorMap tg, tx;
    cudaError_t e = make_tensor_map_sw64(&tg, G, T, n_out, WG_BK, true);
    if (e != cudaSuccess) return e;
    e = make_tensor_map_sw64(&tx, X, T, n_in, WG_BK, true);
    if (e != cudaSuccess) return e;
    const size_t smem = 1024 + (size_t)WG_STAGES * p.stage_bytes + (2 * WG_STAGES + 1) * 8 + 16;
    e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t n_tot = wg_ntot(n_out, n_in);
    WgArgs a{n_out, n_in, T, workspace, n_tot};
    e = launch_maybe_overlapped(wgrad_kernel, dim3(p.tiles_m * p.tiles_n * p.splits), dim3(WG_THREADS), smem, stream,
                                overlap, a, p, st, tg, tx);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    const int RS = wg_rs(p);
    float *part1 = workspace + (int64_t)p.splits * n_tot;
    e = launch_maybe_overlapped(wgrad_reduce1_kernel, dim3((unsigned)((n_tot / 4 + 255) / 256), (unsigned)RS),
                                dim3(256), 0, stream, overlap, (const float *)workspace, p.splits, RS, n_tot, part1);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t n = (int64_t)n_out * n_in + n_out;
    e = launch_maybe_overlapped(wgrad_reduce2_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, overlap,
                                (const float *)part1, RS, (int64_t)n_out * n_in, n_out, dW, db);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

} // namespace swin
