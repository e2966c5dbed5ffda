// The fused shifted-window attention block kernel (fused_block.cuh): path
// choice and launches of its plain variants; the variants with the block's
// LayerNorm and residual folded in are in fused_block_fold.cu.
#include "fused_block.cuh"

namespace swin {

bool fused_supported(int M, int C, int heads)
{
    return (M == 7 || M == 8) && (C == 64 || C == 96 || C == 128) && C == heads * 32;
}

bool fused_fold_supported(int M, int C, int heads, int fold)
{
    // (C = 128 splits a row's y over two warps: no in-thread post-norm there)
    return fused_supported(M, C, heads) && fold >= 0 && fold <= 2 && !(fold == 2 && C == 128);
}

cudaError_t launch_fused(const bf16 *x, const bf16 *Wqkv, const bf16 *bqkv, const bf16 *table, const float *tau,
                         const bf16 *Wproj, const bf16 *bproj, bf16 *out, int mode, const Geom &g, DeviceStatus st,
                         int *sched, cudaStream_t stream, const bf16 *ln_g, const bf16 *ln_b, int fold, int overlap)
{
    if (!sched) return cudaErrorInvalidValue;
    if (fold && (!ln_g || !ln_b || !fused_fold_supported(g.M, g.C, g.C / 32, fold))) return cudaErrorInvalidValue;
    FusedArgs a{x, Wqkv, bqkv, table, Wproj, bproj, tau, out, mode, g, sched, ln_g, ln_b, fold, overlap};
    if (fold) return launch_fused_folded(a, st, stream);
    if (g.M == 7 && g.C == 96) return launch_fused_t<7, 96, 2, 0>(a, st, stream);
    if (g.M == 8 && g.C == 96) return launch_fused_t<8, 96, 2, 0>(a, st, stream);
    if (g.M == 7 && g.C == 64) return launch_fused_t<7, 64, 2, 0>(a, st, stream);
    if (g.M == 8 && g.C == 64) return launch_fused_t<8, 64, 2, 0>(a, st, stream);
    if (g.M == 7 && g.C == 128) return launch_fused_t<7, 128, 1, 0>(a, st, stream);
    if (g.M == 8 && g.C == 128) return launch_fused_t<8, 128, 1, 0>(a, st, stream);
    return cudaErrorInvalidValue;
}

} // namespace swin
