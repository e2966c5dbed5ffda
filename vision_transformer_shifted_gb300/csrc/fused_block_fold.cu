// The fused block kernel (fused_block.cuh) with the transformer block's
// LayerNorm and residual folded in ("Swin Transformer V2" (neura.market), How
// It Works: pre-norm in the original Swin, residual post-norm in V2): a
// translation unit of its own, so that it builds beside the plain variants.
#include "fused_block.cuh"

namespace swin {

cudaError_t launch_fused_folded(const FusedArgs &a, DeviceStatus st, cudaStream_t stream)
{
    const Geom &g = a.g;
    if (a.fold == 1) {
        if (g.M == 7 && g.C == 96) return launch_fused_t<7, 96, 2, 1>(a, st, stream);
        if (g.M == 8 && g.C == 96) return launch_fused_t<8, 96, 2, 1>(a, st, stream);
        if (g.M == 7 && g.C == 64) return launch_fused_t<7, 64, 2, 1>(a, st, stream);
        if (g.M == 8 && g.C == 64) return launch_fused_t<8, 64, 2, 1>(a, st, stream);
        if (g.M == 7 && g.C == 128) return launch_fused_t<7, 128, 1, 1>(a, st, stream);
        if (g.M == 8 && g.C == 128) return launch_fused_t<8, 128, 1, 1>(a, st, stream);
    } else if (a.fold == 2) {
        if (g.M == 7 && g.C == 96) return launch_fused_t<7, 96, 2, 2>(a, st, stream);
        if (g.M == 8 && g.C == 96) return launch_fused_t<8, 96, 2, 2>(a, st, stream);
        if (g.M == 7 && g.C == 64) return launch_fused_t<7, 64, 2, 2>(a, st, stream);
        if (g.M == 8 && g.C == 64) return launch_fused_t<8, 64, 2, 2>(a, st, stream);
    }
    return cudaErrorInvalidValue;
}

} // namespace swin
