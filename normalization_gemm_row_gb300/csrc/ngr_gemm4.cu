// ngr_gemm4.cu -- instantiations and launch of the multicast cluster
// kernel (ngr_gemm4_kernel.cuh): LayerNorm, RMSNorm, no norm or a folded
// weight (LayerNorm or RMSNorm), fp16 or bf16.
#include "ngr_gemm4_kernel.cuh"

namespace ngr {

int launch_gemm4(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl, cudaStream_t stream)
{
    if (norm == kNormLayer)
        return bf16 ? launch_gemm4_variant<kNormLayer, true>(args, grid, pdl, stream)
                    : launch_gemm4_variant<kNormLayer, false>(args, grid, pdl, stream);
    if (norm == kNormRms)
        return bf16 ? launch_gemm4_variant<kNormRms, true>(args, grid, pdl, stream)
                    : launch_gemm4_variant<kNormRms, false>(args, grid, pdl, stream);
    if (norm == kNormNone)
        return bf16 ? launch_gemm4_variant<kNormNone, true>(args, grid, pdl, stream)
                    : launch_gemm4_variant<kNormNone, false>(args, grid, pdl, stream);
    if (norm == kNormFoldLayer)
        return bf16 ? launch_gemm4_variant<kNormFoldLayer, true>(args, grid, pdl, stream)
                    : launch_gemm4_variant<kNormFoldLayer, false>(args, grid, pdl, stream);
    if (norm == kNormFoldRms)
        return bf16 ? launch_gemm4_variant<kNormFoldRms, true>(args, grid, pdl, stream)
                    : launch_gemm4_variant<kNormFoldRms, false>(args, grid, pdl, stream);
    return -9;
}

int gemm4_clusters() { return gemm4_max_clusters(); }

size_t gemm4_smem_bytes() { return Gemm4Smem::alloc; }

}  // namespace ngr
