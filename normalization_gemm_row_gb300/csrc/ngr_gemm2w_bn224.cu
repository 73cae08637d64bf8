// ngr_gemm2w_bn224.cu -- CTA-pair tile kernel instantiations for a 256 x 448
// output tile made of two 224-column sub-tiles that share each x stage
// (5 pipeline stages, one accumulator).
#include "ngr_gemm2_kernel.cuh"

namespace ngr {

int launch_gemm2w_bn224(int norm, bool bf16, const GemmArgs &args, int grid,
                       bool pdl, cudaStream_t stream)
{
    return launch_gemm2_bn<224, 5, 2>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm2w_smem_bn224() { return Gemm2Smem<224, 5, 2>::alloc; }
int gemm2w_max_clusters_bn224() { return gemm2_max_clusters<224, 5, 2>(); }

}  // namespace ngr
