// ngr_gemm2_bn224.cu -- CTA-pair tile kernel instantiations for a 224-column
// N tile (7 pipeline stages).  One translation unit per tile width so they
// compile in parallel.
#include "ngr_gemm2_kernel.cuh"

namespace ngr {

int launch_gemm2_bn224(int norm, bool bf16, const GemmArgs &args, int grid,
                      bool pdl, cudaStream_t stream)
{
    return launch_gemm2_bn<224, 7, 1>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm2_smem_bn224() { return Gemm2Smem<224, 7, 1>::alloc; }
int gemm2_max_clusters_bn224() { return gemm2_max_clusters<224, 7, 1>(); }

}  // namespace ngr
