// ngr_gemm2_bn128.cu -- CTA-pair tile kernel instantiations for a 128-column
// N tile (8 pipeline stages).  One translation unit per tile width so they
// compile in parallel.
#include "ngr_gemm2_kernel.cuh"

namespace ngr {

int launch_gemm2_bn128(int norm, bool bf16, const GemmArgs &args, int grid,
                      bool pdl, cudaStream_t stream)
{
    return launch_gemm2_bn<128, 8, 1>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm2_smem_bn128() { return Gemm2Smem<128, 8, 1>::alloc; }
int gemm2_max_clusters_bn128() { return gemm2_max_clusters<128, 8, 1>(); }

}  // namespace ngr
