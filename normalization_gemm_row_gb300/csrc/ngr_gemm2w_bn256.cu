// ngr_gemm2w_bn256.cu -- CTA-pair tile kernel instantiations for a 256 x 512
// output tile made of two 256-column sub-tiles that share each x stage
// (4 pipeline stages, one accumulator).
#include "ngr_gemm2_kernel.cuh"

namespace ngr {

int launch_gemm2w_bn256(int norm, bool bf16, const GemmArgs &args, int grid,
                       bool pdl, cudaStream_t stream)
{
    return launch_gemm2_bn<256, 4, 2>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm2w_smem_bn256() { return Gemm2Smem<256, 4, 2>::alloc; }
int gemm2w_max_clusters_bn256() { return gemm2_max_clusters<256, 4, 2>(); }

}  // namespace ngr
