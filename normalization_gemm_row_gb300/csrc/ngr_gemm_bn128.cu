// ngr_gemm_bn128.cu -- tile kernel instantiations for a 128-column N tile
// (6 pipeline stages).  One translation unit per tile width so they compile
// in parallel.
#include "ngr_gemm_kernel.cuh"

namespace ngr {

int launch_gemm_bn128(int norm, bool bf16, const GemmArgs &args, int grid,
                     bool pdl, cudaStream_t stream)
{
    return launch_gemm_bn<128, 6>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm_smem_bn128() { return GemmSmem<128, 6>::alloc; }

}  // namespace ngr
