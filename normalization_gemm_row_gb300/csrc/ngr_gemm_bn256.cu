// ngr_gemm_bn256.cu -- tile kernel instantiations for a 256-column N tile
// (4 pipeline stages).  One translation unit per tile width so they compile
// in parallel.
#include "ngr_gemm_kernel.cuh"

namespace ngr {

int launch_gemm_bn256(int norm, bool bf16, const GemmArgs &args, int grid,
                     bool pdl, cudaStream_t stream)
{
    return launch_gemm_bn<256, 4>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm_smem_bn256() { return GemmSmem<256, 4>::alloc; }

}  // namespace ngr
