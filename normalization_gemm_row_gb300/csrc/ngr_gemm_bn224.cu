// ngr_gemm_bn224.cu -- tile kernel instantiations for a 224-column N tile
// (5 pipeline stages).  One translation unit per tile width so they compile
// in parallel.
#include "ngr_gemm_kernel.cuh"

namespace ngr {

int launch_gemm_bn224(int norm, bool bf16, const GemmArgs &args, int grid,
                     bool pdl, cudaStream_t stream)
{
    return launch_gemm_bn<224, 5>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm_smem_bn224() { return GemmSmem<224, 5>::alloc; }

}  // namespace ngr
