// ngr_gemm_bn192.cu -- tile kernel instantiations for a 192-column N tile
// (5 pipeline stages).  One translation unit per tile width so they compile
// in parallel.
#include "ngr_gemm_kernel.cuh"

namespace ngr {

int launch_gemm_bn192(int norm, bool bf16, const GemmArgs &args, int grid,
                     bool pdl, cudaStream_t stream)
{
    return launch_gemm_bn<192, 5>(norm, bf16, args, grid, pdl, stream);
}

size_t gemm_smem_bn192() { return GemmSmem<192, 5>::alloc; }

}  // namespace ngr
