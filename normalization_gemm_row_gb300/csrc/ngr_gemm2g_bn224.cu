// ngr_gemm2g_bn224.cu -- gated (SwiGLU) CTA-pair tile kernel instantiations:
// 256 x 224 output tiles, the gate and up projections as two 224-column
// sub-tiles sharing each x stage (5 pipeline stages).
#include "ngr_gemm2_kernel.cuh"

namespace ngr {

int launch_gemm2g_bn224(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl,
                       cudaStream_t stream)
{
    return launch_gemm2_gated_bn<224, 5>(norm, bf16, args, grid, pdl, stream);
}

}  // namespace ngr
