// ngr_gemm.cu -- host-side choice of the tile kernel variant and its launch.
//
// The tile kernel is persistent (one CTA per SM), so its time is set by the
// CTA that gets the most tiles: ceil(tiles / grid) tiles of BN columns each.
// The planner picks the N tile width that minimises that, with a small
// per-tile overhead term (each tile re-normalizes its x tile and drains its
// accumulator), so that wave quantization on the SM count at hand is
// avoided without shrinking tiles needlessly.
#include "ngr_internal.h"

namespace ngr {

int launch_gemm_bn128(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn192(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn224(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn256(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
size_t gemm_smem_bn128();
size_t gemm_smem_bn192();
size_t gemm_smem_bn224();
size_t gemm_smem_bn256();

static const int kTileWidths[] = {256, 224, 192, 128};

static int stages_for(int bn)
{
    switch (bn) {
    case 128: return 6;
    case 192: return 5;
    case 224: return 5;
    default: return 4;
    }
}

size_t gemm_smem_bytes(int bn, int, bool)
{
    switch (bn) {
    case 128: return gemm_smem_bn128();
    case 192: return gemm_smem_bn192();
    case 224: return gemm_smem_bn224();
    default: return gemm_smem_bn256();
    }
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms)
{
    (void)K;
    const int64_t m_tiles = (M + kBM - 1) / kBM;
    GemmPlan best{256, 4, 1, 0};
    double best_cost = -1.0;
    for (int bn : kTileWidths) {
        const int64_t tiles = m_tiles * ((N + bn - 1) / bn);
        const int64_t grid = tiles < num_sms ? tiles : num_sms;
        const int64_t per_cta = (tiles + grid - 1) / grid;
        const double cost = static_cast<double>(per_cta) * (bn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = GemmPlan{bn, stages_for(bn), static_cast<int>(grid), 0};
        }
    }
    best.smem = gemm_smem_bytes(best.bn, best.stages, true);
    return best;
}

int launch_gemm(int norm, bool silu, bool bf16, const GemmPlan &plan, const GemmArgs &args,
                bool pdl, cudaStream_t stream)
{
    switch (plan.bn) {
    case 128: return launch_gemm_bn128(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 192: return launch_gemm_bn192(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 224: return launch_gemm_bn224(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 256: return launch_gemm_bn256(norm, silu, bf16, args, plan.grid, pdl, stream);
    default: return -9;
    }
}

}  // namespace ngr
