// ngr_gemm.cu -- host-side choice of the tile kernel variant and its launch.
//
// The tile kernel is persistent (one CTA per SM), so its time is set by the
// CTA that gets the most tiles: ceil(tiles / grid) tiles of BN columns each.
// The planner picks the N tile width that minimises that, with a small
// per-tile overhead term (each tile re-normalizes its x tile and drains its
// accumulator), so that wave quantization on the SM count at hand is
// avoided without shrinking tiles needlessly.
#include <cstdlib>
#include <mutex>

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
int launch_gemm2_bn128(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn192(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn224(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn256(int, bool, bool, const GemmArgs &, int, bool, cudaStream_t);
size_t gemm2_smem_bn128();
size_t gemm2_smem_bn192();
size_t gemm2_smem_bn224();
size_t gemm2_smem_bn256();
int gemm2_max_clusters_bn224();

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

static int stages2_for(int bn)
{
    switch (bn) {
    case 128: return 8;
    case 192: return 7;
    case 224: return 7;
    default: return 6;
    }
}

static size_t gemm2_smem_bytes(int bn)
{
    switch (bn) {
    case 128: return gemm2_smem_bn128();
    case 192: return gemm2_smem_bn192();
    case 224: return gemm2_smem_bn224();
    default: return gemm2_smem_bn256();
    }
}

// CTA pairs resident at once on the current device (cached per device).
static int max_pairs(int num_sms)
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = gemm2_max_clusters_bn224();
        cache[dev] = (n > 0 && n <= num_sms / 2) ? n : num_sms / 2;
    }
    return cache[dev];
}

// Relative cost of one N column of a 128-row slice on one SM: the CTA-pair
// kernel streams half the W bytes per FLOP and runs closer to the tensor
// peak (measured), so it is preferred unless its tiles quantize worse.
constexpr double kPairCostFactor = 0.8;

// NGR_PAIR=0 never picks the CTA-pair kernel, NGR_PAIR=1 always does when
// M > 128; unset, the cost model decides.
static int pair_override()
{
    static const int v = [] {
        const char *e = std::getenv("NGR_PAIR");
        if (!e || !e[0]) return -1;
        return e[0] == '0' ? 0 : 1;
    }();
    return v;
}

// NGR_BN=128|192|224|256 restricts the planner to that N tile width.
static int bn_override()
{
    static const int v = [] {
        const char *e = std::getenv("NGR_BN");
        return e ? std::atoi(e) : 0;
    }();
    return v;
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, bool norm)
{
    (void)K;
    (void)norm;
    GemmPlan best{256, 4, 1, 0, false, kBM, 256};
    double best_cost = -1.0;
    for (int bn : kTileWidths) {
        if (bn_override() && bn != bn_override()) continue;
        const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
        const int64_t grid = tiles < num_sms ? tiles : num_sms;
        const int64_t per_cta = (tiles + grid - 1) / grid;
        const double cost = static_cast<double>(per_cta) * (bn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = GemmPlan{bn, stages_for(bn), static_cast<int>(grid), 0, false, kBM, bn};
        }
    }
    if (M > kBM && pair_override() != 0) {
        if (pair_override() == 1) best_cost = 1e300;
        const int pairs = max_pairs(num_sms);
        for (int bn : kTileWidths) {
            if (bn_override() && bn != bn_override()) continue;
            const int64_t tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + bn - 1) / bn);
            const int64_t clusters = tiles < pairs ? tiles : pairs;
            if (clusters < 1) continue;
            const int64_t per = (tiles + clusters - 1) / clusters;
            const double cost = kPairCostFactor * static_cast<double>(per) * (bn + 16);
            if (cost < best_cost) {
                best_cost = cost;
                best = GemmPlan{bn, stages2_for(bn), static_cast<int>(2 * clusters), 0, true,
                                2 * kBM, bn / 2};
            }
        }
    }
    best.smem = best.pair ? gemm2_smem_bytes(best.bn) : gemm_smem_bytes(best.bn, best.stages, true);
    return best;
}

int launch_gemm(int norm, bool silu, bool bf16, const GemmPlan &plan, const GemmArgs &args,
                bool pdl, cudaStream_t stream)
{
    if (plan.pair) {
        switch (plan.bn) {
        case 128: return launch_gemm2_bn128(norm, silu, bf16, args, plan.grid, pdl, stream);
        case 192: return launch_gemm2_bn192(norm, silu, bf16, args, plan.grid, pdl, stream);
        case 224: return launch_gemm2_bn224(norm, silu, bf16, args, plan.grid, pdl, stream);
        case 256: return launch_gemm2_bn256(norm, silu, bf16, args, plan.grid, pdl, stream);
        default: return -9;
        }
    }
    switch (plan.bn) {
    case 128: return launch_gemm_bn128(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 192: return launch_gemm_bn192(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 224: return launch_gemm_bn224(norm, silu, bf16, args, plan.grid, pdl, stream);
    case 256: return launch_gemm_bn256(norm, silu, bf16, args, plan.grid, pdl, stream);
    default: return -9;
    }
}

}  // namespace ngr
