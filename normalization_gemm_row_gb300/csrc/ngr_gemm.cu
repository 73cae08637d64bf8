// ngr_gemm.cu -- host-side choice of the tile kernel variant and its launch.
//
// The tile kernel is persistent (one CTA per SM), so its time is set by the
// CTA that gets the most tiles: ceil(tiles / grid) tiles of BN columns each.
// The planner picks the N tile width that minimises that, with a small
// per-tile overhead term (each tile re-normalizes its x tile and drains its
// accumulator), so that wave quantization on the SM count at hand is
// avoided without shrinking tiles needlessly.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "ngr_internal.h"

namespace ngr {

int launch_gemm_bn128(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn192(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn224(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm_bn256(int, bool, const GemmArgs &, int, bool, cudaStream_t);
size_t gemm_smem_bn128();
size_t gemm_smem_bn192();
size_t gemm_smem_bn224();
size_t gemm_smem_bn256();
int launch_gemm2_bn128(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn192(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn224(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2_bn256(int, bool, const GemmArgs &, int, bool, cudaStream_t);
size_t gemm2_smem_bn128();
size_t gemm2_smem_bn192();
size_t gemm2_smem_bn224();
size_t gemm2_smem_bn256();
int gemm2_max_clusters_bn224();
int launch_gemm2w_bn192(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2w_bn224(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2w_bn256(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2g_bn192(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2g_bn224(int, bool, const GemmArgs &, int, bool, cudaStream_t);
int launch_gemm2g_bn256(int, bool, const GemmArgs &, int, bool, cudaStream_t);
size_t gemm2w_smem_bn192();
size_t gemm2w_smem_bn224();
size_t gemm2w_smem_bn256();

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

static size_t gemm2_smem_bytes(int bn, int nsub)
{
    if (nsub == 2) return bn == 192 ? gemm2w_smem_bn192() : bn == 224 ? gemm2w_smem_bn224() : gemm2w_smem_bn256();
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

// Relative time of one N column of a k block per 128 rows on one SM, from
// measured stage times on GB300: the CTA-pair kernel (256-row tiles) is the
// unit; the single-CTA kernel streams twice the W bytes per FLOP; the
// two-sub-tile pair form reuses each x stage for twice the columns but does
// not overlap its epilogue (the larger per-tile term).  A K split adds the
// partial write and the reduction of each chunk.
constexpr double kSingleCostFactor = 1.25;
constexpr double kPairCostFactor = 1.0;
constexpr double kWideCostFactor = 0.8;
constexpr int kWideTileOverhead = 32;
constexpr int kSplitOverhead = 24;
// A K split pays only when each half keeps a long K: its fill, drain and
// partial reduction are fixed costs.  Measured on GB300 (alternating runs):
// at 512 x 8192 -> 8192 (64 k blocks per half) the split 448-column plan
// takes 55.3 us against 52.0 for unsplit 256 x 224 pair tiles, while at
// 512 x 28672 -> 8192 (224 k blocks per half) it is the fastest (147.0
// against 150-153).
constexpr int kMinKbPerSplit = 128;

size_t split_partial_bytes(int64_t num_tiles, int tw, int splits, int ctas)
{
    return static_cast<size_t>(num_tiles) * static_cast<size_t>(ctas) * 128 * static_cast<size_t>(tw) *
           static_cast<size_t>(splits) * 4;
}

size_t split_counter_bytes(int64_t num_tiles, int tw, int ctas)
{
    return static_cast<size_t>(num_tiles) * static_cast<size_t>(ctas) * 4 *
           static_cast<size_t>((tw + 31) / 32) * 4;
}

size_t mc_split_partial_bytes(int64_t super, int splits)
{
    return static_cast<size_t>(super) * 4 * 4 * kMcChunks * 1024 * static_cast<size_t>(splits) * 4;
}

size_t mc_split_counter_bytes(int64_t super)
{
    return static_cast<size_t>(super) * 4 * 4 * kMcChunks * 4;
}

// Stages of the two-sub-tile CTA-pair kernel for a sub-tile width.
static int stages2w_for(int bn) { return bn == 256 ? 4 : 5; }
static const int kWideWidths[] = {256, 224, 192};

// Tile-kernel restrictions (ngr_set_tile_config): pair -1/0/1, bn 0 or a
// width, nsub 0/1/2.  Initialized from NGR_PAIR, NGR_BN and NGR_NSUB.
static int env_int(const char *name, int dflt)
{
    const char *e = std::getenv(name);
    return (e && e[0]) ? std::atoi(e) : dflt;
}
static std::atomic<int> g_pair{env_int("NGR_PAIR", -1) < 0 ? -1 : (env_int("NGR_PAIR", -1) > 2 ? 1 : env_int("NGR_PAIR", -1))};
static std::atomic<int> g_bn{env_int("NGR_BN", 0)};
static std::atomic<int> g_nsub{env_int("NGR_NSUB", 0)};
// NGR_MAX_SPLITS caps the K split (1 = never split).
static const int g_max_splits = env_int("NGR_MAX_SPLITS", 2);

int set_tile_config(int pair, int bn, int nsub)
{
    if (pair < -1 || pair > 2) return -9;
    if (bn != 0 && bn != 128 && bn != 192 && bn != 224 && bn != 256) return -9;
    if (nsub < 0 || nsub > 2) return -9;
    if (nsub == 2 && (pair == 0 || (bn != 0 && bn != 192 && bn != 224 && bn != 256))) return -9;
    g_pair.store(pair);
    g_bn.store(bn);
    g_nsub.store(nsub);
    return 0;
}

// The cheapest variant allowed by the restrictions (pair, bn, nsub as in
// set_tile_config); none allowed gives a negative cost.  K splits (CTA pair
// only) are weighed when the partials fit in max_split_bytes.
static GemmPlan plan_with(int64_t M, int64_t N, int64_t K, int num_sms, int want_pair,
                          int want_bn, int want_nsub, size_t max_split_bytes, double *cost_out)
{
    GemmPlan best{256, 4, 1, 0, false, kBM, 256, 1, 256, false, 1};
    const int64_t k_blocks = (K + kBK - 1) / kBK;
    double best_cost = -1.0;
    auto take = [&](double cost, const GemmPlan &p) {
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = p;
        }
    };
    if (want_pair != 1 && want_nsub != 2) {
        // With fewer tiles than SMs (at most 128 rows against a narrow W,
        // where streaming W is the work) a K split of up to
        // kMaxSplitsSingle ranges puts more SMs on it.  Measured on GB300 at
        // LayerNorm 128 x 8192 -> 8192: unsplit, 64 CTAs of 128 x 128 tiles
        // ran the product in 67 us at 2.0 TB/s of W.
        const int max_splits = g_max_splits > 1 ? kMaxSplitsSingle : 1;
        for (int bn : kTileWidths) {
            if (want_bn && bn != want_bn) continue;
            const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
            for (int splits = 1; splits <= max_splits; ++splits) {
                if (splits > 1 && (tiles >= num_sms || k_blocks / splits < kMinKbPerSplitSingle ||
                                   split_partial_bytes(tiles, bn, splits, 1) +
                                           split_counter_bytes(tiles, bn, 1) >
                                       max_split_bytes))
                    continue;
                const int64_t units = tiles * splits;
                const int64_t grid = units < num_sms ? units : num_sms;
                const int64_t per_cta = (units + grid - 1) / grid;
                const double cols = static_cast<double>(bn) / splits + 16 + (splits > 1 ? kSplitOverhead : 0);
                take(kSingleCostFactor * static_cast<double>(per_cta) * cols,
                     GemmPlan{bn, stages_for(bn), static_cast<int>(grid), 0, false, kBM, bn, 1, bn, false,
                              splits});
            }
        }
    }
    if (M > kBM && want_pair != 0) {
        const int pairs = max_pairs(num_sms);
        auto consider = [&](int bn, int nsub, int stages, double factor, int overhead) {
            if (want_bn && bn != want_bn) return;
            if (want_nsub && nsub != want_nsub) return;
            const int tw = bn * nsub;
            const int64_t tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + tw - 1) / tw);
            for (int splits = 1; splits <= 2 && splits <= g_max_splits; ++splits) {
                if (splits > 1 && (tiles >= pairs || (k_blocks + 1) / 2 < kMinKbPerSplit ||
                                   split_partial_bytes(tiles, tw, splits) +
                                           split_counter_bytes(tiles, tw) >
                                       max_split_bytes))
                    continue;
                const int64_t units = tiles * splits;
                const int64_t clusters = units < pairs ? units : pairs;
                if (clusters < 1) return;
                const int64_t per = (units + clusters - 1) / clusters;
                const double cols = static_cast<double>(tw) / splits + overhead +
                                    (splits > 1 ? kSplitOverhead : 0);
                take(factor * static_cast<double>(per) * cols,
                     GemmPlan{bn, stages, static_cast<int>(2 * clusters), 0, true, 2 * kBM,
                              bn / 2, nsub, tw, false, splits});
            }
        };
        for (int bn : kTileWidths) consider(bn, 1, stages2_for(bn), kPairCostFactor, 16);
        for (int bn : kWideWidths)
            consider(bn, 2, stages2w_for(bn), kWideCostFactor, kWideTileOverhead);
    }
    *cost_out = best_cost;
    return best;
}

// Clusters of four of the multicast kernel resident at once (cached per
// device).
static int max_clusters4()
{
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        const int n = gemm4_clusters();
        cache[dev] = n > 0 ? n : -1;
    }
    return cache[dev] > 0 ? cache[dev] : 0;
}

// The multicast cluster kernel (M > 256; a norm, a folded weight or a plain
// product): clusters of two CTA pairs sharing each weight box, 512 x 464
// super-tiles.  Measured on GB300
// against the CTA-pair kernel on the same shapes (with the transform in two
// alternating groups and its waits sleeping with a time hint): 0.960 /
// 0.967 / 0.996 at LayerNorm / RMSNorm fp16 / LayerNorm bf16
// 1024 x 8192 -> 8192 (one super-tile per cluster), 0.964 / 0.970 at
// 2048 x 8192 -> 8192 (two), 1.009 at RMSNorm bf16 512 x 8192 -> 28672,
// where it has 3.5 % more columns per SM; at 512 x 14336 -> 49152 it is
// the faster by 4.4 %.  So the planner takes it when its columns per SM
// stay within 4 % of the pair plan's, for any number of super-tiles per
// cluster (NGR_MC_MIN_RUN raises that minimum).
#ifndef NGR_MC_MIN_RUN
#define NGR_MC_MIN_RUN 1
#endif
static bool prefer_multicast(int64_t M, int64_t N, int64_t K, const GemmPlan &pair_plan, int num_sms)
{
    const int clusters = max_clusters4();
    if (clusters <= 0 || M <= 2 * kBM) return false;
    const int64_t super = ((M + kMcRows - 1) / kMcRows) * ((N + kMcCols - 1) / kMcCols);
    const int64_t per_cluster = (super + clusters - 1) / clusters;
    if (per_cluster < NGR_MC_MIN_RUN) return false;
    if (!pair_plan.pair) return false;
    const int64_t m_tiles = (M + pair_plan.bm - 1) / pair_plan.bm;
    const int64_t tiles = m_tiles * ((N + pair_plan.tw - 1) / pair_plan.tw) * pair_plan.splits;
    const int64_t pairs = pair_plan.grid / 2;
    const int64_t per_pair = (tiles + pairs - 1) / pairs;
    (void)num_sms;
    // With several 256-row tiles per weight column and a long K, the pairs
    // that share a weight column drift apart along K and read it from DRAM
    // again: measured at 512 x 49152 -> 14336 (768 k blocks), the pair plan
    // read 1.98-2.02 GB per launch for 1.41 GB of weights, and the multicast
    // kernel, which reads each weight byte once per cluster, took the same
    // time (440-445 against 443 us).  There it may cost up to 25 % more
    // columns per SM.
    const double margin = (m_tiles >= 2 && K >= 512 * kBK) ? 1.25 : 1.04;
    return static_cast<double>(per_cluster * kMcCols) <=
           margin * static_cast<double>(per_pair * pair_plan.tw) / pair_plan.splits;
}

// A two-way K split on the multicast kernel: when the super-tiles fill at
// most half the clusters, each K half is a unit (FP32 partials, the last of
// a chunk's two units finishes it), if the halves keep kMinKbPerSplitMc k
// blocks and the workspace holds the partials.
constexpr int kMinKbPerSplitMc = 32;
static int mc_splits(int64_t M, int64_t N, int64_t K, size_t max_split_bytes)
{
    const int clusters = max_clusters4();
    const int64_t super = ((M + kMcRows - 1) / kMcRows) * ((N + kMcCols - 1) / kMcCols);
    const int64_t k_blocks = (K + kBK - 1) / kBK;
    if (2 * super <= clusters && k_blocks / 2 >= kMinKbPerSplitMc &&
        mc_split_partial_bytes(super, 2) + mc_split_counter_bytes(super) <= max_split_bytes)
        return 2;
    return 1;
}

static GemmPlan multicast_plan(int64_t M, int64_t N, int splits)
{
    const int clusters = max_clusters4();
    const int64_t units = ((M + kMcRows - 1) / kMcRows) * ((N + kMcCols - 1) / kMcCols) * splits;
    GemmPlan p{224, 5, static_cast<int>(4 * (units < clusters ? units : clusters)), 0, true,
               kMcRows, 56, 2, kMcCols, false, splits};
    p.mc = true;
    p.smem = gemm4_smem_bytes();
    return p;
}

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, bool norm,
                   size_t max_split_bytes, bool plain)
{
    const int want = g_pair.load();
    const bool mc_ok = norm || plain;
    if (want == 2 && mc_ok && M > 2 * kBM && max_clusters4() > 0)
        return multicast_plan(M, N, mc_splits(M, N, K, max_split_bytes));
    double cost = -1.0;
    GemmPlan best = plan_with(M, N, K, num_sms, want == 2 ? -1 : want, g_bn.load(), g_nsub.load(),
                              max_split_bytes, &cost);
    if (cost < 0) best = plan_with(M, N, K, num_sms, -1, 0, 0, max_split_bytes, &cost);
    best.smem = best.pair ? gemm2_smem_bytes(best.bn, best.nsub)
                          : gemm_smem_bytes(best.bn, best.stages, true);
    if (want == -1 && mc_ok && g_bn.load() == 0 && g_nsub.load() == 0) {
        // Few super-tiles: the multicast kernel with K split in two, for a
        // normalized product or a long K.  Measured on GB300 against the
        // CTA-pair plans (alternating bursts): 0.942 at RMSNorm fp16 and
        // 0.908 at LayerNorm bf16 512 x 8192 -> 8192, 0.986 at 512 x 28672 ->
        // 8192 without a norm; at 512 x 8192 -> 8192 without a norm (64 k
        // blocks per half) the pair plan stays ahead (1.118).
        const int ms = mc_splits(M, N, K, max_split_bytes);
        if (ms > 1 && (norm || (K + kBK - 1) / kBK >= 256)) return multicast_plan(M, N, ms);
        if (prefer_multicast(M, N, K, best, num_sms)) return multicast_plan(M, N, 1);
    }
    return best;
}

GemmPlan plan_gemm_gated(int64_t M, int64_t N, int num_sms)
{
    // Gate and up sub-tiles of BN columns each: 256 x BN outputs per tile,
    // 2 BN accumulator columns.  The widest tile that does not add a wave.
    const int pairs = max_pairs(num_sms);
    GemmPlan best{224, stages2w_for(224), 2, 0, true, 2 * kBM, 112, 2, 224, true, 1};
    double best_cost = -1.0;
    for (int bn : kWideWidths) {
        if (g_bn.load() && bn != g_bn.load()) continue;
        const int64_t tiles = ((M + 2 * kBM - 1) / (2 * kBM)) * ((N + bn - 1) / bn);
        const int64_t clusters = tiles < pairs ? tiles : pairs;
        if (clusters < 1) continue;
        const int64_t per = (tiles + clusters - 1) / clusters;
        const double cost = static_cast<double>(per) * (bn + kWideTileOverhead / 2);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = GemmPlan{bn, stages2w_for(bn), static_cast<int>(2 * clusters), 0, true,
                            2 * kBM, bn / 2, 2, bn, true, 1};
        }
    }
    best.smem = gemm2_smem_bytes(best.bn, 2);
    return best;
}

int launch_gemm(int norm, bool bf16, const GemmPlan &plan, const GemmArgs &args, bool pdl,
                cudaStream_t stream)
{
    if (plan.mc) return launch_gemm4(norm, bf16, args, plan.grid, pdl, stream);
    if (plan.gated) {
        switch (plan.bn) {
        case 192: return launch_gemm2g_bn192(norm, bf16, args, plan.grid, pdl, stream);
        case 224: return launch_gemm2g_bn224(norm, bf16, args, plan.grid, pdl, stream);
        case 256: return launch_gemm2g_bn256(norm, bf16, args, plan.grid, pdl, stream);
        default: return -9;
        }
    }
    if (plan.pair && plan.nsub == 2) {
        switch (plan.bn) {
        case 192: return launch_gemm2w_bn192(norm, bf16, args, plan.grid, pdl, stream);
        case 224: return launch_gemm2w_bn224(norm, bf16, args, plan.grid, pdl, stream);
        case 256: return launch_gemm2w_bn256(norm, bf16, args, plan.grid, pdl, stream);
        default: return -9;
        }
    }
    if (plan.pair) {
        switch (plan.bn) {
        case 128: return launch_gemm2_bn128(norm, bf16, args, plan.grid, pdl, stream);
        case 192: return launch_gemm2_bn192(norm, bf16, args, plan.grid, pdl, stream);
        case 224: return launch_gemm2_bn224(norm, bf16, args, plan.grid, pdl, stream);
        case 256: return launch_gemm2_bn256(norm, bf16, args, plan.grid, pdl, stream);
        default: return -9;
        }
    }
    switch (plan.bn) {
    case 128: return launch_gemm_bn128(norm, bf16, args, plan.grid, pdl, stream);
    case 192: return launch_gemm_bn192(norm, bf16, args, plan.grid, pdl, stream);
    case 224: return launch_gemm_bn224(norm, bf16, args, plan.grid, pdl, stream);
    case 256: return launch_gemm_bn256(norm, bf16, args, plan.grid, pdl, stream);
    default: return -9;
    }
}

}  // namespace ngr
