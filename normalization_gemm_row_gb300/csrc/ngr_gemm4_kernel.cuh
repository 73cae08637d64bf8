// ngr_gemm4_kernel.cuh -- the fused pre-norm linear layer on clusters of
// two CTA pairs that share each weight box (TMA multicast).
//
// Same computation as gemm2_kernel (a LayerNorm or RMSNorm transform on x
// in shared memory, tcgen05.mma.cta_group::2 into tensor memory, the bias /
// activation epilogue), on 512 x (BN0 + BN1) output super-tiles: cluster
// rank 2p + r is CTA r of pair p; pair p computes rows [m0 + 256 p, +256) of
// the super-tile and both pairs need the same weight rows.  Each weight box
// a CTA needs is split in two row parts, and pair p loads part p of it for
// CTA r of BOTH pairs with one multicast copy: every weight byte crosses
// from L2 to the SMs once per cluster instead of once per pair, which cuts
// the bytes each CTA pulls per stage from x 16 KB + W 29 KB to
// x 16 KB + W 14.5 KB.  The pages' tile-level fusion (the normalized tile
// stays on chip) is unchanged: "LayerNorm 融合算子如何让大模型推理再快 15%？
// 深度拆解 ATB 的实现", §2.1 and §3.1.
//
// Sub-tiles of BN0 = 224 and BN1 = 240 columns: a 464-column super-tile
// lets a 1024 x 8192 output fill the 36 resident clusters of four in one
// wave (2 x 18 super-tiles) and a 512 x 49152 one in three.  Each CTA of a
// pair holds BN/2 weight rows of a sub-tile (112 and 120); the two
// multicast parts are 56 + 56 and 64 + 56 rows, each a whole number of
// 8-row swizzle atoms.  gamma/beta are read by the transform from global
// memory (L1) instead of shared memory, which keeps five 45-KB stages
// within the 227 KB of shared memory.  When the super-tiles fill at most
// half the clusters, K is split in two (units of a super-tile and a K half,
// FP32 partials summed in range order by the last of a chunk's units).
//
// Synchronization (as in gemm2_kernel, plus):
//   full[s]   per CTA: its own x box and both weight parts landed (the
//             expected bytes are this CTA's whole stage, whoever copied them);
//   empty[s]  per CTA, count 2: the commit of each pair's MMA issuer,
//             multicast to all four CTAs -- a producer refills stage s only
//             once both pairs have consumed it, because its multicast
//             writes into both pairs' shared memory.
#pragma once

#include "ngr_gemm2_kernel.cuh"

namespace ngr {

constexpr int kMcBN0 = 224;
constexpr int kMcBN1 = 240;
constexpr int kMcTW = kMcBN0 + kMcBN1;     // columns of a super-tile
constexpr int kMcStages = 5;

struct Gemm4Smem {
    static constexpr int kA = kBM * kBK * 2;             // 16 KB: this CTA's 128 x rows
    static constexpr int kB0 = (kMcBN0 / 2) * kBK * 2;   // 112 weight rows of sub-tile 0
    static constexpr int kB1 = (kMcBN1 / 2) * kBK * 2;   // 120 weight rows of sub-tile 1
    static constexpr int kB = kB0 + kB1;
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + kMcStages * kA;
    static constexpr int off_bar = off_b + kMcStages * kB;
    static constexpr int n_bars = (2 + kMaxParts) * kMcStages + 5;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;
};

// Row parts of a CTA's half of sub-tile j that pair p copies: first row
// and count (multiples of 8).
__device__ __forceinline__ int mc_part_row(int j, int p) { return p == 0 ? 0 : (j == 0 ? 56 : 64); }

template <int NORM, bool BF16>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm4_kernel(const __grid_constant__ GemmArgs args)
{
    using L = Gemm4Smem;
    constexpr int STAGES = kMcStages;
    static_assert(NORM == kNormLayer || NORM == kNormRms || NORM == kNormNone || is_fold(NORM),
                  "the multicast kernel normalizes x or takes it as it is");
    constexpr int kParts = NGR_TRANSFORM_PARTS;
    constexpr uint32_t kReadyCount = 2 * kGroupWarps;
    constexpr bool kRstdOut = NORM == kNormRms && NGR_RMS_RSTD_OUT;
    constexpr uint32_t kIdesc0 = idesc_f16(BF16, 2 * kBM, kMcBN0);
    constexpr uint32_t kIdesc1 = idesc_f16(BF16, 2 * kBM, kMcBN1);
    constexpr uint32_t kTmemCols = 512;
    static_assert(kMcTW <= 512, "accumulator fits in tensor memory");
    static_assert(L::alloc <= 232448, "shared memory");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem + L::off_a;
    uint8_t *sB = smem + L::off_b;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *ready = bars + 2 * STAGES;        // [STAGES * kParts], at the pair leader
    uint64_t *acc_full = bars + (2 + kMaxParts) * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_full + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const int p = static_cast<int>(crank >> 1);      // pair within the cluster
    const int r = static_cast<int>(crank & 1);       // CTA within the pair
    const bool leader = r == 0;                       // the pair's MMA issuer
    const uint32_t pair_leader = crank & ~1u;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};
    // The cluster's last super-tile accumulator, once (the transform warps
    // that help to drain it wait here: a one-shot barrier cannot be confused
    // with an earlier super-tile's phase, however early or late they come).
    __shared__ uint64_t acc_last;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (args.zero_err && blockIdx.x == 0) *args.err = 0;
        prefetch_tmap(&args.map_a);
        prefetch_tmap(&args.map_b);
        prefetch_tmap(&args.map_b2);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);
            for (int q = 0; q < kParts; ++q) mbar_init(&ready[s * kParts + q], kReadyCount);
        }
        mbar_init(&acc_full[0], 1);
        mbar_init(&acc_empty[0], 2 * 4);
        mbar_init(drain, 1);
        mbar_init(&acc_last, 1);
        fence_mbarrier_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // All four CTAs' barriers are initialized before any remote arrive or
    // multicast copy.
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    // Super-tile su: m super-tile su % m_tiles (512 rows), n tile su / m_tiles.
    const int m_tiles = args.m_tiles;
    const int k_blocks = args.k_blocks;
    const int num_tiles = args.num_tiles;
    const int cluster = static_cast<int>(blockIdx.x) >> 2;
    const int n_clusters = static_cast<int>(gridDim.x) >> 2;
    const uint32_t ready_leader = mapa_shared(smem_u32(ready), pair_leader);
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), pair_leader);
    auto m0_of = [&](int su) { return (su % m_tiles) * 4 * kBM + p * 2 * kBM + r * kBM; };
    // Sub-tile 1 wholly past N is neither loaded nor multiplied.
    auto n_sub_of = [&](int su) { return (su / m_tiles) * kMcTW + kMcBN0 < args.N ? 2 : 1; };
    // Work units: (super-tile, K range) pairs; without a split a unit is a
    // super-tile.  (With few super-tiles for the clusters, a K split fills
    // them: each unit writes FP32 partials, and the last of a chunk's units
    // sums them in range order.)
    const int n_splits = max(1, args.k_splits);
    const int num_units = num_tiles * n_splits;
    const int kb_per_split = n_splits > 1 ? args.kb_per_split : k_blocks;
    auto unit_su = [&](int u) { return u / n_splits; };
    auto unit_kb = [&](int u) {
        const int kb0 = (u % n_splits) * kb_per_split;
        return make_int2(kb0, min(k_blocks, kb0 + kb_per_split));
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            pdl_wait();
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            const uint16_t mask = static_cast<uint16_t>((1u << r) | (1u << (2 + r)));
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int u = cluster; ok && u < num_units; u += n_clusters) {
                const int su = unit_su(u);
                const int2 kr = unit_kb(u);
                const int m0 = m0_of(su);
                const int nt0 = (su / m_tiles) * kMcTW;
                const int n_sub = n_sub_of(su);
                const uint32_t tx = static_cast<uint32_t>(L::kA + L::kB0 + (n_sub == 2 ? L::kB1 : 0));
                // This CTA's halves of the two sub-tiles start at these W rows;
                // pair p copies its part of them for CTA r of both pairs.
                const int w0 = nt0 + r * (kMcBN0 / 2) + mc_part_row(0, p);
                const int w1 = nt0 + kMcBN0 + r * (kMcBN1 / 2) + mc_part_row(1, p);
                const CUtensorMap *map1 = p == 0 ? &args.map_b2 : &args.map_b;   // 64 or 56 rows
                for (int kb = kr.x; kb < kr.y; ++kb) {
                    if (!mbar_wait_ahead(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    const int kc = kb * kBK;
                    uint8_t *sb = sB + stage * L::kB;
                    mbar_arrive_expect_tx(&full[stage], tx);
                    tma_load_2d(sA + stage * L::kA, &args.map_a, &full[stage], kc, m0, pol_x);
                    tma_load_2d_mc(sb + mc_part_row(0, p) * 128, &args.map_b, &full[stage], kc, w0, mask,
                                   pol_w);
                    if (n_sub == 2)
                        tma_load_2d_mc(sb + L::kB0 + mc_part_row(1, p) * 128, map1, &full[stage], kc, w1,
                                       mask, pol_w);
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Wait for the copies signalled on this CTA's barriers.
            const int outstanding = fills < STAGES ? static_cast<int>(fills) : STAGES;
            for (int j = 1; ok && j <= outstanding; ++j) {
                int s = stage - j;
                uint32_t ph = phase;
                if (s < 0) { s += STAGES; ph ^= 1u; }
                mbar_wait(&full[s], ph, wc);
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------------ MMA issuer (pair leader)
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint16_t all = 0xF;
            const uint16_t own = static_cast<uint16_t>(0x3u << (2 * p));
            for (int u = cluster; ok && u < num_units; u += n_clusters) {
                if (!mbar_wait_spin(&acc_empty[0], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const int n_sub = n_sub_of(unit_su(u));
                const int2 kr = unit_kb(u);
                for (int kb = kr.x; kb < kr.y; ++kb) {
                    if (!mbar_wait_spin(&ready[stage * kParts], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(sB + stage * L::kB);
                    const uint32_t a_addr = smem_u32(sA + stage * L::kA);
                    constexpr int kStepsPerPart = (kBK / kUmmaK) / kParts;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        if (kParts > 1 && k > 0 && k % kStepsPerPart == 0) {
                            if (!mbar_wait_spin(&ready[stage * kParts + k / kStepsPerPart], phase, wc)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint64_t a_desc = sdesc_kmajor_sw128(a_addr + k * 32);
                        const uint32_t acc = (kb != kr.x || k != 0) ? 1u : 0u;
                        umma_f16_ss_pair(tmem_base, a_desc, sdesc_kmajor_sw128(b_addr + k * 32), kIdesc0, acc);
                        if (n_sub == 2)
                            umma_f16_ss_pair(tmem_base + static_cast<uint32_t>(kMcBN0), a_desc,
                                             sdesc_kmajor_sw128(b_addr + L::kB0 + k * 32), kIdesc1, acc);
                    }
                    if (!ok) break;
                    // Both pairs must be done with the stage before either
                    // producer refills it: the commit reaches all four CTAs.
                    umma_commit_pair(&empty[stage], all);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[0], own);
                if (u + n_clusters >= num_units) umma_commit_pair(&acc_last, own);
                acc_phase ^= 1u;
            }
            umma_commit_pair(drain, static_cast<uint16_t>(1u << crank));
            mbar_wait_long(drain, 0, wc);
        }
    } else if (warp >= kTransformWarp0) {
        const bool epi_warp = warp >= kEpilogueWarp0;
        if (!epi_warp) {
            // ----------------------------------------- transform (A in place)
            const int t = threadIdx.x - kTransformWarp0 * 32;
            transform_role<NORM, BF16, STAGES, L::kA, kParts, !kRstdOut, true>(
                t, cluster, n_clusters, num_units, unit_kb, args.M, args.stats, sA, nullptr, full, wc,
                [&](int u) { return m0_of(unit_su(u)); },
                [&](int st) { mbar_arrive_cluster(ready_leader + 8u * static_cast<uint32_t>(st)); },
                args.gamma_f, args.beta_f, args.K);
        }
        // ----------------------------------------------------- epilogue
        // Epilogue warps drain every super-tile; the transform warps join on
        // the cluster's last one.
        {
            const int q = warp & 3;
            const int e = epi_warp ? 0 : 1 + (warp - kTransformWarp0) / 4;
            uint32_t acc_phase = 0;
            const int N = args.N;
            if constexpr (kRstdOut || is_fold(NORM)) pdl_wait();   // row statistics from the previous grid
            for (int u = cluster; u < num_units; u += n_clusters) {
                const int su = unit_su(u);
                const uint32_t cur_phase = acc_phase;
                acc_phase ^= 1u;
                const bool helped = u + n_clusters >= num_units;
                if (!epi_warp && !helped) continue;
                const int step = (helped ? 3 : 1);
                const int nt0 = (su / m_tiles) * kMcTW;
                const int ncols = min(kMcTW, N - nt0);
                // (helpers: the cluster's last unit's one-shot barrier)
                if (!(epi_warp ? mbar_wait_warp_long(&acc_full[0], cur_phase, wc)
                               : mbar_wait_warp_long(&acc_last, 0, wc)))
                    break;
                tc_fence_after();
                const int row = m0_of(su) + q * 32 + lane;
                float2 so = fold_row_scale<NORM>(args, row);
                if constexpr (kRstdOut)
                    so = make_float2(row < args.M ? rms_out_scale<BF16>(args.stats[row].y) : 0.f, 0.f);
                const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                // Chunks: 7 of 32 over sub-tile 0 ([0, 224)), then 7 of 32 and
                // one of 16 over sub-tile 1 ([224, 464)).
                constexpr int kChunks = kMcChunks;
                // This warp's chunk i is ci = e + i * step, for i < nch.
                int nch = 0;
                for (int ci = e; ci < kChunks && (ci < 14 ? 32 * ci : 448) < ncols; ci += step) ++nch;
                auto load_chunk = [&](int ci, float (&v)[32]) {
                    const int c = ci < 14 ? 32 * ci : 448;
                    if (ci < 14) {
                        uint32_t rr[32];
                        tmem_ld32(t_base + static_cast<uint32_t>(c), rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rr[j]);
                    } else {
                        uint32_t rr[16];
                        tmem_ld16(t_base + static_cast<uint32_t>(c), rr);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(rr[j]);
#pragma unroll
                        for (int j = 16; j < 32; ++j) v[j] = 0.f;
                    }
                };
                auto finish_chunk = [&](int ci, float (&v)[32]) {
                    const int c = ci < 14 ? 32 * ci : 448;
                    epilogue_store32<NORM, BF16, kRstdOut>(v, row, nt0 + c, args, so,
                                                           ci < 14 ? N : min(N, nt0 + kMcTW));
                };
                if (n_splits > 1) {
                    // K split: (1) this unit's FP32 partials of the warp's
                    // chunks (column-major within a chunk, so that each store
                    // of the warp writes one 128-byte line); (2) one fence,
                    // then one counter per chunk (lane i takes the warp's
                    // chunk i); (3) the chunks this unit arrived last at are
                    // summed over the K ranges in range order and finished,
                    // and their counters reset for the next call.
                    const int split = u % n_splits;
                    const size_t blk0 = (static_cast<size_t>(su) * 4 + crank) * 4 * kChunks +
                                        static_cast<size_t>(q) * kChunks;
                    const size_t part_stride = static_cast<size_t>(n_splits) * 1024;
#pragma unroll 1
                    for (int i = 0; i < nch; ++i) {
                        const int ci = e + i * step;
                        float v[32];
                        load_chunk(ci, v);
                        float *mine = args.partials + (blk0 + ci) * part_stride + split * 1024 + lane;
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcg(mine + j * 32, v[j]);
                    }
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane < nch)
                        last = atomicAdd(&args.split_counters[blk0 + e + lane * step], 1) == n_splits - 1;
                    const unsigned last_mask = __ballot_sync(0xffffffffu, last);
                    if (last_mask != 0u) {
                        __threadfence();
#pragma unroll 1
                        for (int i = 0; i < nch; ++i) {
                            if (((last_mask >> i) & 1u) == 0u) continue;
                            const int ci = e + i * step;
                            float own[32];
                            load_chunk(ci, own);
                            const float *part = args.partials + (blk0 + ci) * part_stride + lane;
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                            for (int sp = 0; sp < n_splits; ++sp) {
                                if (sp == split) {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] += own[j];
                                } else {
                                    const float *o = part + sp * 1024;
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] += __ldcg(o + j * 32);
                                }
                            }
                            finish_chunk(ci, v);
                        }
                        __syncwarp();
                        if (lane < nch && ((last_mask >> lane) & 1u))
                            args.split_counters[blk0 + e + lane * step] = 0;
                    }
                } else {
#pragma unroll 1
                    for (int i = 0; i < nch; ++i) {
                        const int ci = e + i * step;
                        float v[32];
                        load_chunk(ci, v);
                        finish_chunk(ci, v);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0 && epi_warp) mbar_arrive_cluster(acc_empty_leader);
            }
        }
    }

    // No CTA frees its tensor memory or leaves while another CTA of the
    // cluster may still write into its shared memory (multicast copies,
    // remote arrivals) or the pair's MMAs may touch it.
    tc_fence_before();
    cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int NORM, bool BF16>
int launch_gemm4_variant(const GemmArgs &args, int grid, bool pdl, cudaStream_t stream)
{
    auto kern = gemm4_kernel<NORM, BF16>;
    constexpr int smem = Gemm4Smem::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return record_cuda_error("cudaFuncSetAttribute(max dynamic smem)", e, cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    return e == cudaSuccess ? 0 : record_cuda_error("cudaLaunchKernelEx (cluster of 4)", e, cudaGetErrorString(e));
}

// Clusters of four of this kernel resident at once on the current device.
inline int gemm4_max_clusters()
{
    auto kern = gemm4_kernel<kNormLayer, false>;
    constexpr int smem = Gemm4Smem::alloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 4;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

}  // namespace ngr
