// ngr_gemm2_kernel.cuh -- the fused pre-norm linear layer on a CTA pair
// (tcgen05 cta_group::2): same computation as gemm_kernel, on 256 x (NSUB BN)
// output tiles.
//
// The two CTAs of a cluster share each tile: CTA r loads rows
// [m0 + 128 r, +128) of x and, for each of the NSUB sub-tiles j, rows
// [n0 + j BN + r BN/2, +BN/2) of W into its own shared memory (no
// multicast), normalizes its own x rows in place, and the even CTA issues
// per K step one tcgen05.mma.cta_group::2 per sub-tile, each reading A from
// both CTAs by rows and its B from both CTAs by columns, accumulating its 128
// rows of D in each CTA's tensor memory.  Per CTA this halves the W bytes
// loaded and read from shared memory per FLOP compared with a single-CTA
// 128 x BN tile; with NSUB = 2 the normalized A stage also serves twice the
// columns, which cuts the shared-memory fill bytes per FLOP by another
// quarter and halves the normalization work per FLOP.  The price is one
// accumulator instead of two: the epilogue of a tile does not overlap the
// next tile's MMAs.
//
// GATED (SwiGLU, NSUB = 2): sub-tile 0 multiplies the gate weight and
// sub-tile 1 the up weight over the same BN output columns, so each output
// tile is 256 x BN and the epilogue writes SiLU(gate) * up from the two
// accumulators ("CANN推理加速库ascend-transformer-boost ATB算子融合实战...",
// Llama2 inference, model structure and fusion opportunities: the FFN's
// SiLU-gated linear transform fused with its matmuls).
//
// The gated tiles with a norm keep x and W in separate rings: a deeper x
// ring that warp 0 fills and the transform normalizes ahead of the MMAs,
// and a W ring that warp 3 fills (split_rings).
//
// Synchronization (barriers are per CTA unless marked "leader"):
//   full[s]        with a norm: this CTA's copies of (x) stage s landed (its
//                  producer's expect_tx); without: the leader's, on which
//                  both CTAs' copies complete (cta_group::2 TMA) -- the MMA
//                  waits on it;
//   ready[s, p]    leader, with a norm: each transform warp of both CTAs
//                  arrives once column part p of its CTA's (x) stage is
//                  normalized (the MMAs of that part's K steps wait on it);
//   empty[s]       the leader's tcgen05.commit, multicast to both CTAs;
//   wfull[s], wempty[s]  split rings: W stage s, the leader's barrier on
//                  which both CTAs' W copies complete, and its release;
//   acc_full[a]    the leader's commit at the end of a tile, multicast;
//   acc_empty[a]   leader: each draining warp of both CTAs arrives after
//                  reading its share of accumulator a.
//
// Draining an accumulator: epilogue warps 12-15 drain every tile.  Without
// a norm the transform warps 4-11 have no other work and drain with them
// (three warps per tensor-memory lane quarter, each taking every third
// 32-column chunk); with a norm they join only on the cluster's last tile,
// when no stage is left to normalize, so that the tail is short.
#pragma once

#include "ngr_gemm_kernel.cuh"

namespace ngr {

// Column parts per stage of the in-place transform (1, 2 or 4): the MMAs of
// a part's K steps are issued once that part of both CTAs' stages is
// normalized.  One part (a single arrival per warp and stage) measured 2-3 %
// faster than two at LayerNorm 1024 x 8192 -> 8192 and RMSNorm
// 512 x 14336 -> 49152, fp16 and bf16: the saved barrier traffic outweighs
// the earlier start of the first K steps.
#ifndef NGR_TRANSFORM_PARTS
#define NGR_TRANSFORM_PARTS 1
#endif
constexpr int kMaxParts = 4;
#ifndef NGR_RMS_RSTD_OUT
#define NGR_RMS_RSTD_OUT 1
#endif


// With a norm, x and W stages can live in separate rings (SPLIT): the W
// ring is one stage shorter than the unified ring of the same tile, and the
// x ring (x box + FP32 gamma/beta box per stage) takes the shared memory
// left, so the transform normalizes x stages ahead of the MMAs that consume
// them.  Measured on GB300: the gated (SwiGLU) tiles run 6 % faster split
// (512 x 8192 -> 2 x 28672, RMSNorm, bf16), the plain two-sub-tile tiles
// 1-5 % slower (their W ring's lost stage costs more than the transform's
// latency); so the gated variants split.  NGR_SPLIT_RINGS: 0 never,
// 1 gated tiles (default), 2 every tile with a norm and two sub-tiles.
#ifndef NGR_SPLIT_RINGS
#define NGR_SPLIT_RINGS 1
#endif
constexpr int kSmemLimit = 232448;   // dynamic shared memory per CTA (227 KB)

template <int BN, int STAGES, int NSUB, bool SPLIT = false>
struct Gemm2Smem {
    static constexpr int kA = kBM * kBK * 2;          // 16 KB: this CTA's 128 x rows
    static constexpr int kBSub = (BN / 2) * kBK * 2;  // this CTA's BN/2 W rows of one sub-tile
    static constexpr int kB = NSUB * kBSub;
    static constexpr int kGB = 2 * kBK * 4;           // FP32 gamma[64], beta[64]
    // Ring depths: W stages, and x stages (equal without SPLIT).
    static constexpr int kBStages = SPLIT ? STAGES - 1 : STAGES;
    static constexpr int kMaxAStages = 12;
    static constexpr int kBarReserve = 8 * ((2 + kMaxParts) * kMaxAStages + 2 * STAGES + 5) + 16;
    static constexpr int kAFit = (kSmemLimit - 1024 - kBarReserve - kBStages * kB) / (kA + kGB);
    static constexpr int kAStages = SPLIT ? (kAFit < kMaxAStages ? kAFit : kMaxAStages) : STAGES;
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + kAStages * kA;
    static constexpr int off_g = off_b + kBStages * kB;
    static constexpr int off_bar = off_g + kAStages * kGB;
    // full/empty/ready[parts] per x stage (per unified stage without
    // SPLIT), full/empty per W stage (SPLIT), acc_full[2], acc_empty[2], drain
    static constexpr int n_bars = (2 + kMaxParts) * kAStages + (SPLIT ? 2 * kBStages : 0) + 5;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;
    static_assert(!SPLIT || kAStages > kBStages, "the x ring is the deeper one");
    static_assert(alloc <= kSmemLimit, "shared memory");
};

// Whether a variant runs separate x and W rings.
template <int NORM, int NSUB, bool GATED>
constexpr bool split_rings()
{
    return (NORM == kNormLayer || NORM == kNormRms) && NSUB == 2 &&
           (NGR_SPLIT_RINGS == 2 || (NGR_SPLIT_RINGS == 1 && GATED));
}


template <int NORM, bool BF16, int BN, int STAGES, int NSUB, bool GATED>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm2_kernel(const __grid_constant__ GemmArgs args)
{
    constexpr bool kSplit = split_rings<NORM, NSUB, GATED>();
    using L = Gemm2Smem<BN, STAGES, NSUB, kSplit>;
    constexpr int SA = L::kAStages;    // x ring (the unified ring without kSplit)
    constexpr int SB = L::kBStages;    // W ring
    constexpr bool kNorm = NORM == kNormLayer || NORM == kNormRms;  // transform stage
    constexpr int kTW = NSUB * BN;                 // accumulator columns of a tile
    constexpr int kOutW = GATED ? BN : kTW;        // output columns of a tile
    static_assert(!GATED || (NSUB == 2 && !is_fold(NORM)), "gated tiles: gate and up sub-tiles");
    // Bytes one stage of this CTA receives when n_sub sub-tiles are in range.
    auto stage_tx = [](int n_sub) -> uint32_t {
        return static_cast<uint32_t>(L::kA + n_sub * L::kBSub + (kNorm ? L::kGB : 0));
    };
    // Accumulators: two of kTW columns with one sub-tile (the epilogue of a
    // tile overlaps the next tile's MMAs), one with two.
    constexpr uint32_t kTmemCols = 512;
    constexpr int kAccBufs = NSUB > 1 ? 1 : 2;
    constexpr uint32_t kIdesc = idesc_f16(BF16, 2 * kBM, BN);
    // ready[s * kParts + p] arrivals: one per warp of the transform group
    // that works on the stage, in each CTA (used with a norm only).
    constexpr uint32_t kReadyCount = 2 * kGroupWarps;
    constexpr int kParts = kNorm ? NGR_TRANSFORM_PARTS : 1;
    // RMSNorm: the transform computes x s gamma in packed 16-bit arithmetic
    // (s a power of two near the row's rstd; transform8_rms16) and the
    // epilogue multiplies each row by rstd / s.
    constexpr bool kRstdOut = NORM == kNormRms && NGR_RMS_RSTD_OUT;
    static_assert(kParts >= 1 && kParts <= kMaxParts && (kBK / kUmmaK) % kParts == 0,
                  "whole K steps per transform part");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "UMMA N for M = 256");
    static_assert((BN / 2) % 8 == 0, "B half tile rows (1024-byte swizzle atoms)");
    static_assert(NSUB >= 1 && kAccBufs * kTW <= 512, "accumulators fit in tensor memory");
    // Warps per CTA that drain every accumulator (and arrive on acc_empty).
    constexpr bool kHelpAlways = !kNorm;
    constexpr bool kHelpLast = kNorm;
    constexpr int kDrainWarps = kHelpAlways ? 12 : 4;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem + L::off_a;
    uint8_t *sB = smem + L::off_b;
    float *sG = reinterpret_cast<float *>(smem + L::off_g);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;                      // [SA] (x) stage landed
    uint64_t *empty = bars + SA;                // [SA] (x) stage released by the MMAs
    uint64_t *ready = bars + 2 * SA;            // [SA * kParts] part of both stages normalized
    uint64_t *acc_full = bars + (2 + kMaxParts) * SA;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_full + 4;
    // kSplit: the W ring's barriers, the leader's full on which both CTAs'
    // W copies complete, and empty (the MMAs' commit, multicast).
    uint64_t *wfull = kSplit ? drain + 1 : full;
    uint64_t *wempty = kSplit ? drain + 1 + SB : empty;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};
    // The last unit's accumulator, once (the transform warps that help to
    // drain it wait here: a one-shot barrier cannot be confused with an
    // earlier unit's phase, however early or late the helpers arrive).
    __shared__ uint64_t acc_last;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (args.zero_err && blockIdx.x == 0) *args.err = 0;
        prefetch_tmap(&args.map_a);
        prefetch_tmap(&args.map_b);
        if constexpr (GATED) prefetch_tmap(&args.map_b2);
        if constexpr (kNorm) prefetch_tmap(&args.map_gb);
        for (int s = 0; s < SA; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            for (int p = 0; p < kParts; ++p) mbar_init(&ready[s * kParts + p], kReadyCount);
        }
        if constexpr (kSplit) {
            for (int s = 0; s < SB; ++s) {
                mbar_init(&wfull[s], 1);
                mbar_init(&wempty[s], 1);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 2 * kDrainWarps);
        }
        mbar_init(drain, 1);
        mbar_init(&acc_last, 1);
        fence_mbarrier_init();
    }
    if (warp == 2) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    // Both CTAs' barriers are initialized before any remote arrive.
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    const int m_tiles = args.m_tiles;   // 256-row pair tiles
    const int k_blocks = args.k_blocks;
    const int num_tiles = args.num_tiles;
    // Work units: (tile, K range) pairs; without a split a unit is a tile.
    const int n_splits = GATED ? 1 : max(1, args.k_splits);
    const int num_units = num_tiles * n_splits;
    const int kb_per_split = n_splits > 1 ? args.kb_per_split : k_blocks;
    auto unit_tile = [&](int u) { return u / n_splits; };
    auto unit_kb0 = [&](int u) { return (u % n_splits) * kb_per_split; };
    auto unit_kb1 = [&](int u) { return min(k_blocks, unit_kb0(u) + kb_per_split); };
    const int cluster = blockIdx.x >> 1;
    const int n_clusters = gridDim.x >> 1;
    // Leader-side addresses of ready[] and acc_empty[] (shared::cluster).
    const uint32_t ready_leader = mapa_shared(smem_u32(ready), 0);
    const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
    const uint32_t wfull_leader = mapa_shared(smem_u32(wfull), 0);
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);

    if (warp == 0 || (kSplit && warp == 3)) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // One ring: warp 0 loads each stage's x and W boxes (and the
            // FP32 gamma/beta box with a norm).  Split rings: warp 0 loads
            // the x ring (x and gamma/beta boxes, on this CTA's barriers),
            // warp 3 the W ring (both CTAs' copies complete on the leader's
            // barrier, which expects the bytes of both).
            const bool x_side = warp == 0;
            const int depth = x_side ? SA : SB;
            uint64_t *rempty = x_side ? empty : wempty;
            pdl_wait();
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int u = cluster; ok && u < num_units; u += n_clusters) {
                const int tile = unit_tile(u);
                const int m0 = (tile % m_tiles) * 2 * kBM + static_cast<int>(rank) * kBM;
                const int nt0 = (tile / m_tiles) * kOutW;
                const int n0 = nt0 + static_cast<int>(rank) * (BN / 2);
                // Sub-tiles wholly past N are neither loaded nor multiplied
                // (gated: both sub-tiles cover the same columns).
                const int n_sub = GATED ? 2 : min(NSUB, (args.N - nt0 + BN - 1) / BN);
                // W box of sub-tile j: its tensor and its first row.
                auto wmap = [&](int j) { return (GATED && j == 1) ? &args.map_b2 : &args.map_b; };
                auto wrow = [&](int j) { return GATED ? n0 : n0 + j * BN; };
                const uint32_t tx = stage_tx(n_sub);
                for (int kb = unit_kb0(u), kb_end = unit_kb1(u); kb < kb_end; ++kb) {
                    if (!mbar_wait_ahead(&rempty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    const int kc = kb * kBK;
                    if constexpr (kSplit) {
                        if (x_side) {
                            mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(L::kA + L::kGB));
                            tma_load_2d(sA + stage * L::kA, &args.map_a, &full[stage], kc, m0, pol_x);
                            tma_load_2d(sG + stage * 2 * kBK, &args.map_gb, &full[stage], kc, 0, pol_x);
                        } else {
                            uint8_t *sb = sB + stage * L::kB;
                            const uint32_t fb = wfull_leader + 8u * static_cast<uint32_t>(stage);
                            if (leader)
                                mbar_arrive_expect_tx(&wfull[stage], static_cast<uint32_t>(2 * n_sub * L::kBSub));
                            for (int j = 0; j < n_sub; ++j)
                                tma_load_2d_pair(sb + j * L::kBSub, wmap(j), fb, kc, wrow(j), pol_w);
                        }
                    } else if constexpr (kNorm) {
                        // Each CTA normalizes its own stage: local barrier.
                        uint8_t *sb = sB + stage * L::kB;
                        mbar_arrive_expect_tx(&full[stage], tx);
                        tma_load_2d(sA + stage * L::kA, &args.map_a, &full[stage], kc, m0, pol_x);
                        for (int j = 0; j < n_sub; ++j)
                            tma_load_2d(sb + j * L::kBSub, wmap(j), &full[stage], kc, wrow(j), pol_w);
                        tma_load_2d(sG + stage * 2 * kBK, &args.map_gb, &full[stage], kc, 0, pol_x);
                    } else {
                        // Both CTAs' copies complete on the leader's barrier,
                        // which expects the bytes of both.
                        uint8_t *sb = sB + stage * L::kB;
                        const uint32_t fb = full_leader + 8u * static_cast<uint32_t>(stage);
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                        tma_load_2d_pair(sA + stage * L::kA, &args.map_a, fb, kc, m0, pol_x);
                        for (int j = 0; j < n_sub; ++j)
                            tma_load_2d_pair(sb + j * L::kBSub, wmap(j), fb, kc, wrow(j), pol_w);
                    }
                    ++fills;
                    if (++stage == depth) { stage = 0; phase ^= 1u; }
                }
            }
            // Copies signalled on this CTA's own barriers: wait for the last
            // fills.  (Copies that complete on the leader's barriers -- all
            // of them without a norm, the W ring's with split rings -- are
            // waited for by the leader alone; the leader's MMAs, and so the
            // final cluster barrier, come after them.)
            const bool own = kSplit ? x_side : kNorm;
            if (own || leader) {
                uint64_t *rfull = (kSplit && !x_side) ? wfull : full;
                const int outstanding = fills < depth ? static_cast<int>(fills) : depth;
                for (int j = 1; j <= outstanding; ++j) {
                    int s = stage - j;
                    uint32_t p = phase;
                    if (s < 0) { s += depth; p ^= 1u; }
                    mbar_wait(&rfull[s], p, wc);
                }
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------- MMA issuer (even CTA)
            int stage = 0;          // x stage (the unified stage without split rings)
            uint32_t phase = 0;
            int wstage = 0;         // W stage (split rings)
            uint32_t wphase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = cluster; ok && u < num_units; u += n_clusters) {
                const int tile = unit_tile(u);
                const int kb0 = unit_kb0(u);
                if (!mbar_wait_spin(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kTW);
                const int n_sub = GATED ? 2 : min(NSUB, (args.N - (tile / m_tiles) * kTW + BN - 1) / BN);
                for (int kb = kb0, kb_end = unit_kb1(u); kb < kb_end; ++kb) {
                    if (kSplit && !mbar_wait_spin(&wfull[wstage], wphase, wc)) { ok = false; break; }
                    if (!mbar_wait_spin(kNorm ? &ready[stage * kParts] : &full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(sB + (kSplit ? wstage : stage) * L::kB);
                    const uint32_t a_addr = smem_u32(sA + stage * L::kA);
                    constexpr int kStepsPerPart = (kBK / kUmmaK) / kParts;
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        if (kParts > 1 && k > 0 && k % kStepsPerPart == 0) {
                            // The next column part of both CTAs' stages.
                            if (!mbar_wait_spin(&ready[stage * kParts + k / kStepsPerPart], phase, wc)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint64_t a_desc = sdesc_kmajor_sw128(a_addr + k * 32);
#pragma unroll
                        for (int j = 0; j < NSUB; ++j) {
                            if (j < n_sub)
                                umma_f16_ss_pair(d_tmem + static_cast<uint32_t>(j * BN), a_desc,
                                                 sdesc_kmajor_sw128(b_addr + j * L::kBSub + k * 32),
                                                 kIdesc, (kb != kb0 || k != 0) ? 1u : 0u);
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair(&empty[stage], 0x3);
                    if (++stage == SA) { stage = 0; phase ^= 1u; }
                    if constexpr (kSplit) {
                        umma_commit_pair(&wempty[wstage], 0x3);
                        if (++wstage == SB) { wstage = 0; wphase ^= 1u; }
                    }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[acc], 0x3);
                if (kHelpLast && u + n_clusters >= num_units) umma_commit_pair(&acc_last, 0x3);
                if (++acc == kAccBufs) { acc = 0; acc_phase ^= 1u; }
            }
            umma_commit_pair(drain, 0x1);
            mbar_wait_long(drain, 0, wc);
        }
    } else if (warp >= kTransformWarp0) {
        const bool epi_warp = warp >= kEpilogueWarp0;
        if (!epi_warp) {
            const int t = threadIdx.x - kTransformWarp0 * 32;
            if constexpr (kNorm) {
                // ----------------------------------------- transform (A in place)
                transform_role<NORM, BF16, SA, L::kA, kParts, !kRstdOut>(
                    t, cluster, n_clusters, num_units, [&](int u) { return make_int2(unit_kb0(u), unit_kb1(u)); },
                    args.M, args.stats, sA, sG, full, wc,
                    [&](int u) { return (unit_tile(u) % m_tiles) * 2 * kBM + static_cast<int>(rank) * kBM; },
                    [&](int st) { mbar_arrive_cluster(ready_leader + 8u * static_cast<uint32_t>(st)); });
            }
        }
        if (epi_warp || kHelpAlways || kHelpLast) {
            // ----------------------------------------------------- epilogue
            const int q = warp & 3;                 // tensor-memory lane quarter
            const int e = epi_warp ? 0 : 1 + (warp - kTransformWarp0) / 4;
            int acc = 0;
            uint32_t acc_phase = 0;
            const int N = args.N;
            if constexpr (is_fold(NORM) || kRstdOut) pdl_wait();  // row statistics from the previous grid
            for (int u = cluster; u < num_units; u += n_clusters) {
                const int tile = unit_tile(u);
                const int split = u % n_splits;
                const int cur = acc;
                const uint32_t cur_phase = acc_phase;
                if (++acc == kAccBufs) { acc = 0; acc_phase ^= 1u; }
                const bool helped = kHelpAlways || (kHelpLast && u + n_clusters >= num_units);
                if (!epi_warp && !helped) continue;
                const int step = (helped ? 3 : 1) * 32;
                const int nt0 = (tile / m_tiles) * kOutW;
                const int ncols = min(kOutW, N - nt0);
                // Warm L1 with this warp's epilogue vectors while the MMAs run.
                for (int c = e * 32; c < ncols; c += step) {
                    if constexpr (is_fold(NORM)) {
                        if (lane == 0) prefetch_l1(args.fold_b + nt0 + c);
                        if (NORM == kNormFoldLayer && lane == 1) prefetch_l1(args.fold_c + nt0 + c);
                    } else {
                        if (lane == 0 && args.bias)
                            prefetch_l1(static_cast<const uint16_t *>(args.bias) + nt0 + c);
                    }
                }
                // (helpers: the last unit's one-shot barrier)
                if (!(epi_warp || kHelpAlways ? mbar_wait_warp_long(&acc_full[cur], cur_phase, wc)
                                              : mbar_wait_warp_long(&acc_last, 0, wc)))
                    break;
                tc_fence_after();
                const int row = (tile % m_tiles) * 2 * kBM + static_cast<int>(rank) * kBM + q * 32 + lane;
                float2 so = fold_row_scale<NORM>(args, row);
                if constexpr (kRstdOut)
                    so = make_float2(row < args.M ? rms_out_scale<BF16>(args.stats[row].y) : 0.f, 0.f);
                const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                        static_cast<uint32_t>(cur * kTW);
                if constexpr (GATED) {
                    // h = SiLU(gate) * up, the gate in columns [0, BN), the
                    // up projection in [BN, 2 BN) of the accumulator.
#pragma unroll 1
                    for (int c = e * 32; c < ncols; c += step) {
                        uint32_t rg[32], ru[32];
                        tmem_ld32(t_base + static_cast<uint32_t>(c), rg);
                        tmem_ld32(t_base + static_cast<uint32_t>(BN + c), ru);
                        tmem_ld_wait();
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            float gj = __uint_as_float(rg[j]), uj = __uint_as_float(ru[j]);
                            if constexpr (kRstdOut) {
                                gj *= so.x;
                                uj *= so.x;
                            }
                            v[j] = silu_f(gj) * uj;
                        }
                        store_row32<BF16>(v, row, nt0 + c, args.y, args.M, N);
                    }
                } else if (n_splits > 1) {
                    // K split: (1) this unit's FP32 partials of the warp's
                    // 32 x 32 chunks; (2) one fence, then one counter per
                    // chunk (lane i takes the i-th chunk); (3) the chunks
                    // this unit arrived last at are summed over the K
                    // ranges in range order and finished.
                    const size_t blk0 = ((static_cast<size_t>(tile) * 2 + rank) * 4 + q) *
                                        static_cast<size_t>(kTW / 32);
                    const size_t part_stride = static_cast<size_t>(n_splits) * 1024;
                    int nch = 0;
#pragma unroll 1
                    for (int c = e * 32; c < ncols; c += step, ++nch) {
                        uint32_t r[32];
                        tmem_ld32(t_base + static_cast<uint32_t>(c), r);
                        tmem_ld_wait();
                        // column-major within the chunk: each store of the
                        // warp writes one contiguous 128-byte line
                        float *mine = args.partials + (blk0 + (c >> 5)) * part_stride + split * 1024 + lane;
#pragma unroll
                        for (int j = 0; j < 32; ++j) __stcg(mine + j * 32, __uint_as_float(r[j]));
                    }
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane < nch)
                        last = atomicAdd(&args.split_counters[blk0 + ((e * 32 + lane * step) >> 5)], 1) ==
                               n_splits - 1;
                    const unsigned last_mask = __ballot_sync(0xffffffffu, last);
                    if (last_mask != 0u) {
                        __threadfence();
#pragma unroll 1
                        for (int i = 0; i < nch; ++i) {
                            if (((last_mask >> i) & 1u) == 0u) continue;
                            const int c = e * 32 + i * step;
                            uint32_t r[32];
                            tmem_ld32(t_base + static_cast<uint32_t>(c), r);
                            tmem_ld_wait();
                            const float *part = args.partials + (blk0 + (c >> 5)) * part_stride + lane;
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                            for (int sp = 0; sp < n_splits; ++sp) {
                                if (sp == split) {
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] += __uint_as_float(r[j]);
                                } else {
                                    const float *o = part + sp * 1024;
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[j] += __ldcg(o + j * 32);
                                }
                            }
                            epilogue_store32<NORM, BF16, kRstdOut>(v, row, nt0 + c, args, so);
                        }
                        __syncwarp();
                        // ready for the next call (every unit of these chunks has arrived)
                        if (lane < nch && ((last_mask >> lane) & 1u))
                            args.split_counters[blk0 + ((e * 32 + lane * step) >> 5)] = 0;
                    }
                } else {
                    // The load of the next chunk is in flight while this one
                    // is finished and stored.
                    uint32_t r[32];
                    int c = e * 32;
                    if (c < ncols) tmem_ld32(t_base + static_cast<uint32_t>(c), r);
#pragma unroll 1
                    while (c < ncols) {
                        tmem_ld_wait();
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        const int cn = c + step;
                        if (cn < ncols) tmem_ld32(t_base + static_cast<uint32_t>(cn), r);
                        epilogue_store32<NORM, BF16, kRstdOut>(v, row, nt0 + c, args, so);
                        c = cn;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (epi_warp || kHelpAlways)
                    if (lane == 0) mbar_arrive_cluster(acc_empty_leader + 8u * static_cast<uint32_t>(cur));
            }
        }
    }

    // Neither CTA frees its tensor memory or leaves while the pair may
    // still touch it (the leader's MMAs write both CTAs' tensor memory; the
    // peer arrives on the leader's barriers).
    tc_fence_before();
    cluster_sync_all();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, kTmemCols);
    }
}

template <int NORM, bool BF16, int BN, int STAGES, int NSUB, bool GATED>
int launch_gemm2_variant(const GemmArgs &args, int grid, bool pdl, cudaStream_t stream)
{
    auto kern = gemm2_kernel<NORM, BF16, BN, STAGES, NSUB, GATED>;
    constexpr int smem = Gemm2Smem<BN, STAGES, NSUB, split_rings<NORM, NSUB, GATED>()>::alloc;
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
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    return e == cudaSuccess ? 0 : record_cuda_error("cudaLaunchKernelEx (CTA pair)", e, cudaGetErrorString(e));
}

// How many CTA pairs of this kernel can be resident at once on the current
// device (pairs must share a GPC, so this can be below SMs / 2).
template <int BN, int STAGES, int NSUB>
int gemm2_max_clusters()
{
    auto kern = gemm2_kernel<kNormNone, false, BN, STAGES, NSUB, false>;
    constexpr int smem = Gemm2Smem<BN, STAGES, NSUB>::alloc;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
    return n;
}

template <int BN, int STAGES, int NSUB>
int launch_gemm2_bn(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl,
                    cudaStream_t stream)
{
#define NGR_CASE2(N_, B_)                                                         \
    if (norm == N_ && bf16 == B_)                                                 \
        return launch_gemm2_variant<N_, B_, BN, STAGES, NSUB, false>(args, grid, pdl, stream);
    NGR_CASE2(kNormLayer, false)
    NGR_CASE2(kNormLayer, true)
    NGR_CASE2(kNormRms, false)
    NGR_CASE2(kNormRms, true)
    NGR_CASE2(kNormNone, false)
    NGR_CASE2(kNormNone, true)
    NGR_CASE2(kNormFoldLayer, false)
    NGR_CASE2(kNormFoldLayer, true)
    NGR_CASE2(kNormFoldRms, false)
    NGR_CASE2(kNormFoldRms, true)
#undef NGR_CASE2
    return -9;
}

// The gated (SwiGLU) tiles: norm none / LayerNorm / RMSNorm.
template <int BN, int STAGES>
int launch_gemm2_gated_bn(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl,
                          cudaStream_t stream)
{
#define NGR_CASEG(N_, B_)                                                         \
    if (norm == N_ && bf16 == B_)                                                 \
        return launch_gemm2_variant<N_, B_, BN, STAGES, 2, true>(args, grid, pdl, stream);
    NGR_CASEG(kNormLayer, false)
    NGR_CASEG(kNormLayer, true)
    NGR_CASEG(kNormRms, false)
    NGR_CASEG(kNormRms, true)
    NGR_CASEG(kNormNone, false)
    NGR_CASEG(kNormNone, true)
#undef NGR_CASEG
    return -9;
}

}  // namespace ngr
