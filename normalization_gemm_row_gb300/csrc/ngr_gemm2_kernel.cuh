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
// Synchronization (barriers are per CTA unless marked "leader"):
//   full[s]        with a norm: this CTA's copies landed (its producer's
//                  expect_tx); without: the leader's, on which both CTAs'
//                  copies complete (cta_group::2 TMA) -- the MMA waits on it;
//   ready[s]       leader, with a norm: each transform warp of both CTAs
//                  arrives once its CTA's stage is normalized;
//   empty[s]       the leader's tcgen05.commit, multicast to both CTAs;
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

// Where the normalized A operand lives in the CTA-pair kernel with a norm:
// 1 = tensor memory (written with tcgen05.st by row-owning threads; the
// MMAs read it from there), 0 = shared memory (normalized in place, like
// the single-CTA kernel).  One switch for one-sub-tile tiles, one for
// two-sub-tile tiles.
#ifndef NGR_PAIR_A_TMEM
#define NGR_PAIR_A_TMEM 0
#endif
#ifndef NGR_PAIR_A_TMEM_WIDE
#define NGR_PAIR_A_TMEM_WIDE 0
#endif
constexpr int kMaxASlots = 8;
// Column parts per stage of the in-place transform (1, 2 or 4): the MMAs of
// a part's K steps are issued once that part of both CTAs' stages is
// normalized.
#ifndef NGR_TRANSFORM_PARTS
#define NGR_TRANSFORM_PARTS 2
#endif
constexpr int kMaxParts = 4;

template <int BN, int STAGES, int NSUB>
struct Gemm2Smem {
    static constexpr int kA = kBM * kBK * 2;          // 16 KB: this CTA's 128 x rows
    static constexpr int kBSub = (BN / 2) * kBK * 2;  // this CTA's BN/2 W rows of one sub-tile
    static constexpr int kB = NSUB * kBSub;
    static constexpr int kGB = 2 * kBK * 4;           // FP32 gamma[64], beta[64]
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + STAGES * kA;
    static constexpr int off_g = off_b + STAGES * kB;
    static constexpr int off_bar = off_g + STAGES * kGB;
    static constexpr int n_bars = (2 + kMaxParts) * STAGES + 5 + kMaxASlots;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;
};


// The transform role of the CTA-pair kernel with A in tensor memory.
// A slot holds SLOT_K of a k block's 64 columns (SLOT_K / 2 tensor-memory
// columns of packed 16-bit pairs); a k block fills HALVES = 64 / SLOT_K
// slots, the j-th of the running sequence going to slot j % SLOTS, which is
// free once the MMAs that read its previous contents have completed
// (a_free, committed by the MMA issuer to both CTAs).  With one slot per k
// block, transform group g takes the k blocks with running index
// it % groups == g; with two, group h fills slot half h of every k block.
// Each warp covers the tensor-memory lane quarter warp % 4, and each lane
// one row: it reads its row's raw x chunks from the swizzled shared-memory
// stage (only read), normalizes them in FP32, packs them to 16-bit pairs
// and stores them with tcgen05.st.
template <int NORM, bool BF16, int STAGES, int KA, int SLOTS, int HALVES, typename M0Fn,
          typename KbFn, typename ArriveFn>
__device__ __forceinline__ void transform_role_tmem(
    int t, int tile0, int tile_step, int num_tiles, KbFn kb_count, int M, const float2 *stats,
    const uint8_t *sA, const float *sG, uint64_t *full, uint64_t *a_free, uint32_t tmem_base,
    uint32_t a_col0, const WaitCtx &wc, M0Fn m0_of, ArriveFn arrive)
{
    constexpr int kChunks = 8 / HALVES;   // 16-byte chunks of a row per slot
    constexpr int kCols = kChunks * 4;    // tensor-memory columns per slot
    static_assert(KA > 0 && kGroupThreads == 128, "a group must cover the four lane quarters");
    static_assert(HALVES == 1 || (HALVES == 2 && kTransformGroups == 2), "one group per slot half");
    const int g = t / kGroupThreads;
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;   // lane quarter this warp may access
    const int r = q * 32 + lane;            // row of the 128-row tile
    const int sw = r & 7;
    const int h = HALVES > 1 ? g : 0;       // slot half this thread fills
    const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + a_col0;
    pdl_wait();
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    for (int tile = tile0; tile < num_tiles; tile += tile_step) {
        const int row = m0_of(tile) + r;
        float2 st = make_float2(0.f, 0.f);
        if (row < M) st = stats[row];
        const float2 so = make_float2(st.y, -st.x * st.y);
        const int k_blocks = kb_count(tile);
        for (int kb = 0; kb < k_blocks; ++kb, ++it) {
            if (HALVES > 1 || it % kTransformGroups == g) {
                if (!mbar_wait_warp(&full[stage], phase, wc)) return;
                const int sidx = it * HALVES + h;
                const int slot = sidx % SLOTS;
                const int use = sidx / SLOTS;
                if (use > 0 && !mbar_wait_warp(&a_free[slot], (use - 1) & 1, wc)) return;
                tc_fence_after();
                const uint8_t *xrow = sA + stage * KA + r * 128;
                const float *gs = sG + stage * 2 * kBK;
                uint32_t packed[kCols];
#pragma unroll
                for (int c0 = 0; c0 < kChunks; ++c0) {
                    const int c = h * kChunks + c0;
                    const uint4 v = *reinterpret_cast<const uint4 *>(xrow + ((c ^ sw) << 4));
                    const float4 g0 = *reinterpret_cast<const float4 *>(gs + 8 * c);
                    const float4 g1 = *reinterpret_cast<const float4 *>(gs + 8 * c + 4);
                    const float2 gg[4] = {make_float2(g0.x, g0.y), make_float2(g0.z, g0.w),
                                          make_float2(g1.x, g1.y), make_float2(g1.z, g1.w)};
                    float2 bb[4];
                    if constexpr (NORM == kNormLayer) {
                        const float4 b0 = *reinterpret_cast<const float4 *>(gs + kBK + 8 * c);
                        const float4 b1 = *reinterpret_cast<const float4 *>(gs + kBK + 8 * c + 4);
                        bb[0] = make_float2(b0.x, b0.y);
                        bb[1] = make_float2(b0.z, b0.w);
                        bb[2] = make_float2(b1.x, b1.y);
                        bb[3] = make_float2(b1.z, b1.w);
                    }
                    const uint4 o = transform8_pk<NORM, BF16>(v, so, gg, bb);
                    packed[4 * c0 + 0] = o.x;
                    packed[4 * c0 + 1] = o.y;
                    packed[4 * c0 + 2] = o.z;
                    packed[4 * c0 + 3] = o.w;
                }
                const uint32_t taddr = tbase + static_cast<uint32_t>(slot * kCols);
                if constexpr (kCols == 32) tmem_st32(taddr, packed);
                else tmem_st16(taddr, packed);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive(stage);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
    }
}

template <int NORM, bool BF16, int BN, int STAGES, int NSUB, bool GATED>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm2_kernel(const __grid_constant__ GemmArgs args)
{
    using L = Gemm2Smem<BN, STAGES, NSUB>;
    constexpr bool kNorm = NORM == kNormLayer || NORM == kNormRms;  // transform stage
    constexpr int kTW = NSUB * BN;                 // accumulator columns of a tile
    constexpr int kOutW = GATED ? BN : kTW;        // output columns of a tile
    static_assert(!GATED || (NSUB == 2 && !is_fold(NORM)), "gated tiles: gate and up sub-tiles");
    // Bytes one stage of this CTA receives when n_sub sub-tiles are in range.
    auto stage_tx = [](int n_sub) -> uint32_t {
        return static_cast<uint32_t>(L::kA + n_sub * L::kBSub + (kNorm ? L::kGB : 0));
    };
    // Accumulators (two of kTW columns when they fit and A is not in tensor
    // memory, else one), then the A slots: a whole k block per slot with one
    // sub-tile, half a k block with two (only 64 columns are left beside a
    // 448-column accumulator).
    constexpr uint32_t kTmemCols = 512;
    constexpr int kSlotK = NSUB > 1 ? 32 : kBK;        // K columns of x per A slot
    constexpr int kHalvesA = kBK / kSlotK;             // A slots per k block
    constexpr int kSlotCols = kSlotK / 2;              // tensor-memory columns per slot
    // (A in tensor memory needs at least two k blocks' slots beside one
    // accumulator: not with a 512-column tile.)
    constexpr bool kATmem = kNorm && !GATED && (NSUB > 1 ? NGR_PAIR_A_TMEM_WIDE : NGR_PAIR_A_TMEM) &&
                            static_cast<int>(kTmemCols) - kTW >= 2 * kHalvesA * kSlotCols;
    constexpr int kAccBufs = (kATmem || NSUB > 1) ? 1 : 2;
    constexpr uint32_t kACol0 = kAccBufs * kTW;
    constexpr int kSlotsFit = static_cast<int>((kTmemCols - kACol0) / kSlotCols);
    constexpr int kASlots = kSlotsFit < kMaxASlots ? kSlotsFit : kMaxASlots;
    static_assert(!kATmem || (kASlots >= 2 * kHalvesA && kASlots % (kHalvesA * kTransformGroups) == 0),
                  "tensor memory: accumulator + A slots");
    constexpr uint32_t kIdesc = idesc_f16(BF16, 2 * kBM, BN);
    // ready[s] arrivals: one per warp of each transform group that works on
    // the stage, in each CTA (used with a norm only).
    constexpr uint32_t kReadyCount = 2 * kGroupWarps * (kATmem ? kHalvesA : 1);
    constexpr int kParts = (kNorm && !kATmem) ? NGR_TRANSFORM_PARTS : 1;
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
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *ready = bars + 2 * STAGES;        // [STAGES * kParts] part of both stages normalized
    uint64_t *acc_full = bars + (2 + kMaxParts) * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_full + 4;
    uint64_t *a_free = acc_full + 5;            // [kMaxASlots] A slot read by the MMAs (commit, multicast)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        if (args.zero_err && blockIdx.x == 0) *args.err = 0;
        prefetch_tmap(&args.map_a);
        prefetch_tmap(&args.map_b);
        if constexpr (GATED) prefetch_tmap(&args.map_b2);
        if constexpr (kNorm) prefetch_tmap(&args.map_gb);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            for (int p = 0; p < kParts; ++p) mbar_init(&ready[s * kParts + p], kReadyCount);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 2 * kDrainWarps);
        }
        mbar_init(drain, 1);
        for (int j = 0; j < kMaxASlots; ++j) mbar_init(&a_free[j], 1);
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
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
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
                    if (!mbar_wait_spin(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    const int kc = kb * kBK;
                    uint8_t *sb = sB + stage * L::kB;
                    if constexpr (kNorm) {
                        // Each CTA normalizes its own stage: local barrier.
                        mbar_arrive_expect_tx(&full[stage], tx);
                        tma_load_2d(sA + stage * L::kA, &args.map_a, &full[stage], kc, m0, pol_x);
                        for (int j = 0; j < n_sub; ++j)
                            tma_load_2d(sb + j * L::kBSub, wmap(j), &full[stage], kc, wrow(j), pol_w);
                        tma_load_2d(sG + stage * 2 * kBK, &args.map_gb, &full[stage], kc, 0, pol_x);
                    } else {
                        // Both CTAs' copies complete on the leader's barrier,
                        // which expects the bytes of both.
                        const uint32_t fb = full_leader + 8u * static_cast<uint32_t>(stage);
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * tx);
                        tma_load_2d_pair(sA + stage * L::kA, &args.map_a, fb, kc, m0, pol_x);
                        for (int j = 0; j < n_sub; ++j)
                            tma_load_2d_pair(sb + j * L::kBSub, wmap(j), fb, kc, wrow(j), pol_w);
                    }
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Copies signalled on this CTA's own barriers: wait for the last
            // fills.  (Without a norm the peer's copies complete on the
            // leader's barriers; the leader's MMAs, and so the final cluster
            // barrier, come after them.)
            if (kNorm || leader) {
                const int outstanding = fills < STAGES ? static_cast<int>(fills) : STAGES;
                for (int j = 1; j <= outstanding; ++j) {
                    int s = stage - j;
                    uint32_t p = phase;
                    if (s < 0) { s += STAGES; p ^= 1u; }
                    mbar_wait(&full[s], p, wc);
                }
            }
        }
    } else if (warp == 1) {
        if (leader && lane == 0) {
            // ------------------------------------- MMA issuer (even CTA)
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int it = 0;
            bool ok = true;
            for (int u = cluster; ok && u < num_units; u += n_clusters) {
                const int tile = unit_tile(u);
                const int kb0 = unit_kb0(u);
                if (!mbar_wait_spin(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kTW);
                const int n_sub = GATED ? 2 : min(NSUB, (args.N - (tile / m_tiles) * kTW + BN - 1) / BN);
                for (int kb = kb0, kb_end = unit_kb1(u); kb < kb_end; ++kb) {
                    if (!mbar_wait_spin(kNorm ? &ready[stage * kParts] : &full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t b_addr = smem_u32(sB + stage * L::kB);
                    if constexpr (kATmem) {
#pragma unroll
                        for (int hh = 0; hh < kHalvesA; ++hh) {
                            const int slot = (it * kHalvesA + hh) % kASlots;
                            const uint32_t a_tmem = tmem_base + kACol0 +
                                                    static_cast<uint32_t>(slot * kSlotCols);
#pragma unroll
                            for (int k = 0; k < kSlotK / kUmmaK; ++k) {
                                const int kk = hh * (kSlotK / kUmmaK) + k;   // K step in the block
#pragma unroll
                                for (int j = 0; j < NSUB; ++j) {
                                    if (j < n_sub)
                                        umma_f16_ts_pair(d_tmem + static_cast<uint32_t>(j * BN),
                                                         a_tmem + static_cast<uint32_t>(k * (kUmmaK / 2)),
                                                         sdesc_kmajor_sw128(b_addr + j * L::kBSub + kk * 32),
                                                         kIdesc, (kb != kb0 || kk != 0) ? 1u : 0u);
                                }
                            }
                            umma_commit_pair(&a_free[slot], 0x3);
                        }
                    } else {
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
                    }
                    if (!ok) break;
                    umma_commit_pair(&empty[stage], 0x3);
                    ++it;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[acc], 0x3);
                if (++acc == kAccBufs) { acc = 0; acc_phase ^= 1u; }
            }
            umma_commit_pair(drain, 0x1);
            mbar_wait(drain, 0, wc);
        }
    } else if (warp >= kTransformWarp0) {
        const bool epi_warp = warp >= kEpilogueWarp0;
        if (!epi_warp) {
            const int t = threadIdx.x - kTransformWarp0 * 32;
            if constexpr (kATmem) {
                // ------------------------------------------ transform (A -> TMEM)
                transform_role_tmem<NORM, BF16, STAGES, L::kA, kASlots, kHalvesA>(
                    t, cluster, n_clusters, num_units, [&](int u) { return unit_kb1(u) - unit_kb0(u); },
                    args.M, args.stats, sA, sG, full, a_free, tmem_base, kACol0, wc,
                    [&](int u) { return (unit_tile(u) % m_tiles) * 2 * kBM + static_cast<int>(rank) * kBM; },
                    [&](int st) { mbar_arrive_cluster(ready_leader + 8u * static_cast<uint32_t>(st)); });
            } else if constexpr (kNorm) {
                // ----------------------------------------- transform (A in place)
                transform_role<NORM, BF16, STAGES, L::kA, kParts>(
                    t, cluster, n_clusters, num_units, [&](int u) { return unit_kb1(u) - unit_kb0(u); },
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
            if constexpr (is_fold(NORM)) pdl_wait();  // row statistics from the previous grid
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
                if (!mbar_wait_warp(&acc_full[cur], cur_phase, wc)) break;
                tc_fence_after();
                const int row = (tile % m_tiles) * 2 * kBM + static_cast<int>(rank) * kBM + q * 32 + lane;
                const float2 so = fold_row_scale<NORM>(args, row);
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
                        for (int j = 0; j < 32; ++j)
                            v[j] = silu_f(__uint_as_float(rg[j])) * __uint_as_float(ru[j]);
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
                            epilogue_store32<NORM, BF16>(v, row, nt0 + c, args, so);
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
                        epilogue_store32<NORM, BF16>(v, row, nt0 + c, args, so);
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
    constexpr int smem = Gemm2Smem<BN, STAGES, NSUB>::alloc;
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
