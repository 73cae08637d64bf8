// ngr_decode.cu -- the fused pre-norm linear layer for decode-sized M
// (M <= 32 tokens), where the weight stream, not the tensor core, bounds the
// time.
//
// Same computation as the tile kernel ("LayerNorm 融合算子如何让大模型推理再快
// 15%？深度拆解 ATB 的实现", §2.1 and §5.2 -- the fused layer at small batch),
// laid out for weight bandwidth:
//  - swap-AB: a 128-row weight tile is the UMMA M side and the (padded)
//    tokens the N side, so D^T[n, m] = sum_k W[n,k] a[m,k] fills all 128
//    tensor-memory lanes even for one token;
//  - the grid is k_groups x n_groups CTAs (one per SM): CTA (kg, ng) owns
//    the k blocks of group kg and the 128-row weight tiles of group ng, so
//    every SM streams about the same number of weight bytes;
//  - each CTA loads its slice of the tokens, x[0:MN, k range of kg], ONCE,
//    and (with a norm) normalizes it in shared memory with the same FP32
//    formula and single rounding as the tile kernel's transform.  The
//    normalized tokens exist only in that CTA's shared memory: nothing
//    normalized is written to device memory, and the weight stream never
//    waits for a normalization.  With a folded weight the raw slice is
//    used and the statistics are applied in the epilogue;
//  - each epilogue warp owns 32 weight rows: it writes the FP32 partial of
//    its k group, and the last of the k groups of a tile (an atomic counter
//    per 32-row slice) sums the partials in k-group order (deterministic),
//    adds the bias, applies the activation and stores y.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ngr_gemm_kernel.cuh"
#include "ngr_internal.h"
#include "ngr_ptx.cuh"

namespace ngr {

constexpr int kDecodeStages = 10;
// The token slice is loaded and normalized in this many parts of k blocks,
// so that the first tile's products start once the first part is ready.
constexpr int kDecodeSliceParts = 4;

// Shared memory: the weight ring, then the token slice (at most XKB k
// blocks of MN rows, each block one 128-byte-swizzled [MN x 64] box).
template <int MN>
struct DecodeSmem {
    static constexpr int kStages = kDecodeStages;
    static constexpr int kXKB = decode_max_kb(MN);
    static constexpr int kW = 128 * kBK * 2;   // 16 KB weight tile
    static constexpr int kXB = MN * kBK * 2;   // one k block of the tokens
    static constexpr int off_w = 0;
    static constexpr int off_x = off_w + kStages * kW;
    static constexpr int off_bar = off_x + kXKB * kXB;
    static constexpr int n_bars = 2 * kStages + 5 + 2 * kDecodeSliceParts;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;
};

template <int NORM, bool BF16, int MN>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs args)
{
    using L = DecodeSmem<MN>;
    constexpr int STAGES = L::kStages;
    constexpr bool kNorm = NORM == kNormLayer || NORM == kNormRms;   // normalize the slice
    constexpr uint32_t kTmemCols = 2 * MN <= 32 ? 32 : 64;
    constexpr uint32_t kIdesc = idesc_f16(BF16, 128, MN);
    static_assert(MN == 16 || MN == 32, "token tile");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sW = smem + L::off_w;
    uint8_t *sX = smem + L::off_x;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *acc_full = bars + 2 * STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_full + 4;
    uint64_t *x_full = acc_full + 5;                        // [parts] a part of the slice has landed
    uint64_t *x_ready = x_full + kDecodeSliceParts;         // [parts] ... and is normalized (4 warps)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};

    // This CTA's k blocks [kb0, kb0 + nkb) and weight tiles [t0, t1).
    const int kg = static_cast<int>(blockIdx.x) % args.k_groups;
    const int ng = static_cast<int>(blockIdx.x) / args.k_groups;
    const int kb0 = kg * args.kb_per_group;
    const int nkb = min(args.k_blocks, kb0 + args.kb_per_group) - kb0;
    const int t0 = static_cast<int>(static_cast<long long>(ng) * args.n_tiles / args.n_groups);
    const int t1 = static_cast<int>(static_cast<long long>(ng + 1) * args.n_tiles / args.n_groups);
    const int n_units = (t1 - t0) * nkb;
    // k blocks per slice part; part q holds local blocks [q pkb, (q + 1) pkb).
    const int pkb = (nkb + kDecodeSliceParts - 1) / kDecodeSliceParts;
    auto part_blocks = [&](int q) { return max(0, min(nkb, (q + 1) * pkb) - q * pkb); };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // The first kernel of a call clears the call's error word.
        if (args.zero_err && blockIdx.x == 0) *args.err = 0;
        prefetch_tmap(&args.map_w);
        prefetch_tmap(&args.map_x);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        mbar_init(drain, 1);
        for (int q = 0; q < kDecodeSliceParts; ++q) {
            mbar_init(&x_full[q], 1);
            mbar_init(&x_ready[q], 4);
        }
        fence_mbarrier_init();
    }
    if (warp == 2) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // The weights never come from the previous grid, the tokens may
            // (the first product of a chain writes them) and the statistics
            // do: the first STAGES weight boxes go out at once, the token
            // slice after the dependency wait.
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
            auto load_slice = [&]() {
                pdl_wait();
                for (int q = 0; q < kDecodeSliceParts; ++q) {
                    const int nb = part_blocks(q);
                    mbar_arrive_expect_tx(&x_full[q], static_cast<uint32_t>(nb * L::kXB));
                    for (int b = q * pkb; b < q * pkb + nb; ++b)
                        tma_load_2d(sX + b * L::kXB, &args.map_x, &x_full[q], (kb0 + b) * kBK, 0, pol_x);
                }
            };
            bool sliced = false;
            int stage = 0;
            uint32_t phase = 0;
            int fills = 0;
            bool ok = true;
            for (int u = 0; u < n_units; ++u) {
                if (!sliced && fills == STAGES) {
                    load_slice();
                    sliced = true;
                }
                if (!mbar_wait_spin(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                const int tile = t0 + u / nkb;
                const int kc = (kb0 + u % nkb) * kBK;
                mbar_arrive_expect_tx(&full[stage], L::kW);
                tma_load_2d(sW + stage * L::kW, &args.map_w, &full[stage], kc, tile * 128, pol_w);
                ++fills;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!sliced) load_slice();
            // Wait for the copies still in flight before the CTA may exit.
            const int outstanding = fills < STAGES ? fills : STAGES;
            for (int j = 1; ok && j <= outstanding; ++j) {
                int s = stage - j;
                uint32_t p = phase;
                if (s < 0) { s += STAGES; p ^= 1u; }
                mbar_wait_long(&full[s], p, wc);
            }
            for (int q = 0; ok && q < kDecodeSliceParts; ++q) mbar_wait_long(&x_full[q], 0, wc);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // -------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const uint32_t x_addr = smem_u32(sX);
            for (int t = t0; ok && t < t1; ++t) {
                if (!mbar_wait_spin(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MN);
                for (int b = 0; b < nkb; ++b) {
                    // the first tile waits for each part of the slice
                    if (t == t0 && b % pkb == 0 && !mbar_wait_spin(&x_ready[b / pkb], 0, wc)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait_spin(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sW + stage * L::kW);
                    const uint32_t b_addr = x_addr + static_cast<uint32_t>(b * L::kXB);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        umma_f16_ss(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32),
                                    sdesc_kmajor_sw128(b_addr + k * 32), kIdesc,
                                    (b != 0 || k != 0) ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait_long(drain, 0, wc);
        }
    } else if (warp >= 4 && warp < 8) {
        // -------------------------------- token slice: normalize in place
        // Thread t owns the 8-column chunks t, t + 128, ... of the slice and
        // normalizes them in every row, so its gamma/beta are loaded once
        // and the rows' statistics come from shared memory.  16-byte chunk c
        // of row r in k block b sits at b kXB + r 128 + ((c ^ (r & 7)) << 4)
        // (128-byte swizzle); rows at or past M are the zero fill and are
        // left alone, columns at or past K are made zero.
        const int tid = threadIdx.x - 128;
        const int rows = min(args.M, MN);
        __shared__ float2 row_so[MN];   // (rstd, -mu rstd) of each token
        if constexpr (kNorm) {
            pdl_wait();   // the statistics and FP32 gamma/beta come from the previous grid
            if (tid < rows) {
                const float2 st = args.stats[tid];
                row_so[tid] = make_float2(st.y, -st.x * st.y);
            }
            named_bar_sync(1, 128);
        }
        for (int q = 0; q < kDecodeSliceParts; ++q) {
            if (!mbar_wait_warp_long(&x_full[q], 0, wc)) break;
            if constexpr (kNorm) {
                constexpr int kRowBatch = 8;
                const int cc_end = (q * pkb + part_blocks(q)) * 8;
                for (int cc = q * pkb * 8 + tid; cc < cc_end; cc += 128) {
                    const int b = cc >> 3, c = cc & 7;
                    const int col = (kb0 + b) * kBK + c * 8;
                    const bool valid = col < args.K;
                    float2 gg[4], bb[4];
                    if (valid) {
                        const float4 g0 = __ldg(reinterpret_cast<const float4 *>(args.gamma_f + col));
                        const float4 g1 = __ldg(reinterpret_cast<const float4 *>(args.gamma_f + col + 4));
                        gg[0] = make_float2(g0.x, g0.y);
                        gg[1] = make_float2(g0.z, g0.w);
                        gg[2] = make_float2(g1.x, g1.y);
                        gg[3] = make_float2(g1.z, g1.w);
                        if constexpr (NORM == kNormLayer) {
                            const float4 b0 = __ldg(reinterpret_cast<const float4 *>(args.beta_f + col));
                            const float4 b1 = __ldg(reinterpret_cast<const float4 *>(args.beta_f + col + 4));
                            bb[0] = make_float2(b0.x, b0.y);
                            bb[1] = make_float2(b0.z, b0.w);
                            bb[2] = make_float2(b1.x, b1.y);
                            bb[3] = make_float2(b1.z, b1.w);
                        }
                    }
                    uint8_t *blk = sX + b * L::kXB;
                    for (int r0 = 0; r0 < rows; r0 += kRowBatch) {
                        uint4 v[kRowBatch];
#pragma unroll
                        for (int i = 0; i < kRowBatch; ++i) {
                            const int r = r0 + i;
                            if (r < rows)
                                v[i] = *reinterpret_cast<const uint4 *>(blk + r * 128 + ((c ^ (r & 7)) << 4));
                        }
#pragma unroll
                        for (int i = 0; i < kRowBatch; ++i) {
                            const int r = r0 + i;
                            if (r < rows)
                                *reinterpret_cast<uint4 *>(blk + r * 128 + ((c ^ (r & 7)) << 4)) =
                                    valid ? transform8_pk<NORM, BF16>(v[i], row_so[r], gg, bb)
                                          : make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&x_ready[q]);
        }
    } else if (warp >= 8) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int M = args.M, N = args.N;
        const int G = args.k_groups;
        pdl_wait();  // the split-K counters are zeroed by the previous grid
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = t0; t < t1; ++t) {
            if (!mbar_wait_warp_long(&acc_full[acc], acc_phase, wc)) break;
            tc_fence_after();
            float v[MN];
            {
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(acc * MN);
                uint32_t r[16];
#pragma unroll
                for (int h = 0; h < MN / 16; ++h) {
                    tmem_ld16(taddr + 16 * h, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[16 * h + j] = __uint_as_float(r[j]);
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }

            const int n = t * 128 + q * 32 + lane;
            bool finish = true;
            if (G > 1) {
                float *part = args.partials + ((static_cast<long long>(t) * kDecodeMaxGroups + kg) * MN) * 128 +
                              q * 32 + lane;
#pragma unroll
                for (int m = 0; m < MN; ++m) __stcg(part + m * 128, v[m]);
                __threadfence();
                int old = 0;
                if (lane == 0) old = atomicAdd(&args.counters[t * 4 + q], 1);
                old = __shfl_sync(0xffffffffu, old, 0);
                finish = (old == G - 1);
                if (finish) {
                    __threadfence();
#pragma unroll
                    for (int m = 0; m < MN; ++m) v[m] = 0.f;
                    for (int jj = 0; jj < G; ++jj) {
                        const float *pp = args.partials +
                                          ((static_cast<long long>(t) * kDecodeMaxGroups + jj) * MN) * 128 +
                                          q * 32 + lane;
#pragma unroll
                        for (int m = 0; m < MN; ++m) v[m] += __ldcg(pp + m * 128);
                    }
                }
            }
            if (finish && n < N) {
                float bn = 0.f, cn = 0.f;
                if constexpr (is_fold(NORM)) {
                    bn = args.fold_b[n];
                    if constexpr (NORM == kNormFoldLayer) cn = args.fold_c[n];
                } else if (args.bias != nullptr) {
                    bn = to_float1<BF16>(args.bias, n);
                }
                uint16_t *y = static_cast<uint16_t *>(args.y);
                for (int m = 0; m < M && m < MN; ++m) {
                    float z;
                    if constexpr (is_fold(NORM)) {
                        // y = rstd acc - rstd mu c + b'
                        const float2 st = args.stats[m];
                        z = fmaf(v[m], st.y, fmaf(-st.x * st.y, cn, bn));
                    } else {
                        z = v[m] + bn;
                    }
                    if (args.act == kActSilu) z = silu_f(z);
                    else if (args.act == kActRelu) z = fmaxf(z, 0.0f);
                    else if (args.act == kActGelu) z = gelu_f(z);
                    if (args.residual != nullptr)
                        z += to_float1<BF16>(static_cast<const uint16_t *>(args.residual) +
                                                 static_cast<long long>(m) * N, n);
                    uint16_t o;
                    if constexpr (BF16) {
                        __nv_bfloat16 h = __float2bfloat16_rn(z);
                        o = *reinterpret_cast<uint16_t *>(&h);
                    } else {
                        __half h = __float2half_rn(z);
                        o = *reinterpret_cast<uint16_t *>(&h);
                    }
                    y[static_cast<long long>(m) * N + n] = o;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

size_t decode_smem_bytes(int mn)
{
    return mn <= 16 ? DecodeSmem<16>::alloc : DecodeSmem<32>::alloc;
}

// The k-group x n-group grid: at most one CTA per SM and kDecodeMaxGroups
// k groups, each group's token slice within the kernel's slice buffer; the
// plan minimises the largest number of (weight tile, k block) units a CTA
// streams, and among equal plans takes fewer k groups (fewer partials).
DecodePlan plan_decode(int64_t n_tiles, int64_t k_blocks, int mn, int num_sms)
{
    DecodePlan best{1, static_cast<int>(k_blocks), 1};
    long long best_cost = -1;
    const int max_kb = decode_max_kb(mn);
    for (int g = 1; g <= kDecodeMaxGroups && g <= k_blocks; ++g) {
        const int kbpg = static_cast<int>((k_blocks + g - 1) / g);
        if (kbpg > max_kb) continue;
        const int groups = static_cast<int>((k_blocks + kbpg - 1) / kbpg);   // non-empty groups
        long long gn = num_sms / groups;
        if (gn > n_tiles) gn = n_tiles;
        if (gn < 1) continue;
        const long long cost = ((n_tiles + gn - 1) / gn) * kbpg;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = DecodePlan{groups, kbpg, static_cast<int>(gn)};
        }
    }
    return best;
}

template <int NORM, bool BF16, int MN>
static int launch_decode_variant(const DecodeArgs &args, bool pdl, cudaStream_t stream)
{
    auto kern = decode_kernel<NORM, BF16, MN>;
    constexpr int smem = DecodeSmem<MN>::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return record_cuda_error("cudaFuncSetAttribute(max dynamic smem)", e, cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(args.k_groups * args.n_groups));
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, kern, args);
    return e == cudaSuccess ? 0 : record_cuda_error("cudaLaunchKernelEx", e, cudaGetErrorString(e));
}

int launch_decode(int norm, bool bf16, int mn, const DecodeArgs &args, bool pdl,
                  cudaStream_t stream)
{
#define NGR_DCASE(N_, B_)                                                         \
    if (norm == N_ && bf16 == B_)                                                 \
        return mn <= 16 ? launch_decode_variant<N_, B_, 16>(args, pdl, stream)    \
                        : launch_decode_variant<N_, B_, 32>(args, pdl, stream);
    NGR_DCASE(kNormNone, false)
    NGR_DCASE(kNormNone, true)
    NGR_DCASE(kNormLayer, false)
    NGR_DCASE(kNormLayer, true)
    NGR_DCASE(kNormRms, false)
    NGR_DCASE(kNormRms, true)
    NGR_DCASE(kNormFoldLayer, false)
    NGR_DCASE(kNormFoldLayer, true)
    NGR_DCASE(kNormFoldRms, false)
    NGR_DCASE(kNormFoldRms, true)
#undef NGR_DCASE
    return -9;
}

}  // namespace ngr
