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
//  - the (weight tile, 64-wide k block) units are split evenly over one CTA
//    per SM as one contiguous run each, so every SM streams the same number
//    of weight bytes without a tail wave; a run that covers part of a weight
//    tile leaves an FP32 partial of that tile (split-K);
//  - the tokens arrive already normalized: at these sizes the statistics
//    kernel writes the normalized rows once (at most 32 x K 16-bit values,
//    which stay in L2), computed exactly as the tile kernel's transform
//    does, instead of every weight tile re-normalizing the same k slice on
//    the weight stream's critical path; with a folded weight the raw rows
//    are used and the statistics are applied in the epilogue;
//  - each epilogue warp owns 32 weight rows: it writes its partial, and the
//    last of the CTAs sharing a tile (an atomic counter per 32-row slice)
//    sums the partials in a fixed order (deterministic), adds the bias,
//    applies the activation and stores y.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ngr_gemm_kernel.cuh"
#include "ngr_internal.h"
#include "ngr_ptx.cuh"

namespace ngr {

template <int MN, int STAGES>
struct DecodeSmem {
    static constexpr int kW = 128 * kBK * 2;   // 16 KB weight tile
    static constexpr int kX = MN * kBK * 2;    // MN x 128 B token tile
    static constexpr int off_w = 0;
    static constexpr int off_x = off_w + STAGES * kW;
    static constexpr int off_bar = off_x + STAGES * kX;
    static constexpr int n_bars = 3 * STAGES + 5;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;
};

// CTA that owns unit u when `units` units are split into `grid` contiguous
// runs, run i = [floor(i units / grid), floor((i+1) units / grid)).
__host__ __device__ __forceinline__ long long decode_owner(long long u, long long units,
                                                           long long grid)
{
    return ((u + 1) * grid - 1) / units;
}

template <int NORM, bool BF16, int MN, int STAGES>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    decode_kernel(const __grid_constant__ DecodeArgs args)
{
    using L = DecodeSmem<MN, STAGES>;
    static_assert(NORM == kNormNone || is_fold(NORM), "tokens arrive normalized or the weight is folded");
    constexpr uint32_t kTx = L::kW + L::kX;
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
    uint64_t *acc_full = bars + 3 * STAGES;
    uint64_t *acc_empty = bars + 3 * STAGES + 2;
    uint64_t *drain = bars + 3 * STAGES + 4;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};

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

    const long long units = args.units;
    const long long G = args.grid;
    const long long u_begin = (static_cast<long long>(blockIdx.x) * units) / G;
    const long long u_end = (static_cast<long long>(blockIdx.x + 1) * units) / G;
    const int KB = args.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // The tokens may come from the previous grid (the statistics
            // kernel's normalized rows, or the first product of a chain);
            // the weights never do.  The first STAGES fills therefore start
            // their weight boxes at once and add the token boxes after the
            // dependency wait, so the weight stream overlaps the previous
            // grid's tail.
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();  // each weight byte is read once
            bool waited = false;
            int deferred_kc[STAGES];
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            for (long long u = u_begin; u < u_end; ++u) {
                const int tile = static_cast<int>(u / KB);
                const int kc = static_cast<int>(u % KB) * kBK;
                if (!waited && fills == STAGES) {
                    pdl_wait();
                    waited = true;
                    for (int s2 = 0; s2 < STAGES; ++s2)
                        tma_load_2d(sX + s2 * L::kX, &args.map_x, &full[s2], deferred_kc[s2], 0, pol_x);
                }
                if (!mbar_wait_spin(&empty[stage], phase ^ 1u, wc)) break;
                mbar_arrive_expect_tx(&full[stage], kTx);
                tma_load_2d(sW + stage * L::kW, &args.map_w, &full[stage], kc, tile * 128, pol_w);
                if (waited)
                    tma_load_2d(sX + stage * L::kX, &args.map_x, &full[stage], kc, 0, pol_x);
                else
                    deferred_kc[stage] = kc;
                ++fills;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!waited) {   // fewer fills than stages (or a failed wait)
                pdl_wait();
                for (int s2 = 0; s2 < static_cast<int>(fills < STAGES ? fills : STAGES); ++s2)
                    tma_load_2d(sX + s2 * L::kX, &args.map_x, &full[s2], deferred_kc[s2], 0, pol_x);
            }
            const int outstanding = fills < STAGES ? static_cast<int>(fills) : STAGES;
            for (int j = 1; j <= outstanding; ++j) {
                int s = stage - j;
                uint32_t p = phase;
                if (s < 0) { s += STAGES; p ^= 1u; }
                mbar_wait(&full[s], p, wc);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // -------------------------------------------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            long long u = u_begin;
            while (ok && u < u_end) {
                const long long tile = u / KB;
                const long long seg_end = (tile + 1) * KB < u_end ? (tile + 1) * KB : u_end;
                if (!mbar_wait_spin(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MN);
                bool first = true;
                for (; u < seg_end; ++u) {
                    if (!mbar_wait_spin(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sW + stage * L::kW);
                    const uint32_t b_addr = smem_u32(sX + stage * L::kX);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        umma_f16_ss(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32),
                                    sdesc_kmajor_sw128(b_addr + k * 32), kIdesc,
                                    (!first || k != 0) ? 1u : 0u);
                    }
                    first = false;
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait(drain, 0, wc);
        }
    } else if (warp >= 8) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;
        const int M = args.M, N = args.N;
        pdl_wait();  // the split-K counters are zeroed by the previous grid
        int acc = 0;
        uint32_t acc_phase = 0;
        long long u = u_begin;
        while (u < u_end) {
            const long long tile = u / KB;
            const long long seg_end = (tile + 1) * KB < u_end ? (tile + 1) * KB : u_end;
            u = seg_end;
            if (!mbar_wait_warp(&acc_full[acc], acc_phase, wc)) break;
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

            const int n = static_cast<int>(tile) * 128 + q * 32 + lane;
            const long long first = decode_owner(tile * KB, units, G);
            const long long last = decode_owner(tile * KB + KB - 1, units, G);
            const int ncontrib = static_cast<int>(last - first + 1);
            bool finish = true;
            if (ncontrib > 1) {
                const int j = static_cast<int>(blockIdx.x - first);
                float *part = args.partials +
                              ((tile * kDecodeMaxContrib + j) * MN) * 128 + q * 32 + lane;
#pragma unroll
                for (int m = 0; m < MN; ++m) __stcg(part + m * 128, v[m]);
                __threadfence();
                int old = 0;
                if (lane == 0) old = atomicAdd(&args.counters[tile * 4 + q], 1);
                old = __shfl_sync(0xffffffffu, old, 0);
                finish = (old == ncontrib - 1);
                if (finish) {
                    __threadfence();
#pragma unroll
                    for (int m = 0; m < MN; ++m) v[m] = 0.f;
                    for (int jj = 0; jj < ncontrib; ++jj) {
                        const float *pp = args.partials +
                                          ((tile * kDecodeMaxContrib + jj) * MN) * 128 + q * 32 + lane;
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
    return mn <= 16 ? DecodeSmem<16, 10>::alloc : DecodeSmem<32, 10>::alloc;
}

// Largest grid (at most one CTA per SM) for which no 128-row weight tile is
// shared by more than kDecodeMaxContrib CTAs.
int plan_decode_grid(int64_t n_tiles, int64_t k_blocks, int num_sms)
{
    const long long units = n_tiles * k_blocks;
    long long g = num_sms < units ? num_sms : units;
    for (; g > 1; --g) {
        int worst = 1;
        for (long long t = 0; t < n_tiles; ++t) {
            const long long a = decode_owner(t * k_blocks, units, g);
            const long long b = decode_owner(t * k_blocks + k_blocks - 1, units, g);
            if (b - a + 1 > worst) worst = static_cast<int>(b - a + 1);
        }
        if (worst <= kDecodeMaxContrib) break;
    }
    return static_cast<int>(g < 1 ? 1 : g);
}

template <int NORM, bool BF16, int MN>
static int launch_decode_variant(const DecodeArgs &args, bool pdl, cudaStream_t stream)
{
    auto kern = decode_kernel<NORM, BF16, MN, 10>;
    constexpr int smem = DecodeSmem<MN, 10>::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return record_cuda_error("cudaFuncSetAttribute(max dynamic smem)", e, cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(args.grid));
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
    NGR_DCASE(kNormFoldLayer, false)
    NGR_DCASE(kNormFoldLayer, true)
    NGR_DCASE(kNormFoldRms, false)
    NGR_DCASE(kNormFoldRms, true)
#undef NGR_DCASE
    return -9;
}

}  // namespace ngr
