// ngr_gemm_kernel.cuh -- the fused pre-norm linear layer as one persistent,
// warp-specialised tcgen05 kernel (steps a2, a3, a4 of the hot path).
//
// What it computes, per output tile y[m0:m0+128, n0:n0+BN]:
//   a[i,k] = (x[i,k] - mu_i) rstd_i gamma_k + beta_k      (LayerNorm)
//          =  x[i,k] rstd_i gamma_k                      (RMSNorm)
//          =  x[i,k]                                     (no norm)
//   y[i,n] = act(sum_k a[i,k] W[n,k] + bias_n)
// "LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现", §2.1
// (tile-level fusion: the normalized tile stays on chip and feeds the
// matmul) and §3.1 (the vector unit normalizes while the cube unit fetches
// weights); "昇腾CANN的MatMul融合玩法，让大模型推理快3倍", §二 strategies 1-3.
//
// GB300 design.  One CTA per SM loops over output tiles (m fastest, so the
// CTAs resident at one time share weight tiles through L2).  Warp roles:
//   warp 0      TMA producer: x tile [128 x 64] and W tile [BN x 64] (both
//               in the 128-byte swizzled K-major layout the tensor core
//               reads), plus FP32 gamma/beta [64] (converted once per call
//               by the statistics kernel), into a STAGES-deep ring;
//   warp 1      MMA issuer: 4 x tcgen05.mma (K = 16 each) per stage into an
//               FP32 accumulator in tensor memory; tcgen05.commit frees the
//               stage and, at the end of a tile, hands the accumulator over;
//   warp 2      allocates and frees tensor memory (2 x BN columns: the
//               epilogue drains one accumulator while the next tile's
//               mainloop fills the other);
//   warps 4-7   transform: normalize + affine the x tile IN PLACE in shared
//               memory (thread t owns row t; FP32 math, one rounding to the
//               16-bit operand type), then fence the generic-proxy writes for
//               the tensor core and signal the MMA warp;
//   warps 8-11  epilogue: tcgen05.ld of its 32 accumulator rows, + bias,
//               SiLU, round to fp16/bf16, 16-byte stores to y.
// The normalized activations exist only in shared memory.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ngr_internal.h"
#include "ngr_ptx.cuh"

namespace ngr {

template <bool BF16>
__device__ __forceinline__ float2 to_float2(uint32_t w)
{
    if constexpr (BF16)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    else
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

template <bool BF16>
__device__ __forceinline__ uint32_t from_float2(float a, float b)
{
    if constexpr (BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

template <bool BF16>
__device__ __forceinline__ float to_float1(const void *p, int i)
{
    if constexpr (BF16)
        return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
    else
        return __half2float(static_cast<const __half *>(p)[i]);
}

__device__ __forceinline__ float silu_f(float z)
{
    return __fdividef(z, 1.0f + __expf(-z));
}

// Normalize + affine 8 consecutive elements held as 4 packed 16-bit pairs.
// g and b point at the FP32 gamma/beta of those 8 columns.
template <int NORM, bool BF16>
__device__ __forceinline__ uint4 transform8(uint4 v, float sc, float of,
                                            const float *g, const float *b)
{
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float4 g0 = *reinterpret_cast<const float4 *>(g);
    const float4 g1 = *reinterpret_cast<const float4 *>(g + 4);
    const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    float bb[8];
    if constexpr (NORM == kNormLayer) {
        const float4 b0 = *reinterpret_cast<const float4 *>(b);
        const float4 b1 = *reinterpret_cast<const float4 *>(b + 4);
        bb[0] = b0.x; bb[1] = b0.y; bb[2] = b0.z; bb[3] = b0.w;
        bb[4] = b1.x; bb[5] = b1.y; bb[6] = b1.z; bb[7] = b1.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = to_float2<BF16>(w[i]);
        float a0, a1;
        if constexpr (NORM == kNormLayer) {
            a0 = fmaf(fmaf(f.x, sc, of), gg[2 * i], bb[2 * i]);
            a1 = fmaf(fmaf(f.y, sc, of), gg[2 * i + 1], bb[2 * i + 1]);
        } else {
            a0 = (f.x * sc) * gg[2 * i];
            a1 = (f.y * sc) * gg[2 * i + 1];
        }
        w[i] = from_float2<BF16>(a0, a1);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int BN>
struct TmemCols {
    static constexpr uint32_t need = 2 * BN;
    static constexpr uint32_t value =
        need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
};

template <int BN, int STAGES>
struct GemmSmem {
    static constexpr int kA = kBM * kBK * 2;        // 16 KB
    static constexpr int kB = BN * kBK * 2;         // BN x 128 B
    static constexpr int kGB = 2 * kBK * 4;         // FP32 gamma[64] then beta[64]
    static constexpr int off_a = 0;
    static constexpr int off_b = off_a + STAGES * kA;
    static constexpr int off_g = off_b + STAGES * kB;
    static constexpr int off_bar = off_g + STAGES * kGB;
    static constexpr int n_bars = 3 * STAGES + 5;
    static constexpr int off_tmem = off_bar + n_bars * 8;
    static constexpr int bytes = off_tmem + 16;
    static constexpr int alloc = bytes + 1024;              // slack to align the base to 1 KB
};

template <int NORM, bool SILU, bool BF16, int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ GemmArgs args)
{
    using L = GemmSmem<BN, STAGES>;
    constexpr bool kNorm = NORM != kNormNone;
    constexpr uint32_t kTx = L::kA + L::kB + (kNorm ? L::kGB : 0);
    constexpr uint32_t kTmemCols = TmemCols<BN>::value;
    constexpr uint32_t kIdesc = idesc_f16(BF16, kBM, BN);
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M = 128");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sA = smem + L::off_a;
    uint8_t *sB = smem + L::off_b;
    float *sG = reinterpret_cast<float *>(smem + L::off_g);    // FP32 gamma, beta per stage
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::off_bar);
    uint64_t *full = bars;                 // TMA landed          (1 arrival + tx)
    uint64_t *empty = bars + STAGES;       // MMA done with stage (1 commit)
    uint64_t *ready = bars + 2 * STAGES;   // transform done      (128 arrivals)
    uint64_t *acc_full = bars + 3 * STAGES;      // [2] accumulator ready (1 commit)
    uint64_t *acc_empty = bars + 3 * STAGES + 2; // [2] accumulator drained (128 arrivals)
    uint64_t *drain = bars + 3 * STAGES + 4;     // final MMA drain (1 commit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::off_tmem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int abort_flag;
    const WaitCtx wc{&abort_flag, args.err, args.timeout_ns};

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // The first kernel of a call clears the call's error word.
        if (args.zero_err && blockIdx.x == 0) *args.err = 0;
        prefetch_tmap(&args.map_a);
        prefetch_tmap(&args.map_b);
        if constexpr (kNorm) prefetch_tmap(&args.map_gb);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&ready[s], 128);
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

    // Let a dependent grid (the next layer) start its prologue early; it
    // still waits for this grid to finish before touching its outputs.
    pdl_launch_dependents();

    const int m_tiles = args.m_tiles;
    const int k_blocks = args.k_blocks;
    const int num_tiles = args.num_tiles;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // x may be the output of the previous grid (the FFN's H).
            pdl_wait();
            const uint64_t pol_x = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int m0 = (tile % m_tiles) * kBM;
                const int n0 = (tile / m_tiles) * BN;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[stage], kTx);
                    const int kc = kb * kBK;
                    tma_load_2d(sA + stage * L::kA, &args.map_a, &full[stage], kc, m0, pol_x);
                    tma_load_2d(sB + stage * L::kB, &args.map_b, &full[stage], kc, n0, pol_w);
                    if constexpr (kNorm)
                        tma_load_2d(sG + stage * 2 * kBK, &args.map_gb, &full[stage], kc, 0, pol_x);
                    ++fills;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // Never leave while a copy into this CTA's shared memory is in
            // flight: wait (bounded) for the last fills of every stage.
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
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
                    if constexpr (kNorm) {
                        if (!mbar_wait(&ready[stage], phase, wc)) { ok = false; break; }
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * L::kA);
                    const uint32_t b_addr = smem_u32(sB + stage * L::kB);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        umma_f16_ss(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32),
                                    sdesc_kmajor_sw128(b_addr + k * 32), kIdesc,
                                    (kb | k) != 0 ? 1u : 0u);
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // All MMAs issued by this thread complete before TMEM is freed.
            umma_commit(drain);
            mbar_wait(drain, 0, wc);
        }
    } else if (warp >= 4 && warp < 8) {
        if constexpr (kNorm) {
            // ---------------------------------------------------- transform
            const int t = threadIdx.x - 128;  // row of the tile this thread owns
            pdl_wait();                       // statistics come from the previous grid
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
                const int row = (tile % m_tiles) * kBM + t;
                float2 st = make_float2(0.f, 0.f);
                if (row < args.M) st = args.stats[row];
                const float sc = st.y;
                const float of = -st.x * st.y;
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!mbar_wait_warp(&full[stage], phase, wc)) { ok = false; break; }
                    const float *g = sG + stage * 2 * kBK;
                    const float *b = g + kBK;
                    uint8_t *arow = sA + stage * L::kA + t * 128;
                    const int sw = t & 7;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        // Logical 16-byte chunk c of this row sits at chunk
                        // c ^ (row % 8) under the 128-byte swizzle; visiting
                        // chunks in logical order keeps the 8 rows of a
                        // quarter-warp on 8 distinct bank groups.
                        uint4 *p = reinterpret_cast<uint4 *>(arow + ((c ^ sw) << 4));
                        *p = transform8<NORM, BF16>(*p, sc, of, g + 8 * c, b + 8 * c);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&ready[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp >= 8) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        int acc = 0;
        uint32_t acc_phase = 0;
        const int M = args.M, N = args.N;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            if (!mbar_wait_warp(&acc_full[acc], acc_phase, wc)) break;
            tc_fence_after();
            const int row = (tile % m_tiles) * kBM + q * 32 + lane;
            const int nt0 = (tile / m_tiles) * BN;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                const int n0 = nt0 + c;
                if (n0 >= N) break;  // uniform across the warp
                uint32_t r[32];
                tmem_ld32(t_base + static_cast<uint32_t>(c), r);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                if (args.bias != nullptr) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (n0 + 8 * j < N) {
                            const uint4 bv = __ldg(reinterpret_cast<const uint4 *>(
                                static_cast<const uint16_t *>(args.bias) + n0 + 8 * j));
                            const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 f = to_float2<BF16>(bw[i]);
                                v[8 * j + 2 * i] += f.x;
                                v[8 * j + 2 * i + 1] += f.y;
                            }
                        }
                    }
                }
                if constexpr (SILU) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]);
                }
                if (row < M) {
                    uint16_t *yrow = static_cast<uint16_t *>(args.y) + static_cast<int64_t>(row) * N;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (n0 + 8 * j < N) {
                            uint4 o;
                            o.x = from_float2<BF16>(v[8 * j + 0], v[8 * j + 1]);
                            o.y = from_float2<BF16>(v[8 * j + 2], v[8 * j + 3]);
                            o.z = from_float2<BF16>(v[8 * j + 4], v[8 * j + 5]);
                            o.w = from_float2<BF16>(v[8 * j + 6], v[8 * j + 7]);
                            *reinterpret_cast<uint4 *>(yrow + n0 + 8 * j) = o;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int NORM, bool SILU, bool BF16, int BN, int STAGES>
int launch_gemm_variant(const GemmArgs &args, int grid, bool pdl, cudaStream_t stream)
{
    auto kern = gemm_kernel<NORM, SILU, BF16, BN, STAGES>;
    constexpr int smem = GemmSmem<BN, STAGES>::alloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess)
        return record_cuda_error("cudaFuncSetAttribute(max dynamic smem)", e, cudaGetErrorString(e));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kGemmThreads);
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

// Dispatch one BN over the (norm, activation, dtype) combinations the
// library uses.
template <int BN, int STAGES>
int launch_gemm_bn(int norm, bool silu, bool bf16, const GemmArgs &args, int grid,
                   bool pdl, cudaStream_t stream)
{
#define NGR_CASE(N_, S_, B_)                                                      \
    if (norm == N_ && silu == S_ && bf16 == B_)                                   \
        return launch_gemm_variant<N_, S_, B_, BN, STAGES>(args, grid, pdl, stream);
    NGR_CASE(kNormLayer, false, false)
    NGR_CASE(kNormLayer, false, true)
    NGR_CASE(kNormRms, false, false)
    NGR_CASE(kNormRms, false, true)
    NGR_CASE(kNormNone, true, false)
    NGR_CASE(kNormNone, true, true)
    NGR_CASE(kNormNone, false, false)
    NGR_CASE(kNormNone, false, true)
#undef NGR_CASE
    return -9;
}

}  // namespace ngr
