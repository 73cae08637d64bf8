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
// CTAs resident at one time share weight tiles through L2), or, with fewer
// tiles than SMs, over (tile, K range) units whose FP32 partials the last
// unit of each chunk sums in range order.  Warp roles:
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
//   warps 4-11  transform: normalize + affine the x tile IN PLACE in shared
//               memory (each thread one 16-byte chunk column of 4 rows;
//               packed FP32x2 math, one rounding to the 16-bit operand
//               type), then fence the generic-proxy writes for the tensor
//               core and signal the MMA warp;
//   warps 12-15 epilogue: tcgen05.ld of its 32 accumulator rows, + bias,
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

// GELU, exact form: z Phi(z) = z (1 + erf(z / sqrt 2)) / 2.
__device__ __forceinline__ float gelu_f(float z)
{
    return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

// The epilogue activation of 32 values (`act` is uniform across the warp).
__device__ __forceinline__ void apply_act32(int act, float (&v)[32])
{
    if (act == kActSilu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]);
    } else if (act == kActRelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.0f);
    } else if (act == kActGelu) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_f(v[j]);
    }
}

// A 32-byte store (one full L2 sector) of 8 words.
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&w)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Round 32 values of one output row to the 16-bit type and store the
// columns [n0, n0 + 32) that lie inside [0, N) (N % 8 == 0); rows at or past
// M are skipped.  Each lane writes its own row, so whole 32-byte sectors
// are stored where y and its row pitch allow it (half-sector writes from
// every SM at once are what makes a tile's output slow to drain), else
// 16-byte pieces.
template <bool BF16>
__device__ __forceinline__ void store_row32(const float (&v)[32], int row, int n0, void *y, int M,
                                            int N, int n_lim = -1)
{
    if (row >= M) return;
    if (n_lim < 0) n_lim = N;     // columns stored: [n0, min(n0 + 32, n_lim)); row pitch N
    uint16_t *yrow = static_cast<uint16_t *>(y) + static_cast<int64_t>(row) * N;
    uint32_t o[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] = from_float2<BF16>(v[2 * j], v[2 * j + 1]);
    const bool sectors = ((reinterpret_cast<uintptr_t>(y) | static_cast<uintptr_t>(N) * 2u) & 31u) == 0;
    if (sectors && n0 + 32 <= n_lim) {
        st_global_v8(yrow + n0, *reinterpret_cast<const uint32_t(*)[8]>(&o[0]));
        st_global_v8(yrow + n0 + 16, *reinterpret_cast<const uint32_t(*)[8]>(&o[8]));
        return;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (n0 + 8 * j < n_lim)
            *reinterpret_cast<uint4 *>(yrow + n0 + 8 * j) =
                make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
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

// Two consecutive 16-bit values as FP32 (exact).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w)
{
    if constexpr (BF16)
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    else
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// Normalize + affine 8 elements with packed FP32x2 arithmetic:
// LayerNorm a = (x * rstd + (-mu * rstd)) * gamma + beta, RMSNorm
// a = (x * rstd) * gamma; one rounding to the 16-bit type at the end.
// so = (rstd, -mu * rstd) of the row; g[4], b[4] = gamma/beta pairs of the
// 8 columns.  (RMSNorm with the row scale in the epilogue: transform8_rms16.)
template <int NORM, bool BF16>
__device__ __forceinline__ uint4 transform8_pk(uint4 v, float2 so, const float2 (&g)[4],
                                               const float2 (&b)[4])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
    const float2 sc = make_float2(so.x, so.x);
    const float2 of = make_float2(so.y, so.y);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = unpack2<BF16>(w[i]);
        float2 a;
        if constexpr (NORM == kNormLayer)
            a = __ffma2_rn(__ffma2_rn(f, sc, of), g[i], b[i]);
        else
            a = __fmul2_rn(__fmul2_rn(f, sc), g[i]);
        o[i] = from_float2<BF16>(a.x, a.y);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// RMSNorm with the row's scale left to the epilogue: the transform computes
// a' = x s gamma, s = 2^e a power of two close to the row's rstd, in packed
// 16-bit arithmetic, and the epilogue multiplies the accumulator by
// rstd / s.  The product of two 16-bit values is exact in FP32, so
// round16(x s gamma) is the single rounding the FP32 form would make, and
// it is made here by one packed multiply per two elements, with no
// conversions.  Multiplying by s is exact (it moves the exponent) and keeps
// a' at the scale of the normalized row, so fp16 does not overflow where
// x rstd gamma would not; bf16's range needs no scale (s = 1).
__device__ __forceinline__ int rms_scale_exp(float rstd)
{
    const int e = ((__float_as_int(rstd) >> 23) & 0xff) - 127;   // floor(log2 rstd)
    return min(max(e, -14), 15);                                  // a normal fp16 power of two
}

// s, twice, as a packed 16-bit pair.
template <bool BF16>
__device__ __forceinline__ uint32_t rms_in_scale2(float rstd)
{
    if constexpr (BF16) {
        return 0x3f803f80u;                                       // (1.0, 1.0)
    } else {
        const uint32_t h = static_cast<uint32_t>(rms_scale_exp(rstd) + 15) << 10;
        return h | (h << 16);
    }
}

// rstd / s, exact in FP32.
template <bool BF16>
__device__ __forceinline__ float rms_out_scale(float rstd)
{
    if constexpr (BF16)
        return rstd;
    else
        return rstd * __int_as_float((127 - rms_scale_exp(rstd)) << 23);
}

// a * b on two packed 16-bit values, rounded to nearest even, subnormals kept.
template <bool BF16>
__device__ __forceinline__ uint32_t mul2_16(uint32_t a, uint32_t b)
{
    uint32_t d;
    if constexpr (BF16)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// a' = x s gamma for 8 elements (RMSNorm, row scale in the epilogue):
// s2 = (s, s), g2[4] = the gamma pairs of the 8 columns, all packed 16-bit.
template <bool BF16>
__device__ __forceinline__ uint4 transform8_rms16(uint4 v, uint32_t s2, const uint32_t (&g2)[4])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = mul2_16<BF16>(BF16 ? w[i] : mul2_16<BF16>(w[i], s2), g2[i]);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// The epilogue of 32 accumulator columns [n0, n0 + 32) of one row: + bias,
// or with a folded norm y = rstd acc + (-mu rstd) c[n] + b'[n] (so =
// (rstd, -mu rstd) of the row), then the activation, + residual, rounding,
// 16-byte stores.  With ROW_SCALE_OUT the accumulator is first multiplied
// by so.x (the row's rstd, left out of an RMSNorm transform).
template <int NORM, bool BF16, bool ROW_SCALE_OUT = false>
__device__ __forceinline__ void epilogue_store32(float (&v)[32], int row, int n0,
                                                 const GemmArgs &args, float2 so, int n_lim = -1)
{
    // Columns at or past n_lim (default N) are neither read nor stored.
    const int M = args.M, N = n_lim < 0 ? args.N : n_lim;
    if constexpr (ROW_SCALE_OUT) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= so.x;
    }
    if constexpr (is_fold(NORM)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (n0 + 8 * j < N) {
                const float4 b0 = __ldg(reinterpret_cast<const float4 *>(args.fold_b + n0 + 8 * j));
                const float4 b1 = __ldg(reinterpret_cast<const float4 *>(args.fold_b + n0 + 8 * j + 4));
                float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
                if constexpr (NORM == kNormFoldLayer) {
                    const float4 c0 = __ldg(reinterpret_cast<const float4 *>(args.fold_c + n0 + 8 * j));
                    const float4 c1 = __ldg(reinterpret_cast<const float4 *>(args.fold_c + n0 + 8 * j + 4));
                    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) bb[i] = fmaf(so.y, cc[i], bb[i]);
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) v[8 * j + i] = fmaf(v[8 * j + i], so.x, bb[i]);
            }
        }
    } else if (args.bias != nullptr) {
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
    apply_act32(args.act, v);
    if (args.residual != nullptr && row < M) {
        const uint16_t *rrow = static_cast<const uint16_t *>(args.residual) + static_cast<int64_t>(row) * args.N;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (n0 + 8 * j < N) {
                const uint4 rv = __ldg(reinterpret_cast<const uint4 *>(rrow + n0 + 8 * j));
                const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = to_float2<BF16>(rw[i]);
                    v[8 * j + 2 * i] += f.x;
                    v[8 * j + 2 * i + 1] += f.y;
                }
            }
        }
    }
    store_row32<BF16>(v, row, n0, args.y, M, args.N, N);
}

// (rstd, -mu rstd) of `row` for the folded epilogue.
template <int NORM>
__device__ __forceinline__ float2 fold_row_scale(const GemmArgs &args, int row)
{
    if constexpr (is_fold(NORM)) {
        float2 st = make_float2(0.f, 0.f);
        if (row < args.M) st = args.stats[row];
        return make_float2(st.y, NORM == kNormFoldLayer ? -st.x * st.y : 0.f);
    } else {
        return make_float2(1.f, 0.f);
    }
}

// The transform role, shared by the tile kernels.  Transform thread t
// (0 <= t < kTransformThreads) belongs to group t / kGroupThreads; group g
// normalizes the stages of the k blocks with running index % groups == g.
// A stage is normalized in PARTS column parts of 64 / PARTS columns each,
// and after each part one lane per warp calls arrive(stage * PARTS + part),
// so that the tensor core can start on the first columns of a stage while
// the rest are still being normalized.  Within a part, thread u owns 16-byte
// chunk u % CP (CP = 8 / PARTS chunks, 8 columns each) of the part, for the
// rows r0 + 16 PARTS i, where the PARTS threads of a quarter-warp that share
// a chunk take rows whose index differs by 8 / PARTS: the quarter-warp then
// covers 8 distinct 16-byte positions of the 128-byte swizzle pattern
// (conflict free), and gamma/beta of the chunk are read once per part.
// After its stores each thread fences them for the async proxy.
// m0_of(unit) gives the unit's first x row in this CTA and kb_range(unit)
// the k blocks [x, y) it covers (all of them unless K is split).
// gamma/beta come from each stage's FP32 box in shared memory (sG), or,
// with GB_GLOBAL, from the FP32 rows g_glob / b_glob in global memory: a
// thread then issues the loads of its chunks before waiting for the stage
// (they do not depend on it) and treats columns at or past K as zero.
template <int NORM, bool BF16, int STAGES, int KA, int PARTS = 1, bool ROW_SCALE = true,
          bool GB_GLOBAL = false, typename M0Fn, typename KbFn, typename ArriveFn>
__device__ __forceinline__ void transform_role(int t, int tile0, int tile_step, int num_tiles,
                                               KbFn kb_range, int M, const float2 *stats,
                                               uint8_t *sA, const float *sG, uint64_t *full,
                                               const WaitCtx &wc, M0Fn m0_of, ArriveFn arrive,
                                               const float *g_glob = nullptr,
                                               const float *b_glob = nullptr, int K = 0)
{
    static_assert(PARTS == 1 || PARTS == 2 || PARTS == 4, "a part is a whole number of 16-byte chunks");
    static_assert(kGroupThreads == 128 || kGroupThreads == 256, "a group is 4 or 8 warps");
    constexpr int kCP = 8 / PARTS;                    // chunks of a row per part
    constexpr int kRowStride = 16 * PARTS * (kGroupThreads / 128);  // rows between a thread's rows
    constexpr int kRows = kBM / kRowStride;           // rows per thread
    constexpr int kBatch = kRows < 8 ? kRows : 8;
    constexpr int kS = 8 / PARTS;                     // row offset of a quarter-warp's row sets
    // A group waits on a stage barrier kTransformGroups fills after its
    // previous one; with more groups than stages it could be two phases
    // ahead, which a parity wait cannot tell from a completed phase.
    static_assert(kTransformGroups <= STAGES, "more transform groups than pipeline stages");
    const int g = t / kGroupThreads;
    const int u = t % kGroupThreads;
    const int cl = u % kCP;                           // chunk within the part
    const int j = (u / kCP) % PARTS;                  // row set within the quarter-warp
    const int qw = u >> 3;                            // quarter-warp of the group
    const int r0 = (qw % kS) + 8 * (qw / kS) + kS * j;
    const int lane = threadIdx.x & 31;
    // Without a norm (the multicast kernel's plain product) the role only
    // relays each landed stage to the MMA issuer.
    constexpr bool kMath = NORM == kNormLayer || NORM == kNormRms;
    pdl_wait();                          // statistics come from the previous grid
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;                          // running k-block index over this CTA's tiles
    for (int tile = tile0; tile < num_tiles; tile += tile_step) {
        const int m0 = m0_of(tile);
        float2 so[kRows];
        uint32_t s2[kRows];                  // RMSNorm, row scale in the epilogue: (s, s)
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int row = m0 + r0 + kRowStride * i;
            float2 st = make_float2(0.f, 0.f);
            if (kMath && row < M) st = stats[row];
            so[i] = make_float2(st.y, -st.x * st.y);
            s2[i] = rms_in_scale2<BF16>(st.y);
        }
        const int2 kr = kb_range(tile);
        for (int kb = kr.x; kb < kr.y; ++kb, ++it) {
            if (it % kTransformGroups == g) {
                if constexpr (!kMath) {
                    // No norm: only relay each landed stage to the MMA issuer.
                    if (!mbar_wait_warp_ahead(&full[stage], phase, wc)) return;
                    __syncwarp();
#pragma unroll
                    for (int part = 0; part < PARTS; ++part)
                        if (lane == 0) arrive(stage * PARTS + part);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    continue;
                }
                float4 qg[GB_GLOBAL ? PARTS : 1][4];
                if constexpr (GB_GLOBAL) {
#pragma unroll
                    for (int part = 0; part < PARTS; ++part) {
                        const int col = kb * kBK + 8 * (cl + kCP * part);
                        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                        const bool in = col < K;
                        qg[part][0] = in ? __ldg(reinterpret_cast<const float4 *>(g_glob + col)) : z;
                        qg[part][1] = in ? __ldg(reinterpret_cast<const float4 *>(g_glob + col + 4)) : z;
                        if constexpr (NORM == kNormLayer) {
                            qg[part][2] = in ? __ldg(reinterpret_cast<const float4 *>(b_glob + col)) : z;
                            qg[part][3] = in ? __ldg(reinterpret_cast<const float4 *>(b_glob + col + 4)) : z;
                        }
                    }
                }
                if (!mbar_wait_warp_ahead(&full[stage], phase, wc)) return;
#pragma unroll
                for (int part = 0; part < PARTS; ++part) {
                    const int c = cl + kCP * part;    // logical chunk: columns 8c .. 8c+7
                    float4 q[4];
                    if constexpr (GB_GLOBAL) {
                        q[0] = qg[part][0];
                        q[1] = qg[part][1];
                        if constexpr (NORM == kNormLayer) {
                            q[2] = qg[part][2];
                            q[3] = qg[part][3];
                        }
                    } else {
                        // gamma/beta of the chunk; the two halves are read in
                        // separate instructions so that a quarter-warp touches
                        // 8 distinct 16-byte slots of one 128-byte line each time.
                        const float *gp = sG + stage * 2 * kBK + 8 * c;
                        q[0] = *reinterpret_cast<const float4 *>(gp);
                        q[1] = *reinterpret_cast<const float4 *>(gp + 4);
                        if constexpr (NORM == kNormLayer) {
                            q[2] = *reinterpret_cast<const float4 *>(gp + kBK);
                            q[3] = *reinterpret_cast<const float4 *>(gp + kBK + 4);
                        }
                    }
                    const float2 gg[4] = {make_float2(q[0].x, q[0].y), make_float2(q[0].z, q[0].w),
                                          make_float2(q[1].x, q[1].y), make_float2(q[1].z, q[1].w)};
                    float2 bb[4];
                    if constexpr (NORM == kNormLayer) {
                        bb[0] = make_float2(q[2].x, q[2].y);
                        bb[1] = make_float2(q[2].z, q[2].w);
                        bb[2] = make_float2(q[3].x, q[3].y);
                        bb[3] = make_float2(q[3].z, q[3].w);
                    }
                    // gamma pairs as packed 16-bit values (exact: gamma is a 16-bit input)
                    uint32_t g2[4];
                    if constexpr (!ROW_SCALE)
#pragma unroll
                        for (int q2 = 0; q2 < 4; ++q2) g2[q2] = from_float2<BF16>(gg[q2].x, gg[q2].y);
                    const int pc = (c ^ (r0 & 7)) << 4;   // swizzled chunk offset (same for all rows)
                    uint8_t *base = sA + stage * KA + r0 * 128 + pc;
                    // Rows in batches of up to 8: all loads of a batch are in
                    // flight before its first store.
#pragma unroll
                    for (int b0 = 0; b0 < kRows; b0 += kBatch) {
                        uint4 v[kBatch];
#pragma unroll
                        for (int i = 0; i < kBatch; ++i)
                            v[i] = *reinterpret_cast<const uint4 *>(base + (b0 + i) * kRowStride * 128);
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            uint4 o;
                            if constexpr (ROW_SCALE)
                                o = transform8_pk<NORM, BF16>(v[i], so[b0 + i], gg, bb);
                            else
                                o = transform8_rms16<BF16>(v[i], s2[b0 + i], g2);
                            *reinterpret_cast<uint4 *>(base + (b0 + i) * kRowStride * 128) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) arrive(stage * PARTS + part);
                }
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
    }
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

template <int NORM, bool BF16, int BN, int STAGES>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_kernel(const __grid_constant__ GemmArgs args)
{
    using L = GemmSmem<BN, STAGES>;
    constexpr bool kNorm = NORM == kNormLayer || NORM == kNormRms;  // transform stage
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
            mbar_init(&ready[s], kGroupWarps);
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
    // Work units: (tile, K range) pairs; without a split a unit is a tile.
    // (With fewer tiles than SMs -- up to 128 rows against a narrow W -- a
    // K split streams W on more SMs.)
    const int n_splits = max(1, args.k_splits);
    const int num_units = num_tiles * n_splits;
    const int kb_per_split = n_splits > 1 ? args.kb_per_split : k_blocks;
    auto unit_tile = [&](int u) { return u / n_splits; };
    auto unit_kb0 = [&](int u) { return (u % n_splits) * kb_per_split; };
    auto unit_kb1 = [&](int u) { return min(k_blocks, unit_kb0(u) + kb_per_split); };

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
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                const int tile = unit_tile(u);
                const int m0 = (tile % m_tiles) * kBM;
                const int n0 = (tile / m_tiles) * BN;
                for (int kb = unit_kb0(u), kb_end = unit_kb1(u); kb < kb_end; ++kb) {
                    if (!mbar_wait_ahead(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
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
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                if (!mbar_wait_spin(&acc_empty[acc], acc_phase ^ 1u, wc)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                const int kb0 = unit_kb0(u);
                for (int kb = kb0, kb_end = unit_kb1(u); kb < kb_end; ++kb) {
                    if (!mbar_wait_spin(&full[stage], phase, wc)) { ok = false; break; }
                    if constexpr (kNorm) {
                        if (!mbar_wait_spin(&ready[stage], phase, wc)) { ok = false; break; }
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * L::kA);
                    const uint32_t b_addr = smem_u32(sB + stage * L::kB);
#pragma unroll
                    for (int k = 0; k < kBK / kUmmaK; ++k) {
                        umma_f16_ss(d_tmem, sdesc_kmajor_sw128(a_addr + k * 32),
                                    sdesc_kmajor_sw128(b_addr + k * 32), kIdesc,
                                    (kb != kb0 || k != 0) ? 1u : 0u);
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
            mbar_wait_long(drain, 0, wc);
        }
    } else if (warp >= kTransformWarp0 && warp < kEpilogueWarp0) {
        if constexpr (kNorm) {
            // ---------------------------------------------------- transform
            transform_role<NORM, BF16, STAGES, L::kA>(
                threadIdx.x - kTransformWarp0 * 32, blockIdx.x, gridDim.x, num_units,
                [&](int u) { return make_int2(unit_kb0(u), unit_kb1(u)); }, args.M, args.stats, sA, sG, full, wc,
                [&](int u) { return (unit_tile(u) % m_tiles) * kBM; },
                [&](int st) { mbar_arrive(&ready[st]); });
        }
    } else if (warp >= kEpilogueWarp0) {
        // --------------------------------------------------------- epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        int acc = 0;
        uint32_t acc_phase = 0;
        const int N = args.N;
        if constexpr (is_fold(NORM)) pdl_wait();  // row statistics from the previous grid
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const int tile = unit_tile(u);
            if (!mbar_wait_warp_long(&acc_full[acc], acc_phase, wc)) break;
            tc_fence_after();
            const int row = (tile % m_tiles) * kBM + q * 32 + lane;
            const float2 so = fold_row_scale<NORM>(args, row);
            const int nt0 = (tile / m_tiles) * BN;
            const uint32_t t_base = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                    static_cast<uint32_t>(acc * BN);
            const int nch = (min(BN, N - nt0) + 31) / 32;   // 32-column chunks inside N
            if (n_splits > 1) {
                // K split: (1) this unit's FP32 partials of the warp's
                // 32 x 32 chunks (column-major within a chunk, so that each
                // store of the warp writes one 128-byte line); (2) one fence,
                // then one counter per chunk (lane i takes chunk i); (3) the
                // chunks this unit arrived last at are summed over the K
                // ranges in range order and finished, and their counters
                // reset for the next call.
                const int split = u % n_splits;
                const size_t blk0 = (static_cast<size_t>(tile) * 4 + q) * (BN / 32);
                const size_t part_stride = static_cast<size_t>(n_splits) * 1024;
#pragma unroll 1
                for (int i = 0; i < nch; ++i) {
                    uint32_t r[32];
                    tmem_ld32(t_base + static_cast<uint32_t>(32 * i), r);
                    tmem_ld_wait();
                    float *mine = args.partials + (blk0 + i) * part_stride + split * 1024 + lane;
#pragma unroll
                    for (int j = 0; j < 32; ++j) __stcg(mine + j * 32, __uint_as_float(r[j]));
                }
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane < nch) last = atomicAdd(&args.split_counters[blk0 + lane], 1) == n_splits - 1;
                const unsigned last_mask = __ballot_sync(0xffffffffu, last);
                if (last_mask != 0u) {
                    __threadfence();
#pragma unroll 1
                    for (int i = 0; i < nch; ++i) {
                        if (((last_mask >> i) & 1u) == 0u) continue;
                        uint32_t r[32];
                        tmem_ld32(t_base + static_cast<uint32_t>(32 * i), r);
                        tmem_ld_wait();
                        const float *part = args.partials + (blk0 + i) * part_stride + lane;
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
                        epilogue_store32<NORM, BF16>(v, row, nt0 + 32 * i, args, so);
                    }
                    __syncwarp();
                    if (lane < nch && ((last_mask >> lane) & 1u)) args.split_counters[blk0 + lane] = 0;
                }
            } else {
#pragma unroll 1
                for (int i = 0; i < nch; ++i) {
                    uint32_t r[32];
                    tmem_ld32(t_base + static_cast<uint32_t>(32 * i), r);
                    tmem_ld_wait();
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    epilogue_store32<NORM, BF16>(v, row, nt0 + 32 * i, args, so);
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

template <int NORM, bool BF16, int BN, int STAGES>
int launch_gemm_variant(const GemmArgs &args, int grid, bool pdl, cudaStream_t stream)
{
    auto kern = gemm_kernel<NORM, BF16, BN, STAGES>;
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

// Dispatch one BN over the (norm, dtype) combinations the library uses
// (the activation is a runtime argument).
template <int BN, int STAGES>
int launch_gemm_bn(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl,
                   cudaStream_t stream)
{
#define NGR_CASE(N_, B_)                                                          \
    if (norm == N_ && bf16 == B_)                                                 \
        return launch_gemm_variant<N_, B_, BN, STAGES>(args, grid, pdl, stream);
    NGR_CASE(kNormLayer, false)
    NGR_CASE(kNormLayer, true)
    NGR_CASE(kNormRms, false)
    NGR_CASE(kNormRms, true)
    NGR_CASE(kNormNone, false)
    NGR_CASE(kNormNone, true)
    NGR_CASE(kNormFoldLayer, false)
    NGR_CASE(kNormFoldLayer, true)
    NGR_CASE(kNormFoldRms, false)
    NGR_CASE(kNormFoldRms, true)
#undef NGR_CASE
    return -9;
}

}  // namespace ngr
