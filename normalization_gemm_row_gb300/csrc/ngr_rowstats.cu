// ngr_rowstats.cu -- step a1: per-row FP32 statistics of x [M, K].
//
// "LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现", §1.1: the
// statistics are a reduction over each row (a sum and a sum of squares);
// §2.3: they are computed in FP32.  One CTA reduces one row with 16-byte
// loads.  LayerNorm uses shifted sums so that a large row mean (inputs
// centred far from zero) does not cancel the variance:
//  - each thread forms (n, mean, M2) of its own elements from sums of
//    (x - s), s its first element;
//  - a warp re-centres its threads' triples on lane 0's mean m0
//    (sum n (mean - m0) and sum M2 + n (mean - m0)^2 add exactly like plain
//    sums), which costs no more than a factor 32 in cancellation because m0
//    is the mean of 32 of the warp's own elements;
//  - the 8 warps are merged with the parallel-variance update of Chan,
//    Golub and LeVeque (1979):
//      n = na + nb,  d = mb - ma,  mean = ma + d nb / n,
//      M2 = M2a + M2b + d^2 na nb / n.
// var = M2 / K (biased), rstd = 1 / sqrt(var + eps).  RMSNorm: rstd =
// 1 / sqrt(sum x^2 / K + eps) and mu = 0.
//
// On request the kernel also writes the normalized rows
// xhat = (x - mu) rstd gamma + beta (RMSNorm: x rstd gamma), with the FP32
// arithmetic and the single rounding of the tile kernel's transform: the
// norm that follows a product writes its output this way (the fused
// pre-norm paths never write normalized rows).
//
// When the rows are padded (K is the padded pitch, a multiple of 8), only the
// first k_valid columns count: the padding is excluded from the LayerNorm
// sums and every mean divides by k_valid.
//
// The same launch converts gamma and beta to FP32 once per call (the GEMM's
// producer streams them with the tiles) and zeroes the split-K counters of
// the kernel that follows (the decode kernel's, or a tile kernel's when its
// plan splits K) when asked to, so that they start from zero every call; as
// the first kernel of a call it also clears the call's error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "ngr_internal.h"
#include "ngr_ptx.cuh"

namespace ngr {

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if constexpr (BF16) {
            __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
            float2 p = __bfloat1622float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        } else {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 p = __half22float2(h);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
        }
    }
}

// Normalize 8 elements: a = (x rstd + (-mu rstd)) gamma + beta in FP32
// (RMSNorm: (x rstd) gamma), one rounding to the 16-bit type.
template <bool BF16>
__device__ __forceinline__ float2 unpack_pair(uint32_t w)
{
    if constexpr (BF16)
        return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
    else
        return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

template <int NORM, bool BF16>
__device__ __forceinline__ uint4 normalize8(const uint4 &v, const uint4 &g, const uint4 &b,
                                            float sc, float of)
{
    const uint32_t wx[4] = {v.x, v.y, v.z, v.w};
    const uint32_t wg[4] = {g.x, g.y, g.z, g.w};
    const uint32_t wb[4] = {b.x, b.y, b.z, b.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 fx = unpack_pair<BF16>(wx[i]);
        const float2 fg = unpack_pair<BF16>(wg[i]);
        float a0, a1;
        if constexpr (NORM == kNormLayer) {
            const float2 fb = unpack_pair<BF16>(wb[i]);
            a0 = fmaf(fmaf(fx.x, sc, of), fg.x, fb.x);
            a1 = fmaf(fmaf(fx.y, sc, of), fg.y, fb.y);
        } else {
            a0 = (fx.x * sc) * fg.x;
            a1 = (fx.y * sc) * fg.y;
        }
        if constexpr (BF16) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
            o[i] = *reinterpret_cast<const uint32_t *>(&h);
        } else {
            const __half2 h = __floats2half2_rn(a0, a1);
            o[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// A 16-bit value's bits as FP32.
template <bool BF16>
__device__ __forceinline__ float half_bits_to_float(uint32_t h)
{
    if constexpr (BF16)
        return __uint_as_float(h << 16);
    else
        return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

// Merge (nb, mb, m2b) into (n, mean, m2): the parallel-variance update.
__device__ __forceinline__ void chan_merge(float &n, float &mean, float &m2, float nb, float mb,
                                           float m2b)
{
    const float nt = n + nb;
    if (nt > 0.f) {
        const float d = mb - mean;
        const float wb = __fdividef(nb, nt);   // 0 <= nb <= nt: well inside its range
        mean = fmaf(d, wb, mean);
        m2 = m2 + m2b + d * d * (n * wb);
        n = nt;
    }
}

constexpr int kStatsThreads = 256;

// One CTA per row (grid-stride over rows): every thread issues all of its
// 16-byte loads of the row at once, so a row costs one memory round trip.
// At most 32 registers, so that 8 CTAs (2048 threads) fit on an SM and the
// rows of a batch of up to 8 x SMs run in a single wave.  The variant that
// also writes the normalized rows (the norm after a product) holds a row of
// up to 8192 elements in registers between its two passes and runs at most
// 64 registers, 4 CTAs per SM.
constexpr int kStatsCtasPerSm = 8;
constexpr int kXhatCtasPerSm = 4;

template <int NORM, bool BF16, bool XHAT>
__global__ void __launch_bounds__(kStatsThreads, XHAT ? kXhatCtasPerSm : kStatsCtasPerSm) rowstats_kernel(
    const uint4 *__restrict__ x, int64_t M, int64_t K, float eps,
    float2 *__restrict__ stats, const void *__restrict__ gamma,
    const void *__restrict__ beta, float *__restrict__ gamma_f,
    float *__restrict__ beta_f, int *__restrict__ counters, int n_counters,
    int *__restrict__ err_to_clear, uint4 *__restrict__ xhat, int64_t k_valid)
{
    // The dependent GEMM may start its prologue while this grid runs; it
    // waits for this grid's completion before reading the statistics.
    pdl_launch_dependents();
    // Launched as a dependent of the product that wrote x (the norm after a
    // GEMM), wait for that grid; otherwise this returns at once.
    pdl_wait();

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int wid = tid >> 5;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    if (err_to_clear && gtid == 0) *err_to_clear = 0;
    if (counters) {
        for (int64_t i = gtid; i < n_counters; i += gstride) counters[i] = 0;
    }
    if (gamma_f) {
        for (int64_t k = gtid; k < K; k += gstride) {
            if constexpr (BF16) {
                gamma_f[k] = __bfloat162float(static_cast<const __nv_bfloat16 *>(gamma)[k]);
                if (beta_f)
                    beta_f[k] = beta ? __bfloat162float(static_cast<const __nv_bfloat16 *>(beta)[k]) : 0.f;
            } else {
                gamma_f[k] = __half2float(static_cast<const __half *>(gamma)[k]);
                if (beta_f)
                    beta_f[k] = beta ? __half2float(static_cast<const __half *>(beta)[k]) : 0.f;
            }
        }
    }

    __shared__ float red[3][kStatsThreads / 32];
    __shared__ float2 row_stats;
    const int64_t vec_per_row = K >> 3;  // 8 elements per 16-byte vector
    // With XHAT and rows of at most 4 vectors per thread (K <= 8192) the
    // statistics pass keeps the row in registers for the output pass.
    uint4 keep[4];
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const uint4 *xr = x + row * vec_per_row;
        if constexpr (NORM == kNormLayer) {
            // This thread's elements as shifted sums in packed FP32x2, shift
            // = its first element.  Slots past the row read as the shift
            // itself (they add exactly zero); a padded row's zero padding,
            // in its last vector only, is taken out afterwards by the thread
            // that read it.
            const int nvec = static_cast<int>(vec_per_row);
            const uint32_t h = tid < nvec ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short *>(xr + tid))) : 0u;
            const float s = half_bits_to_float<BF16>(h);
            const uint32_t hh = h | (h << 16);
            const float2 ns = make_float2(-s, -s);
            float2 s1p = make_float2(0.f, 0.f), s2p = make_float2(0.f, 0.f);
#pragma unroll 1
            for (int v0 = tid; v0 < nvec; v0 += 4 * kStatsThreads) {
                uint4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int v = v0 + u * kStatsThreads;
                    q[u] = v < nvec ? __ldg(xr + v) : make_uint4(hh, hh, hh, hh);
                }
                if constexpr (XHAT) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) keep[u] = q[u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 d = __fadd2_rn(unpack_pair<BF16>(w[i]), ns);
                        s1p = __fadd2_rn(s1p, d);
                        s2p = __ffma2_rn(d, d, s2p);
                    }
                }
            }
            float s1 = s1p.x + s1p.y, s2 = s2p.x + s2p.y;
            float n = tid < nvec ? 8.f * static_cast<float>((nvec - 1 - tid) / kStatsThreads + 1) : 0.f;
            const int pad = nvec * 8 - static_cast<int>(k_valid);
            if (pad > 0 && (nvec - 1) % kStatsThreads == tid) {
                // Each padding zero added (0 - s) to s1 and s^2 to s2.
                const float p = static_cast<float>(pad);
                n -= p;
                s1 = fmaf(p, s, s1);
                s2 = fmaf(-p * s, s, s2);
            }
            // (n, mean, M2) of this thread, then re-centred on lane 0's mean
            // (a mean of the warp's own elements) so that the warp's sums
            // need plain additions only.
            const float s1n = n > 0.f ? __fdividef(s1, n) : 0.f;
            const float mean_t = s + s1n;
            const float m2_t = fmaxf(s2 - s1 * s1n, 0.f);
            const float sw = __shfl_sync(0xffffffffu, mean_t, 0);
            const float dt = mean_t - sw;
            float a1 = n * dt;
            float a2 = fmaf(a1, dt, m2_t);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                n += __shfl_xor_sync(0xffffffffu, n, off);
                a1 += __shfl_xor_sync(0xffffffffu, a1, off);
                a2 += __shfl_xor_sync(0xffffffffu, a2, off);
            }
            const float a1n = n > 0.f ? __fdividef(a1, n) : 0.f;
            const float mean = sw + a1n;
            const float m2 = fmaxf(a2 - a1 * a1n, 0.f);
            if (lane == 0) {
                red[0][wid] = n;
                red[1][wid] = mean;
                red[2][wid] = m2;
            }
            __syncthreads();
            if (tid == 0) {
                float tn = red[0][0], tm = red[1][0], t2 = red[2][0];
                for (int w = 1; w < kStatsThreads / 32; ++w) chan_merge(tn, tm, t2, red[0][w], red[1][w], red[2][w]);
                const float var = t2 / static_cast<float>(k_valid);
                row_stats = make_float2(tm, 1.0f / sqrtf(var + eps));
                stats[row] = row_stats;
            }
            __syncthreads();
        } else {
            float ss = 0.f;
            for (int64_t v0 = tid; v0 < vec_per_row; v0 += 4 * kStatsThreads) {
                uint4 q[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = v0 + static_cast<int64_t>(u) * kStatsThreads;
                    if (v < vec_per_row) q[u] = __ldg(xr + v);
                }
                if constexpr (XHAT) {
#pragma unroll
                    for (int u = 0; u < 4; ++u) keep[u] = q[u];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = v0 + static_cast<int64_t>(u) * kStatsThreads;
                    if (v >= vec_per_row) break;
                    float f[8];
                    unpack8<BF16>(q[u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) red[0][wid] = ss;
            __syncthreads();
            if (tid == 0) {
                float t = 0.f;
                for (int w = 0; w < kStatsThreads / 32; ++w) t += red[0][w];
                row_stats = make_float2(0.f, 1.0f / sqrtf(t / static_cast<float>(k_valid) + eps));
                stats[row] = row_stats;
            }
            __syncthreads();
        }
        if constexpr (XHAT) {
            // The row is still in L1: normalize it and write it out.
            const float sc = row_stats.y;
            const float of = NORM == kNormLayer ? -row_stats.x * row_stats.y : 0.f;
            const uint4 *gv = static_cast<const uint4 *>(gamma);
            const uint4 *bv = static_cast<const uint4 *>(beta);
            uint4 *out = xhat + row * vec_per_row;
            if (vec_per_row <= 4 * kStatsThreads) {
                // The row is in registers (keep[u] = vector tid + u threads):
                // all gamma/beta loads in flight at once, then the stores.
                uint4 gq[4], bq[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = tid + static_cast<int64_t>(u) * kStatsThreads;
                    if (v < vec_per_row) {
                        gq[u] = __ldg(gv + v);
                        bq[u] = NORM == kNormLayer ? __ldg(bv + v) : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int64_t v = tid + static_cast<int64_t>(u) * kStatsThreads;
                    if (v < vec_per_row) out[v] = normalize8<NORM, BF16>(keep[u], gq[u], bq[u], sc, of);
                }
            } else {
#pragma unroll 1
                for (int64_t v = tid; v < vec_per_row; v += kStatsThreads)
                    out[v] = normalize8<NORM, BF16>(__ldg(xr + v), __ldg(gv + v),
                                                    NORM == kNormLayer ? __ldg(bv + v) : make_uint4(0, 0, 0, 0),
                                                    sc, of);
            }
            __syncthreads();   // row_stats is rewritten by the next row
        }
    }
}

int launch_rowstats(int norm, bool bf16, const void *x, int64_t M, int64_t K,
                    float eps, float2 *stats, const void *gamma,
                    const void *beta, float *gamma_f, float *beta_f,
                    int *counters, int n_counters, int *err_to_clear,
                    int num_sms, cudaStream_t stream, void *xhat, int64_t k_valid, bool pdl)
{
    if (k_valid < 0) k_valid = K;
    const int threads = kStatsThreads;
    int64_t blocks = M;
    const int64_t cap = static_cast<int64_t>(num_sms) * (xhat ? kXhatCtasPerSm : kStatsCtasPerSm);   // one wave
    if (blocks > cap) blocks = cap;
    const int64_t kblocks = (K + threads - 1) / threads;
    if (gamma_f && blocks < kblocks) blocks = kblocks < cap ? kblocks : cap;
    if (blocks < 1) blocks = 1;
    const uint4 *xv = static_cast<const uint4 *>(x);
    dim3 grid(static_cast<unsigned>(blocks)), block(threads);
    uint4 *xh = static_cast<uint4 *>(xhat);
    // As a programmatic dependent (pdl) the grid may be scheduled while the
    // previous one finishes; the kernel waits for it before reading x.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
#define NGR_STATS(N_, B_)                                                                     \
    if (xh)                                                                                   \
        cudaLaunchKernelEx(&cfg, rowstats_kernel<N_, B_, true>, xv, M, K, eps, stats, gamma,  \
                           beta, gamma_f, beta_f, counters, n_counters, err_to_clear, xh,     \
                           k_valid);                                                          \
    else                                                                                      \
        cudaLaunchKernelEx(&cfg, rowstats_kernel<N_, B_, false>, xv, M, K, eps, stats, gamma, \
                           beta, gamma_f, beta_f, counters, n_counters, err_to_clear,         \
                           static_cast<uint4 *>(nullptr), k_valid);
    if (norm == kNormLayer) {
        if (bf16) { NGR_STATS(kNormLayer, true) } else { NGR_STATS(kNormLayer, false) }
    } else {
        if (bf16) { NGR_STATS(kNormRms, true) } else { NGR_STATS(kNormRms, false) }
    }
#undef NGR_STATS
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : record_cuda_error("row statistics launch", e, cudaGetErrorString(e));
}

}  // namespace ngr
