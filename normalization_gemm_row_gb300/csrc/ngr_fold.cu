// ngr_fold.cu -- step a7's one-time preparation: the inference-mode weight
// fold of the pre-norm linear layer.
//
// "LayerNorm 融合算子如何让大模型推理再快 15%？深度拆解 ATB 的实现", §6.2: in
// inference gamma and beta are fixed, so gamma can be folded into the
// following matmul's weight beforehand.  Written out,
//   y[i,n] = rstd_i sum_k x[i,k] W'[n,k] - rstd_i mu_i c[n] + b'[n],
//   W'[n,k] = gamma_k W[n,k],  c[n] = sum_k W'[n,k],
//   b'[n] = sum_k beta_k W[n,k] + bias[n]
// (RMSNorm: mu = 0, no beta).  This kernel makes W' (rounded once to the
// weight type), c from the ROUNDED W' (so the mean term cancels exactly what
// the GEMM accumulates) and b', all in one pass over W: one CTA per output
// row n, 16-byte loads, FP32 sums.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ngr_gemm_kernel.cuh"
#include "ngr_internal.h"

namespace ngr {

constexpr int kFoldThreads = 256;

template <bool BF16, bool HAS_BETA>
__global__ void __launch_bounds__(kFoldThreads) fold_prepare_kernel(
    const uint4 *__restrict__ gamma, const uint4 *__restrict__ beta, const uint4 *__restrict__ W,
    const void *__restrict__ bias, int64_t K, int64_t N, uint4 *__restrict__ Wf,
    float *__restrict__ c_out, float *__restrict__ b_out)
{
    __shared__ float red[2][kFoldThreads / 32];
    const int tid = threadIdx.x;
    const int64_t vecs = K >> 3;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        const uint4 *wr = W + n * vecs;
        uint4 *fr = Wf + n * vecs;
        float c = 0.f, b = 0.f;
        for (int64_t v = tid; v < vecs; v += kFoldThreads) {
            const uint4 wv = __ldg(wr + v);
            const uint4 gv = __ldg(gamma + v);
            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
            const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
            uint32_t bw[4] = {0u, 0u, 0u, 0u};
            if constexpr (HAS_BETA) {
                const uint4 bv = __ldg(beta + v);
                bw[0] = bv.x; bw[1] = bv.y; bw[2] = bv.z; bw[3] = bv.w;
            }
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 w2 = to_float2<BF16>(ww[i]);
                const float2 g2 = to_float2<BF16>(gw[i]);
                // The product of two 16-bit values is exact in FP32, so W'
                // is rounded exactly once.
                o[i] = from_float2<BF16>(g2.x * w2.x, g2.y * w2.y);
                const float2 r2 = to_float2<BF16>(o[i]);
                c += r2.x + r2.y;
                if constexpr (HAS_BETA) {
                    const float2 b2 = to_float2<BF16>(bw[i]);
                    b = fmaf(b2.x, w2.x, b);
                    b = fmaf(b2.y, w2.y, b);
                }
            }
            fr[v] = make_uint4(o[0], o[1], o[2], o[3]);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
        }
        if ((tid & 31) == 0) {
            red[0][tid >> 5] = c;
            red[1][tid >> 5] = b;
        }
        __syncthreads();
        if (tid == 0) {
            float tc = 0.f, tb = 0.f;
            for (int w = 0; w < kFoldThreads / 32; ++w) {
                tc += red[0][w];
                tb += red[1][w];
            }
            if (bias) tb += to_float1<BF16>(bias, static_cast<int>(n));
            c_out[n] = tc;
            b_out[n] = tb;
        }
        __syncthreads();
    }
}

// The same fold for any K and N and 2-byte-aligned operands, one element at
// a time: W' is written as [N, K8] rows (K8 = K rounded up to a multiple of
// 8, zero columns past K) and cb as [2, N8] (c, then b'; zero past N), the
// layouts the folded layer reads.  Every W' element is still rounded once
// and c still sums the rounded values.
template <bool BF16, bool HAS_BETA>
__global__ void __launch_bounds__(kFoldThreads) fold_prepare_any_kernel(
    const uint16_t *__restrict__ gamma, const uint16_t *__restrict__ beta,
    const uint16_t *__restrict__ W, const void *__restrict__ bias, int64_t K, int64_t N,
    int64_t K8, int64_t N8, uint16_t *__restrict__ Wf, float *__restrict__ cb)
{
    __shared__ float red[2][kFoldThreads / 32];
    const int tid = threadIdx.x;
    for (int64_t n = blockIdx.x; n < N; n += gridDim.x) {
        float c = 0.f, b = 0.f;
        for (int64_t k = tid; k < K8; k += kFoldThreads) {
            uint16_t o = 0;
            if (k < K) {
                const float w = to_float1<BF16>(W + n * K, static_cast<int>(k));
                const float g = to_float1<BF16>(gamma, static_cast<int>(k));
                const uint32_t r = from_float2<BF16>(g * w, 0.f);
                o = static_cast<uint16_t>(r & 0xffffu);
                c += to_float1<BF16>(&o, 0);
                if constexpr (HAS_BETA) b = fmaf(to_float1<BF16>(beta, static_cast<int>(k)), w, b);
            }
            Wf[n * K8 + k] = o;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            c += __shfl_xor_sync(0xffffffffu, c, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
        }
        if ((tid & 31) == 0) {
            red[0][tid >> 5] = c;
            red[1][tid >> 5] = b;
        }
        __syncthreads();
        if (tid == 0) {
            float tc = 0.f, tb = 0.f;
            for (int w = 0; w < kFoldThreads / 32; ++w) {
                tc += red[0][w];
                tb += red[1][w];
            }
            if (bias) tb += to_float1<BF16>(bias, static_cast<int>(n));
            cb[n] = tc;
            cb[N8 + n] = tb;
        }
        __syncthreads();
    }
    if (blockIdx.x == 0)
        for (int64_t n = N + tid; n < N8; n += kFoldThreads) cb[n] = cb[N8 + n] = 0.f;
}

int launch_fold_prepare_any(int norm, bool bf16, const void *gamma, const void *beta,
                            const void *W, const void *bias, int64_t K, int64_t N, void *Wf,
                            float *cb, int num_sms, cudaStream_t stream)
{
    int64_t blocks = N;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kFoldThreads);
    const int64_t K8 = (K + 7) & ~static_cast<int64_t>(7), N8 = (N + 7) & ~static_cast<int64_t>(7);
    const uint16_t *g = static_cast<const uint16_t *>(gamma);
    const uint16_t *bt = static_cast<const uint16_t *>(beta);
    const uint16_t *w = static_cast<const uint16_t *>(W);
    uint16_t *f = static_cast<uint16_t *>(Wf);
    const bool has_beta = norm == kNormLayer;
#define NGR_FOLD_ANY(B_, H_) \
    fold_prepare_any_kernel<B_, H_><<<grid, block, 0, stream>>>(g, bt, w, bias, K, N, K8, N8, f, cb)
    if (bf16) {
        if (has_beta) NGR_FOLD_ANY(true, true); else NGR_FOLD_ANY(true, false);
    } else {
        if (has_beta) NGR_FOLD_ANY(false, true); else NGR_FOLD_ANY(false, false);
    }
#undef NGR_FOLD_ANY
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : record_cuda_error("fold preparation launch", e, cudaGetErrorString(e));
}

int launch_fold_prepare(int norm, bool bf16, const void *gamma, const void *beta, const void *W,
                        const void *bias, int64_t K, int64_t N, void *Wf, float *cb, int num_sms,
                        cudaStream_t stream)
{
    int64_t blocks = N;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kFoldThreads);
    const uint4 *g = static_cast<const uint4 *>(gamma);
    const uint4 *bt = static_cast<const uint4 *>(beta);
    const uint4 *w = static_cast<const uint4 *>(W);
    uint4 *f = static_cast<uint4 *>(Wf);
    const bool has_beta = norm == kNormLayer;
    if (bf16) {
        if (has_beta)
            fold_prepare_kernel<true, true><<<grid, block, 0, stream>>>(g, bt, w, bias, K, N, f, cb, cb + N);
        else
            fold_prepare_kernel<true, false><<<grid, block, 0, stream>>>(g, bt, w, bias, K, N, f, cb, cb + N);
    } else {
        if (has_beta)
            fold_prepare_kernel<false, true><<<grid, block, 0, stream>>>(g, bt, w, bias, K, N, f, cb, cb + N);
        else
            fold_prepare_kernel<false, false><<<grid, block, 0, stream>>>(g, bt, w, bias, K, N, f, cb, cb + N);
    }
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : record_cuda_error("fold preparation launch", e, cudaGetErrorString(e));
}

}  // namespace ngr
