// ngr_pad.cu -- copies that let the single-layer entry points take any K
// and N ("昇腾CANN的MatMul融合玩法，让大模型推理快3倍", §五 optimization 1: a
// 513 x 14337 activation against a 49152 x 14337 weight, sizes that are not
// multiples of the aligned access width).
//
// The tile and decode kernels read x and W through TMA, whose row pitch
// must be a multiple of 16 bytes, and store y with 16-byte stores.  When K
// or N is not a multiple of 8 the library copies the operands into the
// workspace with rows padded to a multiple of 8 elements (the padding is
// zero, so the products are unchanged; the statistics kernel counts only
// the K real columns), runs the aligned path, and copies the real N columns
// of the padded output back.  The copies read and write 16-bit elements one
// at a time, so the caller's pointers need only 2-byte alignment here.
#include <cuda_runtime.h>

#include "ngr_internal.h"

namespace ngr {

constexpr int kPadThreads = 256;

// dst[r, c] = r < rows && c < cols ? src[r * src_pitch + c] : 0 for
// r < dst_rows, c < dst_cols (dst_cols % 8 == 0, dst 16-byte aligned); one
// 16-byte vector per thread.
__global__ void __launch_bounds__(kPadThreads) pad_rows_kernel(
    const uint16_t *__restrict__ src, int64_t rows, int64_t cols, int64_t src_pitch,
    uint4 *__restrict__ dst, int64_t dst_cols, int64_t dst_rows)
{
    const int64_t vecs = dst_cols >> 3;
    const int64_t total = dst_rows * vecs;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / vecs;
        const int64_t c0 = (i - r * vecs) << 3;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (r < rows) {
            const uint16_t *s = src + r * src_pitch;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t c = c0 + 2 * j;
                const uint32_t lo = c < cols ? __ldg(s + c) : 0u;
                const uint32_t hi = c + 1 < cols ? __ldg(s + c + 1) : 0u;
                w[j] = lo | (hi << 16);
            }
        }
        dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// dst[r * cols + c] = src[r * src_pitch + c] for c < cols.
__global__ void __launch_bounds__(kPadThreads) unpad_rows_kernel(
    const uint16_t *__restrict__ src, int64_t rows, int64_t cols, int64_t src_pitch,
    uint16_t *__restrict__ dst)
{
    const int64_t total = rows * cols;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / cols;
        const int64_t c = i - r * cols;
        dst[i] = src[r * src_pitch + c];
    }
}

static unsigned grid_for(int64_t work, int num_sms)
{
    int64_t b = (work + kPadThreads - 1) / kPadThreads;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (b > cap) b = cap;
    return static_cast<unsigned>(b < 1 ? 1 : b);
}

int launch_pad_rows(const void *src, int64_t rows, int64_t cols, int64_t src_pitch, void *dst,
                    int64_t dst_cols, int num_sms, cudaStream_t stream, int64_t dst_rows)
{
    if (dst_rows < rows) dst_rows = rows;
    if (dst_rows <= 0) return 0;
    pad_rows_kernel<<<grid_for(dst_rows * (dst_cols >> 3), num_sms), kPadThreads, 0, stream>>>(
        static_cast<const uint16_t *>(src), rows, cols, src_pitch, static_cast<uint4 *>(dst),
        dst_cols, dst_rows);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : record_cuda_error("padding copy launch", e, cudaGetErrorString(e));
}

int launch_unpad_rows(const void *src, int64_t rows, int64_t cols, int64_t src_pitch, void *dst,
                      int num_sms, cudaStream_t stream)
{
    if (rows <= 0) return 0;
    unpad_rows_kernel<<<grid_for(rows * cols, num_sms), kPadThreads, 0, stream>>>(
        static_cast<const uint16_t *>(src), rows, cols, src_pitch, static_cast<uint16_t *>(dst));
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? 0 : record_cuda_error("unpadding copy launch", e, cudaGetErrorString(e));
}

}  // namespace ngr
