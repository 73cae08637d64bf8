// ngr_noalloc.cu -- a variant of the fused LayerNorm + linear entry point
// for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// where device allocation is forbidden or unavailable (a region whose memory
// is planned up front, a host runtime that owns every device allocation and
// exposes none, an embedding that only passes tensors in and out).  For them
// this file keeps the scratch the layer needs -- the per-row statistics,
// gamma and beta as FP32, and the error word -- in one fixed array in the
// library's own device memory, so the caller passes only inputs and outputs.
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it, at its full size, until the process exits.
//
// Limits: M <= NGR_NOALLOC_MAX_M and K <= NGR_NOALLOC_MAX_K (ngr.h); larger
// sizes are rejected with NGR_ERR_SHAPE before anything runs.  This path
// always uses the tile kernel (it keeps no split-K partials).
//
// Sharing: all calls, from any thread or stream, use the same array, which
// keeps whatever the last call wrote.  Each call rewrites the statistics and
// the FP32 gamma/beta it reads and clears the error word first, so nothing
// carries over between calls that are ordered; calls that overlap on the GPU
// race on the array and must not be issued.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "ngr.h"
#include "ngr_internal.h"

namespace ngr {
namespace {

constexpr size_t kNaHeader = 256;
constexpr size_t kNaStats = static_cast<size_t>(NGR_NOALLOC_MAX_M) * 8;
constexpr size_t kNaGB = static_cast<size_t>(NGR_NOALLOC_MAX_K) * 4;  // one FP32 row
constexpr size_t kNaBytes = kNaHeader + kNaStats + 2 * kNaGB;

// The scratch itself.  In host code this name is only a host-side stand-in;
// the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

constexpr int kNaMaxDevices = 64;
std::mutex g_na_mu;
void *g_na_ptr[kNaMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device with that device current (the first call on a device does it).
int scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices)
        return NGR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return NGR_ERR_CUDA;
        g_na_ptr[dev] = p;
    }
    *out = g_na_ptr[dev];
    return NGR_OK;
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                              const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                              const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn na_encode()
{
    static EncodeFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

bool na_map(CUtensorMap *m, CUtensorMapDataType t, void *ptr, uint64_t cols, uint64_t rows,
            uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw)
{
    EncodeFn enc = na_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, t, 2, ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
               sw == CU_TENSOR_MAP_SWIZZLE_NONE ? CU_TENSOR_MAP_L2_PROMOTION_NONE
                                                : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ngr

using namespace ngr;

extern "C" int ngr_fused_layernorm_linear_noalloc(const void *x, const void *gamma,
                                                  const void *beta, const void *W,
                                                  const void *bias, float eps, int64_t M,
                                                  int64_t K, int64_t N, int dtype, void *y,
                                                  ngr_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (M < 0 || K <= 0 || N <= 0 || N >= (int64_t(1) << 31)) return NGR_ERR_SHAPE;
    if (M > NGR_NOALLOC_MAX_M || K > NGR_NOALLOC_MAX_K) return NGR_ERR_SHAPE;
    if (K % 8 != 0 || N % 8 != 0) return NGR_ERR_ALIGN;
    if (M == 0) return NGR_OK;
    if (!x || !gamma || !beta || !W || !y) return NGR_ERR_NULL;
    if (!al16(x) || !al16(gamma) || !al16(beta) || !al16(W) || !al16(y) || (bias && !al16(bias)))
        return NGR_ERR_ALIGN;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return NGR_ERR_CUDA;
    if (major != 10 || minor != 3) return NGR_ERR_ARCH;

    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != NGR_OK) return rc;
    char *s = static_cast<char *>(base);
    int *err = reinterpret_cast<int *>(s);
    float2 *stats = reinterpret_cast<float2 *>(s + kNaHeader);
    float *gamma_f = reinterpret_cast<float *>(s + kNaHeader + kNaStats);
    float *beta_f = reinterpret_cast<float *>(s + kNaHeader + kNaStats + kNaGB);
    const bool bf16 = dtype == NGR_BF16;

    // Step a1 (also converts gamma/beta to FP32 and clears the error word).
    rc = launch_rowstats(kNormLayer, bf16, x, M, K, eps, stats, gamma, beta, gamma_f, beta_f,
                         nullptr, 0, err, sms, stream);
    if (rc != NGR_OK) return rc;

    // Steps a2-a4: the tile kernel, as a programmatic dependent of a1.
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    const GemmPlan plan = plan_gemm(M, N, K, sms, true);
    const CUtensorMapDataType t16 =
        bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!na_map(&a.map_a, t16, const_cast<void *>(x), K, M, K * 2, kBK, kBM,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
        !na_map(&a.map_b, t16, const_cast<void *>(W), K, N, K * 2, kBK,
                static_cast<uint32_t>(plan.b_rows), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !na_map(&a.map_gb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, gamma_f, K, 2, kNaGB, kBK, 2,
                CU_TENSOR_MAP_SWIZZLE_NONE))
        return NGR_ERR_CUDA;
    a.stats = stats;
    a.bias = bias;
    a.y = y;
    a.err = err;
    a.zero_err = 0;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.m_tiles = static_cast<int>((M + plan.bm - 1) / plan.bm);
    a.n_tiles = static_cast<int>((N + plan.tw - 1) / plan.tw);
    a.k_blocks = static_cast<int>((K + kBK - 1) / kBK);
    a.num_tiles = a.m_tiles * a.n_tiles;
    a.timeout_ns = 2000ull * 1000000ull;
    a.act = kActNone;
    a.k_splits = 1;   // no K split: the scratch holds no partials
    a.kb_per_split = a.k_blocks;
    rc = launch_gemm(kNormLayer, bf16, plan, a, true, stream);
    if (rc != NGR_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? NGR_OK : NGR_ERR_CUDA;
}
