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

// Device address of the scratch in the CUDA context current on this
// thread, looked up once per context (the first call in a context does it,
// with that context's device current) and kept for later calls.  The cache
// is keyed on the context's process-unique ID, so a context created after a
// cudaDeviceReset, or a caller's own non-primary context on the same device,
// gets its own lookup instead of an address from a module instance that is
// gone or different.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <typename Fn>
Fn driver_fn(const char *name, int version)
{
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(p);
}

struct CtxEntry {
    unsigned long long id;
    void *ptr;
};
constexpr int kNaMaxContexts = 64;
std::mutex g_na_mu;
CtxEntry g_na_cache[kNaMaxContexts] = {};
int g_na_next = 0;

int scratch_address(void **out)
{
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    if (!get_current || !get_id)
        return record_cuda_error("cudaGetDriverEntryPointByVersion(cuCtxGetCurrent/cuCtxGetId)", 0, "");
    std::lock_guard<std::mutex> lock(g_na_mu);
    CUcontext ctx = nullptr;
    CUresult r = get_current(&ctx);
    if (r != CUDA_SUCCESS) return record_cuda_error("cuCtxGetCurrent", static_cast<int>(r), "");
    void *p = nullptr;
    if (!ctx) {
        // No context yet on this thread: the symbol lookup brings up the
        // current device's primary context.
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return record_cuda_error("cudaGetSymbolAddress (no-alloc scratch)", e, cudaGetErrorString(e));
        r = get_current(&ctx);
        if (r != CUDA_SUCCESS || !ctx) return record_cuda_error("cuCtxGetCurrent", static_cast<int>(r), "");
    }
    unsigned long long id = 0;
    r = get_id(ctx, &id);
    if (r != CUDA_SUCCESS) return record_cuda_error("cuCtxGetId", static_cast<int>(r), "");
    for (const CtxEntry &c : g_na_cache)
        if (c.ptr && c.id == id) {
            *out = c.ptr;
            return NGR_OK;
        }
    if (!p) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return record_cuda_error("cudaGetSymbolAddress (no-alloc scratch)", e, cudaGetErrorString(e));
    }
    g_na_cache[g_na_next] = CtxEntry{id, p};
    g_na_next = (g_na_next + 1) % kNaMaxContexts;
    *out = p;
    return NGR_OK;
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
    if (!map_2d(&a.map_a, x, bf16, M, K, kBM) ||
        !map_2d(&a.map_b, W, bf16, N, K, static_cast<uint32_t>(plan.b_rows)) ||
        (plan.mc && !map_2d(&a.map_b2, W, bf16, N, K, 64)) ||
        !map_gb(&a.map_gb, gamma_f, K, kNaGB))
        return NGR_ERR_CUDA;
    a.stats = stats;
    a.gamma_f = gamma_f;
    a.beta_f = beta_f;
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
    a.timeout_ns = wait_timeout_ns();
    a.act = kActNone;
    a.k_splits = 1;   // no K split: the scratch holds no partials
    a.kb_per_split = a.k_blocks;
    rc = launch_gemm(kNormLayer, bf16, plan, a, true, stream);
    if (rc != NGR_OK) return rc;
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error("kernel launch (no-alloc)", e, cudaGetErrorString(e));
    if (debug_mode()) return ngr_noalloc_error(stream_);
    return NGR_OK;
}

extern "C" int ngr_noalloc_error(ngr_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != NGR_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return record_cuda_error("cudaStreamSynchronize", e, cudaGetErrorString(e));
    int v = 0;
    e = cudaMemcpy(&v, base, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return record_cuda_error("cudaMemcpy (no-alloc error word)", e, cudaGetErrorString(e));
    if (v != 0) {
        e = cudaMemset(base, 0, sizeof(int));
        if (e != cudaSuccess) return record_cuda_error("cudaMemset (no-alloc error word)", e, cudaGetErrorString(e));
    }
    return v == 0 ? NGR_OK : NGR_ERR_TIMEOUT;
}
