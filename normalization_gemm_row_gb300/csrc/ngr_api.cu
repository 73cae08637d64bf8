// ngr_api.cu -- the C ABI declared in include/ngr.h: argument checks,
// workspace layout, TMA descriptor encoding, choice of kernel and launch on
// the caller's stream.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>
#include <vector>

#include "ngr.h"
#include "ngr_internal.h"
#include "ngr_ptx.cuh"

namespace ngr {

namespace {
thread_local char g_last_error[512] = "";

// Per-thread kernel timing (see ngr_kernel_timing_start): the library's own
// events, two per kernel slot, reused across timing sessions.
constexpr int kSlots = NGR_MAX_KERNELS_PER_CALL;
thread_local std::vector<cudaEvent_t> t_events;
thread_local std::vector<int> t_count;  // kernels recorded per timed call
thread_local bool t_armed = false;
thread_local int t_calls = 0;           // calls to time in this session
thread_local int t_call = 0;            // index of the current call
thread_local int t_kernel = 0;          // index of the next kernel in the call

void events_reset() { t_kernel = 0; }
void events_call_done()
{
    if (t_armed && t_call < t_calls) ++t_call;
}
void event_before(cudaStream_t s)
{
    if (t_armed && t_call < t_calls && t_kernel < kSlots)
        cudaEventRecord(t_events[2 * (t_call * kSlots + t_kernel)], s);
}
void event_after(cudaStream_t s)
{
    if (t_armed && t_call < t_calls && t_kernel < kSlots) {
        cudaEventRecord(t_events[2 * (t_call * kSlots + t_kernel) + 1], s);
        ++t_kernel;
        t_count[t_call] = t_kernel;
    }
}
}  // namespace

int record_cuda_error(const char *what, int code, const char *detail)
{
    std::snprintf(g_last_error, sizeof(g_last_error), "%s failed: code %d (%s)", what, code,
                  detail ? detail : "");
    return -7;
}

namespace {

constexpr size_t kHeaderBytes = 256;  // error word + padding
constexpr int kMaxDevices = 64;

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
    size_t stats = 0, gamma_f = 0, beta_f = 0;
    // padded copies (single-layer ops with K or N not a multiple of 8)
    size_t xp = 0, wp = 0, gp = 0, bp = 0, biasp = 0, yp = 0;
    bool padded = false;
    // K-split counters and partials of the split-eligible product
    size_t split_cnt = 0, split_cnt_bytes = 0, split_part = 0, split_part_bytes = 0;
    size_t partials = 0, counters = 0, counters2 = 0, h = 0;
    size_t total = 0;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round8(int64_t v) { return (v + 7) & ~static_cast<int64_t>(7); }

// Room for a K split of an M x Nout product (K_in input columns), reserved
// only where the tiles are few for a GPU's SMs: on the CTA-pair and
// multicast kernels (M > 128) a two-way split when the output has few
// 256 x 448 tiles; on the
// single-CTA kernel (M <= 128) up to kMaxSplitsSingle ways when the output
// has fewer than 256 tiles of 128 columns and K_in is long enough to split.
// The largest counters and partials over the tile widths, so that any plan
// fits.  Independent of the device.
void split_reserve(int64_t M, int64_t Nout, int64_t K_in, size_t *cnt_bytes, size_t *part_bytes)
{
    *cnt_bytes = *part_bytes = 0;
    if (M <= kBM) {
        if ((Nout + 127) / 128 >= 256 || (K_in + kBK - 1) / kBK < 2 * kMinKbPerSplitSingle) return;
        for (int tw : {128, 192, 224, 256}) {
            const int64_t tiles = (Nout + tw - 1) / tw;
            *cnt_bytes = std::max(*cnt_bytes, split_counter_bytes(tiles, tw, 1));
            *part_bytes = std::max(*part_bytes, split_partial_bytes(tiles, tw, kMaxSplitsSingle, 1));
        }
        return;
    }
    const int64_t mt = (M + 2 * kBM - 1) / (2 * kBM);
    if (mt * ((Nout + 447) / 448) > 48) return;
    for (int tw : {128, 192, 224, 256, 384, 448, 512}) {
        const int64_t tiles = mt * ((Nout + tw - 1) / tw);
        *cnt_bytes = std::max(*cnt_bytes, split_counter_bytes(tiles, tw));
        *part_bytes = std::max(*part_bytes, split_partial_bytes(tiles, tw, 2));
    }
    if (M > 2 * kBM) {   // the multicast kernel's 512 x 464 super-tiles, split in two
        const int64_t super = ((M + kMcRows - 1) / kMcRows) * ((Nout + kMcCols - 1) / kMcCols);
        *cnt_bytes = std::max(*cnt_bytes, mc_split_counter_bytes(super));
        *part_bytes = std::max(*part_bytes, mc_split_partial_bytes(super, 2));
    }
}

// Ops that take any K and N (through padded copies).
bool single_layer_op(int op)
{
    return op == NGR_OP_LAYERNORM_LINEAR || op == NGR_OP_RMSNORM_LINEAR ||
           op == NGR_OP_LINEAR_SILU || op == NGR_OP_NORM_LINEAR;
}

// Workspace regions, in order: header | stats | gamma_f | beta_f |
// normalized rows (decode sizes) | decode partials | counters of the first
// GEMM | counters of the second GEMM (FFN / MLP chains) | H.
//
// Ops with a norm: LayerNorm/RMSNorm linear, the general norm + activation
// layer, the MLP chain and both SwiGLU forms (sized for the worst case: a
// call without a norm uses less).  At decode sizes (M <= 32) the first GEMM
// runs on the decode kernel except for SwiGLU, whose gated tiles run on the
// CTA-pair kernel at every M; the second GEMM of a chain (K output
// columns) always takes the decode kernel there.
WsLayout ws_layout(int op, int64_t M, int64_t K_, int64_t N_, bool h_in_ws)
{
    WsLayout L;
    size_t off = kHeaderBytes;
    // A single layer with K or N not a multiple of 8 runs on rows padded to
    // K8 / N8; the padded copies follow the regular regions.
    const bool pad = single_layer_op(op) && (K_ % 8 != 0 || N_ % 8 != 0);
    const int64_t K = pad ? round8(K_) : K_;
    const int64_t N = pad ? round8(N_) : N_;
    const bool norm = op == NGR_OP_LAYERNORM_LINEAR || op == NGR_OP_RMSNORM_LINEAR ||
                      op == NGR_OP_NORM_LINEAR || op == NGR_OP_MLP || op == NGR_OP_SWIGLU ||
                      op == NGR_OP_MLP_SWIGLU;
    const bool gated = op == NGR_OP_SWIGLU || op == NGR_OP_MLP_SWIGLU;
    const bool chain = op == NGR_OP_FFN || op == NGR_OP_MLP || op == NGR_OP_MLP_SWIGLU;
    const bool post_norm = op == NGR_OP_LINEAR_RESIDUAL_NORM;
    const bool decode = M > 0 && M <= kDecodeMaxM;
    if (norm) {
        L.stats = off;
        off += align256(static_cast<size_t>(M) * 8);
        L.gamma_f = off;
        off += align256(static_cast<size_t>(K) * 4);
        L.beta_f = off;
        off += align256(static_cast<size_t>(K) * 4);
    }
    if (decode) {
        const int64_t mn = M <= 16 ? 16 : 32;
        const int64_t tiles1 = gated ? 0 : ceil_div(N, 128);
        const int64_t tiles2 = chain ? ceil_div(K, 128) : 0;
        const int64_t tmax = tiles1 > tiles2 ? tiles1 : tiles2;
        L.partials = off;
        off += align256(static_cast<size_t>(tmax) * kDecodeMaxGroups * mn * 128 * 4);
        L.counters = off;
        off += align256(static_cast<size_t>(tiles1) * 4 * 4);
        L.counters2 = off;
        off += align256(static_cast<size_t>(tiles2) * 4 * 4);
    }
    if (chain && h_in_ws) {
        L.h = off;
        off += align256(static_cast<size_t>(M) * static_cast<size_t>(N) * 2);
    }
    if (post_norm) {
        // statistics of the output rows; h [M, N] when the caller keeps none
        L.stats = off;
        off += align256(static_cast<size_t>(M) * 8);
        if (h_in_ws) {
            L.h = off;
            off += align256(static_cast<size_t>(M) * static_cast<size_t>(N) * 2);
        }
    }
    {
        // the product that may split K: the single layer's, or the chain's
        // second (K output columns)
        const bool single = single_layer_op(op) || post_norm;
        const int64_t nout = single ? N : K;
        const int64_t kin = single ? K : N;
        if ((single || chain) && !decode) {
            split_reserve(M, nout, kin, &L.split_cnt_bytes, &L.split_part_bytes);
            L.split_cnt = off;
            off += align256(L.split_cnt_bytes);
            L.split_part = off;
            off += align256(L.split_part_bytes);
        }
    }
    if (pad) {
        L.padded = true;
        L.xp = off;
        off += align256(static_cast<size_t>(M) * static_cast<size_t>(K) * 2);
        L.wp = off;
        off += align256(static_cast<size_t>(N_) * static_cast<size_t>(K) * 2);
        L.gp = off;
        off += align256(static_cast<size_t>(K) * 2);
        L.bp = off;
        off += align256(static_cast<size_t>(K) * 2);
        L.biasp = off;
        off += align256(static_cast<size_t>(N) * 2);
        L.yp = off;
        off += align256(static_cast<size_t>(M) * static_cast<size_t>(N) * 2);
    }
    L.total = off;
    return L;
}

// ------------------------------------------------------------- device info
struct DevInfo {
    bool ready = false;
    bool arch_ok = false;
    int sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[kMaxDevices];

int current_device_info(DevInfo *out)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_error("cudaGetDevice", e, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return NGR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return NGR_ERR_CUDA;
        d.arch_ok = (major == 10 && minor == 3);
        d.sms = sms;
        d.ready = true;
    }
    *out = d;
    return d.arch_ok ? NGR_OK : NGR_ERR_ARCH;
}

}  // namespace

// ------------------------------------------------------------ environment
bool debug_mode()
{
    static const bool on = [] {
        const char *v = std::getenv("NGR_DEBUG");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

bool trace_mode()
{
    static const bool on = [] {
        const char *v = std::getenv("NGR_TRACE");
        return v && v[0] && std::strcmp(v, "0") != 0;
    }();
    return on;
}

unsigned long long wait_timeout_ns()
{
    static const unsigned long long ns = [] {
        const char *v = std::getenv("NGR_WAIT_TIMEOUT_MS");
        long long ms = v ? std::atoll(v) : 0;
        if (ms <= 0) ms = 2000;
        return static_cast<unsigned long long>(ms) * 1000000ull;
    }();
    return ns;
}

// ---------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Row-major [rows, cols] 16-bit matrix, box {64 columns, box_rows rows},
// 128-byte swizzle (the layout the tensor core reads K-major operands in).
bool aligned2(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }

bool map_2d(CUtensorMap *m, const void *ptr, bool bf16, int64_t rows, int64_t cols,
            uint32_t box_rows)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        record_cuda_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", 0, "");
        return false;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                           const_cast<void *>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_cuda_error("cuTensorMapEncodeTiled (2-D)", static_cast<int>(r), "");
        return false;
    }
    return true;
}

// FP32 gamma and beta as the two rows of a [2, K] matrix whose rows are
// `row_stride` bytes apart; box {64 columns, 2 rows}, no swizzle.
bool map_gb(CUtensorMap *m, const float *gamma_f, int64_t K, size_t row_stride)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) {
        record_cuda_error("cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", 0, "");
        return false;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), 2};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_stride)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBK), 2};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(gamma_f),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_cuda_error("cuTensorMapEncodeTiled (gamma/beta)", static_cast<int>(r), "");
        return false;
    }
    return true;
}

namespace {

// ------------------------------------------------------------- validation
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int64_t kMaxDim = int64_t(1) << 31;

int check_sizes(int64_t M, int64_t K, int64_t N, int dtype)
{
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (M < 0 || K <= 0 || N <= 0) return NGR_ERR_SHAPE;
    if (M >= kMaxDim || K >= kMaxDim || N >= kMaxDim) return NGR_ERR_SHAPE;
    if (K % 8 != 0 || N % 8 != 0) return NGR_ERR_ALIGN;
    return NGR_OK;
}

// The K-split counters start every call at zero (the kernels also reset
// each counter after its last use); first on the stream, before any kernel.
int zero_split_counters(const WsLayout &L, char *ws, cudaStream_t stream)
{
    if (L.split_cnt_bytes == 0) return NGR_OK;
    const cudaError_t e = cudaMemsetAsync(ws + L.split_cnt, 0, L.split_cnt_bytes, stream);
    return e == cudaSuccess ? NGR_OK : record_cuda_error("cudaMemsetAsync (split counters)", e,
                                                         cudaGetErrorString(e));
}

int finish(int rc, void *ws, cudaStream_t stream)
{
    if (rc != NGR_OK) return rc;
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return record_cuda_error("kernel launch", e, cudaGetErrorString(e));
    if (debug_mode()) return ngr_workspace_error(ws, reinterpret_cast<ngr_stream_t>(stream));
    return NGR_OK;
}

// One linear layer y = act(norm(x) W^T + bias) on its own, given the
// workspace regions.  `stats_ready` says whether a preceding grid on the
// stream produced what this one reads (then it is launched as a
// programmatic dependent).
int launch_layer(int norm, int act, bool bf16, const void *x, const void *W,
                 const void *bias, int64_t M, int64_t K, int64_t N, void *y,
                 char *ws, const WsLayout &L, size_t counters_off, bool pdl,
                 const DevInfo &di, cudaStream_t stream, const float *fold_c = nullptr,
                 const float *fold_b = nullptr, int64_t w_rows = -1,
                 const void *residual = nullptr, bool may_split = false)
{
    // W has w_rows rows (N unless the output is padded past W's rows; the
    // tensor maps zero-fill the rest).
    if (w_rows < 0) w_rows = N;
    // A kernel launched as a programmatic dependent is never a call's first.
    const int zero_err = pdl ? 0 : 1;
    int *err = reinterpret_cast<int *>(ws);
    const bool has_norm = norm == kNormLayer || norm == kNormRms;   // transform stage
    const bool has_stats = norm != kNormNone;
    float2 *stats = has_stats ? reinterpret_cast<float2 *>(ws + L.stats) : nullptr;
    float *gf = has_norm ? reinterpret_cast<float *>(ws + L.gamma_f) : nullptr;
    if (M <= kDecodeMaxM) {
        DecodeArgs d;
        std::memset(&d, 0, sizeof(d));
        const int mn = M <= 16 ? 16 : 32;
        if (!map_2d(&d.map_w, W, bf16, w_rows, K, 128) || !map_2d(&d.map_x, x, bf16, M, K, mn))
            return NGR_ERR_CUDA;
        d.stats = stats;
        d.gamma_f = gf;
        d.beta_f = norm == kNormLayer ? reinterpret_cast<float *>(ws + L.beta_f) : nullptr;
        d.bias = bias;
        d.fold_c = fold_c;
        d.fold_b = fold_b;
        d.residual = residual;
        d.y = y;
        d.partials = reinterpret_cast<float *>(ws + L.partials);
        d.counters = reinterpret_cast<int *>(ws + counters_off);
        d.err = err;
        d.zero_err = zero_err;
        d.M = static_cast<int>(M);
        d.N = static_cast<int>(N);
        d.K = static_cast<int>(K);
        d.n_tiles = static_cast<int>(ceil_div(N, 128));
        d.k_blocks = static_cast<int>(ceil_div(K, kBK));
        const DecodePlan dp = plan_decode(d.n_tiles, d.k_blocks, mn, di.sms);
        d.k_groups = dp.k_groups;
        d.kb_per_group = dp.kb_per_group;
        d.n_groups = dp.n_groups;
        if (trace_mode())
            std::fprintf(stderr, "ngr: decode kernel M=%lld N=%lld K=%lld norm=%d MN=%d grid=%d x %d (k blocks per group %d)\n",
                         static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K),
                         norm, mn, dp.k_groups, dp.n_groups, dp.kb_per_group);
        d.timeout_ns = wait_timeout_ns();
        d.act = act;
        return launch_decode(norm, bf16, mn, d, pdl, stream);
    }
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    const GemmPlan plan = plan_gemm(M, N, K, di.sms, has_norm,
                                    may_split ? L.split_cnt_bytes + L.split_part_bytes : 0,
                                    norm == kNormNone || is_fold(norm));
    if (trace_mode())
        std::fprintf(stderr, "ngr: tile kernel M=%lld N=%lld K=%lld norm=%d %s BN=%d x %d splits=%d stages=%d grid=%d smem=%zu\n",
                     static_cast<long long>(M), static_cast<long long>(N), static_cast<long long>(K), norm,
                     plan.pair ? "cta-pair" : "single-cta", plan.bn, plan.nsub, plan.splits, plan.stages,
                     plan.grid, plan.smem);
    if (!map_2d(&a.map_a, x, bf16, M, K, kBM) ||
        !map_2d(&a.map_b, W, bf16, w_rows, K, static_cast<uint32_t>(plan.b_rows)))
        return NGR_ERR_CUDA;
    // The multicast kernel's second weight map: 64-row parts of the 240-row sub-tile.
    if (plan.mc && !map_2d(&a.map_b2, W, bf16, w_rows, K, 64)) return NGR_ERR_CUDA;
    if (has_norm && !map_gb(&a.map_gb, gf, K, L.beta_f - L.gamma_f)) return NGR_ERR_CUDA;
    a.stats = stats;
    a.gamma_f = gf;
    a.beta_f = has_norm ? reinterpret_cast<float *>(ws + L.beta_f) : nullptr;
    a.bias = bias;
    a.fold_c = fold_c;
    a.fold_b = fold_b;
    a.residual = residual;
    a.y = y;
    a.err = err;
    a.zero_err = zero_err;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(N);
    a.K = static_cast<int>(K);
    a.m_tiles = static_cast<int>(ceil_div(M, plan.bm));
    a.n_tiles = static_cast<int>(ceil_div(N, plan.tw));
    a.k_blocks = static_cast<int>(ceil_div(K, kBK));
    a.num_tiles = a.m_tiles * a.n_tiles;
    a.timeout_ns = wait_timeout_ns();
    a.act = act;
    a.k_splits = plan.splits > 1 ? plan.splits : 1;
    a.kb_per_split = static_cast<int>(ceil_div(a.k_blocks, a.k_splits));
    if (a.k_splits > 1) {
        a.split_counters = reinterpret_cast<int *>(ws + L.split_cnt);
        a.partials = reinterpret_cast<float *>(ws + L.split_part);
    }
    return launch_gemm(norm, bf16, plan, a, pdl, stream);
}

// Whether the product launch_layer runs for these sizes (with the split
// regions of L) splits K, and so needs its split counters at zero.
bool product_splits(int norm, int64_t M, int64_t K, int64_t N, const WsLayout &L, const DevInfo &di)
{
    if (M <= kDecodeMaxM || L.split_cnt_bytes == 0) return false;
    const bool has_norm = norm == kNormLayer || norm == kNormRms;
    return plan_gemm(M, N, K, di.sms, has_norm, L.split_cnt_bytes + L.split_part_bytes,
                     norm == kNormNone || is_fold(norm)).splits > 1;
}

// The gated (SwiGLU) layer h = SiLU(norm(x) Wg^T) * (norm(x) Wu^T) on the
// CTA-pair kernel, at any M.
int launch_gated(int norm, bool bf16, const void *x, const void *Wg, const void *Wu, int64_t M,
                 int64_t K, int64_t F, void *h, char *ws, const WsLayout &L, bool pdl,
                 const DevInfo &di, cudaStream_t stream)
{
    GemmArgs a;
    std::memset(&a, 0, sizeof(a));
    const bool has_norm = norm == kNormLayer || norm == kNormRms;
    const GemmPlan plan = plan_gemm_gated(M, F, di.sms);
    if (trace_mode())
        std::fprintf(stderr, "ngr: gated tile kernel M=%lld F=%lld K=%lld norm=%d BN=%d stages=%d grid=%d smem=%zu\n",
                     static_cast<long long>(M), static_cast<long long>(F), static_cast<long long>(K), norm,
                     plan.bn, plan.stages, plan.grid, plan.smem);
    if (!map_2d(&a.map_a, x, bf16, M, K, kBM) ||
        !map_2d(&a.map_b, Wg, bf16, F, K, static_cast<uint32_t>(plan.b_rows)) ||
        !map_2d(&a.map_b2, Wu, bf16, F, K, static_cast<uint32_t>(plan.b_rows)))
        return NGR_ERR_CUDA;
    if (has_norm && !map_gb(&a.map_gb, reinterpret_cast<float *>(ws + L.gamma_f), K,
                            L.beta_f - L.gamma_f))
        return NGR_ERR_CUDA;
    a.stats = has_norm ? reinterpret_cast<float2 *>(ws + L.stats) : nullptr;
    a.y = h;
    a.err = reinterpret_cast<int *>(ws);
    a.zero_err = pdl ? 0 : 1;
    a.act = kActNone;
    a.M = static_cast<int>(M);
    a.N = static_cast<int>(F);
    a.K = static_cast<int>(K);
    a.m_tiles = static_cast<int>(ceil_div(M, plan.bm));
    a.n_tiles = static_cast<int>(ceil_div(F, plan.tw));
    a.k_blocks = static_cast<int>(ceil_div(K, kBK));
    a.num_tiles = a.m_tiles * a.n_tiles;
    a.timeout_ns = wait_timeout_ns();
    return launch_gemm(norm, bf16, plan, a, pdl, stream);
}

int norm_linear(int op, int norm, int act, const void *x, const void *gamma, const void *beta,
                const void *W, const void *bias, float eps, int64_t M, int64_t K, int64_t N,
                int dtype, void *y, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (M < 0 || K <= 0 || N <= 0 || M >= kMaxDim || K >= kMaxDim || N >= kMaxDim)
        return NGR_ERR_SHAPE;
    if (M == 0) return NGR_OK;
    if (!x || !W || !y || !ws) return ws ? NGR_ERR_NULL : (x && W && y ? NGR_ERR_WORKSPACE : NGR_ERR_NULL);
    if (norm != kNormNone && !gamma) return NGR_ERR_NULL;
    if (norm == kNormLayer && !beta) return NGR_ERR_NULL;
    const bool pad = K % 8 != 0 || N % 8 != 0;
    // Aligned shapes need 16-byte pointers; padded ones are copied with
    // 2-byte accesses, except y when N needs no padding (stored directly).
    auto ok_ptr = [&](const void *p) {
        return !p || (pad ? aligned2(p) : aligned16(p));
    };
    if (!ok_ptr(x) || !ok_ptr(W) || !ok_ptr(gamma) || !ok_ptr(beta) || !ok_ptr(bias) ||
        !(N % 8 != 0 ? aligned2(y) : aligned16(y)))
        return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    const WsLayout L = ws_layout(op, M, K, N, false);
    if (ws_bytes < L.total) return NGR_ERR_WORKSPACE;
    DevInfo di;
    int rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool bf16 = dtype == NGR_BF16;
    char *w = static_cast<char *>(ws);
    if (debug_mode() && cudaMemsetAsync(w, 0, 4, stream) != cudaSuccess) return NGR_ERR_CUDA;
    const bool decode = M <= kDecodeMaxM;
    const bool need_stats = norm != kNormNone || decode;
    // With the statistics kernel first on the stream, it zeroes the K-split
    // counters itself (no separate memset before it).
    const bool stats_zero = need_stats && !decode && L.split_cnt_bytes != 0;
    if (!stats_zero && product_splits(norm, M, round8(K), round8(N), L, di)) {
        rc = zero_split_counters(L, w, stream);
        if (rc != NGR_OK) return rc;
    }
    // Padded operands: rows of K8 (N8) elements with zero tails.
    const int64_t K8 = round8(K), N8 = round8(N);
    const void *xa = x, *Wa = W, *ga = gamma, *ba = beta, *biasa = bias;
    void *ya = y;
    if (pad) {
        // An operand is copied when its rows need padding or its pointer
        // is not 16-byte aligned (the kernels read it with TMA or 16-byte
        // loads).
        auto copy = [&](const void *src, int64_t rows, size_t off, const void **dst) {
            if (!src || (K8 == K && aligned16(src))) return 0;
            *dst = w + off;
            return launch_pad_rows(src, rows, K, K, w + off, K8, di.sms, stream);
        };
        rc = copy(x, M, L.xp, &xa);
        if (rc == 0) rc = copy(W, N, L.wp, &Wa);
        if (rc == 0) rc = copy(gamma, 1, L.gp, &ga);
        if (rc == 0) rc = copy(beta, 1, L.bp, &ba);
        if (rc != 0) return rc;
        if (bias) {
            rc = launch_pad_rows(bias, 1, N, N, w + L.biasp, N8, di.sms, stream);
            if (rc != 0) return rc;
            biasa = w + L.biasp;
        }
        if (N8 != N) ya = w + L.yp;
    }
    events_reset();
    if (need_stats) {
        event_before(stream);
        rc = launch_rowstats(norm == kNormNone ? kNormRms : norm, bf16, xa,
                             norm == kNormNone ? 0 : M, K8, eps,
                             reinterpret_cast<float2 *>(w + L.stats), ga, ba,
                             norm == kNormNone ? nullptr : reinterpret_cast<float *>(w + L.gamma_f),
                             norm == kNormLayer ? reinterpret_cast<float *>(w + L.beta_f)
                                                : (norm == kNormRms ? reinterpret_cast<float *>(w + L.beta_f) : nullptr),
                             decode ? reinterpret_cast<int *>(w + L.counters)
                                    : (stats_zero ? reinterpret_cast<int *>(w + L.split_cnt) : nullptr),
                             decode ? static_cast<int>(ceil_div(N8, 128) * 4)
                                    : (stats_zero ? static_cast<int>(L.split_cnt_bytes / 4) : 0),
                             reinterpret_cast<int *>(w), di.sms, stream, nullptr, K);
        event_after(stream);
        if (rc != NGR_OK) return rc;
    }
    event_before(stream);
    rc = launch_layer(norm, act, bf16, xa, Wa, biasa, M, K8, N8, ya, w, L, L.counters, need_stats,
                      di, stream, nullptr, nullptr, N, nullptr, true);
    event_after(stream);
    if (rc == NGR_OK && ya != y) rc = launch_unpad_rows(ya, M, N, N8, y, di.sms, stream);
    events_call_done();
    return finish(rc, ws, stream);
}

// The folded layer: statistics of x (a1), then one GEMM on raw x against the
// folded weight with the statistics applied in the epilogue (a7).
int folded_linear(int norm, const void *x, const void *Wf, const float *cb, float eps,
                  int64_t M, int64_t K, int64_t N, int dtype, void *y, void *ws,
                  size_t ws_bytes, cudaStream_t stream)
{
    if (norm != kNormLayer && norm != kNormRms) return NGR_ERR_ARG;
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (M < 0 || K <= 0 || N <= 0 || M >= kMaxDim || K >= kMaxDim || N >= kMaxDim)
        return NGR_ERR_SHAPE;
    if (M == 0) return NGR_OK;
    if (!x || !Wf || !cb || !y) return NGR_ERR_NULL;
    if (!ws) return NGR_ERR_WORKSPACE;
    // Wf and cb come from ngr_fold_prepare: [N, K8] rows and [2, N8].  x and y
    // go through zero-padded copies when K or N is not a multiple of 8.
    const bool pad = K % 8 != 0 || N % 8 != 0;
    if (!aligned16(Wf) || !aligned16(cb)) return NGR_ERR_ALIGN;
    if (pad ? (!aligned2(x) || !aligned2(y)) : (!aligned16(x) || !aligned16(y)))
        return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    const WsLayout L = ws_layout(norm == kNormLayer ? NGR_OP_LAYERNORM_LINEAR : NGR_OP_RMSNORM_LINEAR,
                                 M, K, N, false);
    if (ws_bytes < L.total) return NGR_ERR_WORKSPACE;
    DevInfo di;
    int rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool bf16 = dtype == NGR_BF16;
    char *w = static_cast<char *>(ws);
    if (debug_mode() && cudaMemsetAsync(w, 0, 4, stream) != cudaSuccess) return NGR_ERR_CUDA;
    const int64_t K8 = round8(K), N8 = round8(N);
    const void *xa = x;
    void *ya = y;
    if (pad) {
        if (K8 != K || !aligned16(x)) {
            rc = launch_pad_rows(x, M, K, K, w + L.xp, K8, di.sms, stream);
            if (rc != 0) return rc;
            xa = w + L.xp;
        }
        if (N8 != N || !aligned16(y)) ya = w + L.yp;
    }
    const bool decode = M <= kDecodeMaxM;
    // The statistics kernel, first on the stream, zeroes the K-split counters.
    events_reset();
    event_before(stream);
    rc = launch_rowstats(norm, bf16, xa, M, K8, eps, reinterpret_cast<float2 *>(w + L.stats), nullptr,
                         nullptr, nullptr, nullptr,
                         decode ? reinterpret_cast<int *>(w + L.counters)
                                : (L.split_cnt_bytes != 0 ? reinterpret_cast<int *>(w + L.split_cnt) : nullptr),
                         decode ? static_cast<int>(ceil_div(N8, 128) * 4) : static_cast<int>(L.split_cnt_bytes / 4),
                         reinterpret_cast<int *>(w), di.sms, stream, nullptr, K);
    event_after(stream);
    if (rc != NGR_OK) return rc;
    event_before(stream);
    rc = launch_layer(norm == kNormLayer ? kNormFoldLayer : kNormFoldRms, kActNone, bf16, xa, Wf,
                      nullptr, M, K8, N8, ya, w, L, L.counters, true, di, stream, cb, cb + N8, N,
                      nullptr, true);
    event_after(stream);
    if (rc == NGR_OK && ya != y) rc = launch_unpad_rows(ya, M, N, N8, y, di.sms, stream);
    events_call_done();
    return finish(rc, ws, stream);
}

// y = act(norm(x) W1^T + b1) W2^T + b2 (the FFN is norm none, SiLU, no
// biases): statistics (and, at decode sizes, the normalized rows and zeroed
// split-K counters), then two GEMMs, the second a programmatic dependent of
// the first; H [M, F] is written once and read once.
int mlp_chain(int op, int norm, int act, const void *x, const void *gamma, const void *beta,
              const void *W1, const void *b1, const void *W2, const void *b2, float eps,
              int64_t M, int64_t K, int64_t F, int dtype, void *h, void *y, void *ws,
              size_t ws_bytes, cudaStream_t stream, int64_t k_valid = -1)
{
    int rc = check_sizes(M, K, F, dtype);
    if (rc != NGR_OK) return rc;
    if (M == 0) return NGR_OK;
    if (!x || !W1 || !W2 || !y) return NGR_ERR_NULL;
    if (norm != kNormNone && !gamma) return NGR_ERR_NULL;
    if (norm == kNormLayer && !beta) return NGR_ERR_NULL;
    if (!ws) return NGR_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(y) ||
        (h && !aligned16(h)) || (gamma && !aligned16(gamma)) || (beta && !aligned16(beta)) ||
        (b1 && !aligned16(b1)) || (b2 && !aligned16(b2)))
        return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    const WsLayout L = ws_layout(op, M, K, F, h == nullptr);
    if (ws_bytes < L.total) return NGR_ERR_WORKSPACE;
    DevInfo di;
    rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool bf16 = dtype == NGR_BF16;
    char *w = static_cast<char *>(ws);
    void *H = h ? h : static_cast<void *>(w + L.h);
    if (debug_mode() && cudaMemsetAsync(w, 0, 4, stream) != cudaSuccess) return NGR_ERR_CUDA;
    const bool decode = M <= kDecodeMaxM;
    const bool need_stats = norm != kNormNone || decode;
    if (product_splits(kNormNone, M, F, K, L, di)) {   // the second product
        rc = zero_split_counters(L, w, stream);
        if (rc != NGR_OK) return rc;
    }
    events_reset();
    if (need_stats) {
        event_before(stream);
        // Both GEMMs' split-K counters (adjacent) are zeroed here.
        const int n_counters =
            decode ? static_cast<int>((L.counters2 - L.counters) / 4 + ceil_div(K, 128) * 4) : 0;
        rc = launch_rowstats(norm == kNormNone ? kNormRms : norm, bf16, x,
                             norm == kNormNone ? 0 : M, K, eps,
                             norm == kNormNone ? nullptr : reinterpret_cast<float2 *>(w + L.stats),
                             gamma, beta,
                             norm == kNormNone ? nullptr : reinterpret_cast<float *>(w + L.gamma_f),
                             norm == kNormNone ? nullptr : reinterpret_cast<float *>(w + L.beta_f),
                             decode ? reinterpret_cast<int *>(w + L.counters) : nullptr, n_counters,
                             reinterpret_cast<int *>(w), di.sms, stream, nullptr, k_valid);
        event_after(stream);
        if (rc != NGR_OK) return rc;
    }
    event_before(stream);
    rc = launch_layer(norm, act, bf16, x, W1, b1, M, K, F, H, w, L, L.counters, need_stats, di,
                      stream);
    event_after(stream);
    if (rc != NGR_OK) return rc;
    event_before(stream);
    rc = launch_layer(kNormNone, kActNone, bf16, H, W2, b2, M, F, K, y, w, L, L.counters2, true, di,
                      stream, nullptr, nullptr, -1, nullptr, true);
    event_after(stream);
    events_call_done();
    return finish(rc, ws, stream);
}

// SwiGLU h = SiLU(norm(x) Wg^T) * (norm(x) Wu^T) (gated CTA-pair kernel),
// and with Wd the Llama MLP y = h Wd^T (a second, plain GEMM).
int swiglu_chain(int op, int norm, const void *x, const void *gamma, const void *beta,
                 const void *Wg, const void *Wu, const void *Wd, float eps, int64_t M, int64_t K,
                 int64_t F, int dtype, void *h, void *y, void *ws, size_t ws_bytes,
                 cudaStream_t stream, int64_t k_valid = -1)
{
    const bool down = op == NGR_OP_MLP_SWIGLU;
    int rc = check_sizes(M, K, F, dtype);
    if (rc != NGR_OK) return rc;
    if (M == 0) return NGR_OK;
    if (!x || !Wg || !Wu || (down ? (!Wd || !y) : !h)) return NGR_ERR_NULL;
    if (norm != kNormNone && !gamma) return NGR_ERR_NULL;
    if (norm == kNormLayer && !beta) return NGR_ERR_NULL;
    if (!ws) return NGR_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(Wg) || !aligned16(Wu) || (Wd && !aligned16(Wd)) ||
        (y && !aligned16(y)) || (h && !aligned16(h)) || (gamma && !aligned16(gamma)) ||
        (beta && !aligned16(beta)))
        return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    const WsLayout L = ws_layout(op, M, K, F, down && h == nullptr);
    if (ws_bytes < L.total) return NGR_ERR_WORKSPACE;
    DevInfo di;
    rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool bf16 = dtype == NGR_BF16;
    char *w = static_cast<char *>(ws);
    void *H = h ? h : static_cast<void *>(w + L.h);
    if (debug_mode() && cudaMemsetAsync(w, 0, 4, stream) != cudaSuccess) return NGR_ERR_CUDA;
    const bool decode = M <= kDecodeMaxM;
    const bool need_stats = norm != kNormNone || (down && decode);
    if (down && product_splits(kNormNone, M, F, K, L, di)) {   // the down projection
        rc = zero_split_counters(L, w, stream);
        if (rc != NGR_OK) return rc;
    }
    events_reset();
    if (need_stats) {
        event_before(stream);
        rc = launch_rowstats(norm == kNormNone ? kNormRms : norm, bf16, x,
                             norm == kNormNone ? 0 : M, K, eps,
                             norm == kNormNone ? nullptr : reinterpret_cast<float2 *>(w + L.stats),
                             gamma, beta,
                             norm == kNormNone ? nullptr : reinterpret_cast<float *>(w + L.gamma_f),
                             norm == kNormNone ? nullptr : reinterpret_cast<float *>(w + L.beta_f),
                             down && decode ? reinterpret_cast<int *>(w + L.counters2) : nullptr,
                             down && decode ? static_cast<int>(ceil_div(K, 128) * 4) : 0,
                             reinterpret_cast<int *>(w), di.sms, stream, nullptr, k_valid);
        event_after(stream);
        if (rc != NGR_OK) return rc;
    }
    event_before(stream);
    rc = launch_gated(norm, bf16, x, Wg, Wu, M, K, F, H, w, L, need_stats, di, stream);
    event_after(stream);
    if (rc != NGR_OK) return rc;
    if (down) {
        event_before(stream);
        rc = launch_layer(kNormNone, kActNone, bf16, H, Wd, nullptr, M, F, K, y, w, L, L.counters2,
                          true, di, stream, nullptr, nullptr, -1, nullptr, true);
        event_after(stream);
    }
    events_call_done();
    return finish(rc, ws, stream);
}

// h = x W^T + bias (+ residual), written once; y = norm(h) over its N
// columns: the product's epilogue adds the bias and the residual, then the
// statistics kernel reads each h row once, computes its statistics and
// writes the normalized row (gamma, beta of length N).
int linear_residual_norm(int norm, const void *x, const void *W, const void *bias,
                         const void *residual, const void *gamma, const void *beta, float eps,
                         int64_t M, int64_t K, int64_t N, int dtype, void *h, void *y, void *ws,
                         size_t ws_bytes, cudaStream_t stream, int64_t n_valid = -1)
{
    if (norm != kNormLayer && norm != kNormRms) return NGR_ERR_ARG;
    int rc = check_sizes(M, K, N, dtype);
    if (rc != NGR_OK) return rc;
    if (M == 0) return NGR_OK;
    if (!x || !W || !gamma || !y || (norm == kNormLayer && !beta)) return NGR_ERR_NULL;
    if (!ws) return NGR_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(W) || !aligned16(gamma) || !aligned16(y) ||
        (beta && !aligned16(beta)) || (bias && !aligned16(bias)) ||
        (residual && !aligned16(residual)) || (h && !aligned16(h)))
        return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    const WsLayout L = ws_layout(NGR_OP_LINEAR_RESIDUAL_NORM, M, K, N, h == nullptr);
    if (ws_bytes < L.total) return NGR_ERR_WORKSPACE;
    DevInfo di;
    rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool bf16 = dtype == NGR_BF16;
    char *w = static_cast<char *>(ws);
    void *H = h ? h : static_cast<void *>(w + L.h);
    if (debug_mode() && cudaMemsetAsync(w, 0, 4, stream) != cudaSuccess) return NGR_ERR_CUDA;
    const bool decode = M <= kDecodeMaxM;
    if (product_splits(kNormNone, M, K, N, L, di)) {
        rc = zero_split_counters(L, w, stream);
        if (rc != NGR_OK) return rc;
    }
    events_reset();
    if (decode) {
        // the decode product's split-K counters start from zero
        event_before(stream);
        rc = launch_rowstats(kNormRms, bf16, x, 0, K, 0.f, nullptr, nullptr, nullptr, nullptr,
                             nullptr, reinterpret_cast<int *>(w + L.counters),
                             static_cast<int>(ceil_div(N, 128) * 4), reinterpret_cast<int *>(w),
                             di.sms, stream);
        event_after(stream);
        if (rc != NGR_OK) return rc;
    }
    event_before(stream);
    rc = launch_layer(kNormNone, kActNone, bf16, x, W, bias, M, K, N, H, w, L, L.counters, decode,
                      di, stream, nullptr, nullptr, -1, residual, true);
    event_after(stream);
    if (rc != NGR_OK) return rc;
    // The norm over each h row, launched as a programmatic dependent of the
    // product: its CTAs take the SMs the product leaves and wait for the
    // product's grid before reading h.
    event_before(stream);
    rc = launch_rowstats(norm, bf16, H, M, N, eps, reinterpret_cast<float2 *>(w + L.stats), gamma,
                         beta, nullptr, nullptr, nullptr, 0, nullptr, di.sms, stream, y, n_valid, true);
    event_after(stream);
    events_call_done();
    return finish(rc, ws, stream);
}

// ---------------------------------------------- any K and N for the chains
// The chains, SwiGLU and the post-GEMM norm take any K and N (F) the same
// way the single layer does ("昇腾CANN的MatMul融合玩法，让大模型推理快3倍",
// §五 optimization 1): every operand is copied into rows padded with zeros
// to a multiple of 8 elements (weights also get zero rows up to a multiple
// of 8), the aligned implementation runs on the padded problem with its
// statistics counting only the real columns, and the real columns of the
// outputs are copied back.  Zero weight rows and zero biases make the padded
// hidden units act(0) = 0 (SiLU, ReLU, GELU and SiLU-gating all map 0 to
// 0), and their zero weight columns in the next product add nothing.  The
// copies follow the aligned implementation's own workspace regions.

bool chain_op(int op)
{
    return op == NGR_OP_FFN || op == NGR_OP_MLP || op == NGR_OP_SWIGLU ||
           op == NGR_OP_MLP_SWIGLU || op == NGR_OP_LINEAR_RESIDUAL_NORM;
}

bool needs_pad(int op, int64_t K, int64_t N)
{
    return chain_op(op) && (K % 8 != 0 || N % 8 != 0);
}

// The padded copies of a chain op, in workspace order (each 256-byte
// aligned), after ws_layout(op, M, K8, N8, h_in_ws).
struct PadRegions {
    size_t x = 0, g = 0, b = 0, w1 = 0, b1 = 0, w2 = 0, b2 = 0, w3 = 0, res = 0, h = 0, y = 0;
    size_t total = 0;
};

PadRegions pad_regions(int op, int64_t M, int64_t K, int64_t N, bool h_in_ws, size_t base)
{
    PadRegions R;
    const size_t K8 = static_cast<size_t>(round8(K)), N8 = static_cast<size_t>(round8(N));
    const size_t m = static_cast<size_t>(M);
    size_t off = base;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    const bool post = op == NGR_OP_LINEAR_RESIDUAL_NORM;
    R.x = take(m * K8 * 2);
    if (post) {
        R.w1 = take(N8 * K8 * 2);   // W
        R.b1 = take(N8 * 2);        // bias
        R.res = take(m * N8 * 2);   // residual
        R.g = take(N8 * 2);
        R.b = take(N8 * 2);
        R.y = take(m * N8 * 2);
        if (!h_in_ws) R.h = take(m * N8 * 2);
    } else {
        R.g = take(K8 * 2);
        R.b = take(K8 * 2);
        R.w1 = take(N8 * K8 * 2);   // W1 or W_gate
        if (op == NGR_OP_SWIGLU || op == NGR_OP_MLP_SWIGLU) {
            R.w3 = take(N8 * K8 * 2);   // W_up
        } else {
            R.b1 = take(N8 * 2);
            R.b2 = take(K8 * 2);
        }
        if (op != NGR_OP_SWIGLU) {
            R.w2 = take(K8 * N8 * 2);   // W2 or W_down
            R.y = take(m * K8 * 2);
        }
        if (op == NGR_OP_SWIGLU || !h_in_ws) R.h = take(m * N8 * 2);
    }
    R.total = off;
    return R;
}

// Workspace bytes of any op at any K and N.
size_t ws_total(int op, int64_t M, int64_t K, int64_t N, bool h_in_ws)
{
    if (!needs_pad(op, K, N)) return ws_layout(op, M, K, N, h_in_ws).total;
    const size_t inner = ws_layout(op, M, round8(K), round8(N), h_in_ws).total;
    return pad_regions(op, M, K, N, h_in_ws, inner).total;
}

// Checks shared by the padded wrappers: sizes, dtype, 2-byte pointers,
// the workspace; fills *inner and *R.
int pad_prologue(int op, int64_t M, int64_t K, int64_t N, int dtype, bool h_in_ws, void *ws,
                 size_t ws_bytes, std::initializer_list<const void *> ptrs, size_t *inner,
                 PadRegions *R, DevInfo *di)
{
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (M < 0 || K <= 0 || N <= 0 || M >= kMaxDim || K >= kMaxDim || N >= kMaxDim)
        return NGR_ERR_SHAPE;
    if (!ws) return NGR_ERR_WORKSPACE;
    for (const void *p : ptrs)
        if (p && !aligned2(p)) return NGR_ERR_ALIGN;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return NGR_ERR_ALIGN;
    *inner = ws_layout(op, M, round8(K), round8(N), h_in_ws).total;
    *R = pad_regions(op, M, K, N, h_in_ws, *inner);
    if (ws_bytes < R->total) return NGR_ERR_WORKSPACE;
    return current_device_info(di);
}

// Copy a [rows, cols] operand (nullptr stays nullptr) into the workspace at
// `off` as [rows8, round8(cols)] with zero padding.
int pad_in(const void *src, int64_t rows, int64_t cols, int64_t rows8, char *ws, size_t off,
           const void **out, const DevInfo &di, cudaStream_t stream)
{
    if (!src) {
        *out = nullptr;
        return NGR_OK;
    }
    *out = ws + off;
    return launch_pad_rows(src, rows, cols, cols, ws + off, round8(cols), di.sms, stream, rows8);
}

int mlp_chain_any(int op, int norm, int act, const void *x, const void *gamma, const void *beta,
                  const void *W1, const void *b1, const void *W2, const void *b2, float eps,
                  int64_t M, int64_t K, int64_t F, int dtype, void *h, void *y, void *ws,
                  size_t ws_bytes, cudaStream_t stream)
{
    if (!needs_pad(op, K, F))
        return mlp_chain(op, norm, act, x, gamma, beta, W1, b1, W2, b2, eps, M, K, F, dtype, h, y,
                         ws, ws_bytes, stream);
    if (!x || !W1 || !W2 || !y) return NGR_ERR_NULL;
    if (norm != kNormNone && !gamma) return NGR_ERR_NULL;
    if (norm == kNormLayer && !beta) return NGR_ERR_NULL;
    size_t inner = 0;
    PadRegions R;
    DevInfo di;
    int rc = pad_prologue(op, M, K, F, dtype, h == nullptr, ws, ws_bytes,
                          {x, gamma, beta, W1, b1, W2, b2, h, y}, &inner, &R, &di);
    if (rc != NGR_OK || M == 0) return rc;
    char *w = static_cast<char *>(ws);
    const int64_t K8 = round8(K), F8 = round8(F);
    const void *xp, *gp, *bp, *W1p, *b1p, *W2p, *b2p;
    rc = pad_in(x, M, K, M, w, R.x, &xp, di, stream);
    if (rc == NGR_OK) rc = pad_in(gamma, 1, K, 1, w, R.g, &gp, di, stream);
    if (rc == NGR_OK) rc = pad_in(beta, 1, K, 1, w, R.b, &bp, di, stream);
    if (rc == NGR_OK) rc = pad_in(W1, F, K, F8, w, R.w1, &W1p, di, stream);
    if (rc == NGR_OK) rc = pad_in(b1, 1, F, 1, w, R.b1, &b1p, di, stream);
    if (rc == NGR_OK) rc = pad_in(W2, K, F, K8, w, R.w2, &W2p, di, stream);
    if (rc == NGR_OK) rc = pad_in(b2, 1, K, 1, w, R.b2, &b2p, di, stream);
    if (rc != NGR_OK) return rc;
    void *Hp = h ? static_cast<void *>(w + R.h) : nullptr;
    rc = mlp_chain(op, norm, act, xp, gp, bp, W1p, b1p, W2p, b2p, eps, M, K8, F8, dtype, Hp,
                   w + R.y, ws, inner, stream, K);
    if (rc == NGR_OK) rc = launch_unpad_rows(w + R.y, M, K, K8, y, di.sms, stream);
    if (rc == NGR_OK && h) rc = launch_unpad_rows(Hp, M, F, F8, h, di.sms, stream);
    return rc;
}

int swiglu_chain_any(int op, int norm, const void *x, const void *gamma, const void *beta,
                     const void *Wg, const void *Wu, const void *Wd, float eps, int64_t M,
                     int64_t K, int64_t F, int dtype, void *h, void *y, void *ws,
                     size_t ws_bytes, cudaStream_t stream)
{
    const bool down = op == NGR_OP_MLP_SWIGLU;
    if (!needs_pad(op, K, F))
        return swiglu_chain(op, norm, x, gamma, beta, Wg, Wu, Wd, eps, M, K, F, dtype, h, y, ws,
                            ws_bytes, stream);
    if (!x || !Wg || !Wu || (down ? (!Wd || !y) : !h)) return NGR_ERR_NULL;
    if (norm != kNormNone && !gamma) return NGR_ERR_NULL;
    if (norm == kNormLayer && !beta) return NGR_ERR_NULL;
    const bool h_in_ws = down && h == nullptr;
    size_t inner = 0;
    PadRegions R;
    DevInfo di;
    int rc = pad_prologue(op, M, K, F, dtype, h_in_ws, ws, ws_bytes,
                          {x, gamma, beta, Wg, Wu, Wd, h, y}, &inner, &R, &di);
    if (rc != NGR_OK || M == 0) return rc;
    char *w = static_cast<char *>(ws);
    const int64_t K8 = round8(K), F8 = round8(F);
    const void *xp, *gp, *bp, *Wgp, *Wup, *Wdp = nullptr;
    rc = pad_in(x, M, K, M, w, R.x, &xp, di, stream);
    if (rc == NGR_OK) rc = pad_in(gamma, 1, K, 1, w, R.g, &gp, di, stream);
    if (rc == NGR_OK) rc = pad_in(beta, 1, K, 1, w, R.b, &bp, di, stream);
    if (rc == NGR_OK) rc = pad_in(Wg, F, K, F8, w, R.w1, &Wgp, di, stream);
    if (rc == NGR_OK) rc = pad_in(Wu, F, K, F8, w, R.w3, &Wup, di, stream);
    if (rc == NGR_OK && down) rc = pad_in(Wd, K, F, K8, w, R.w2, &Wdp, di, stream);
    if (rc != NGR_OK) return rc;
    void *Hp = h ? static_cast<void *>(w + R.h) : nullptr;
    rc = swiglu_chain(op, norm, xp, gp, bp, Wgp, Wup, Wdp, eps, M, K8, F8, dtype, Hp,
                      down ? w + R.y : nullptr, ws, inner, stream, K);
    if (rc == NGR_OK && down) rc = launch_unpad_rows(w + R.y, M, K, K8, y, di.sms, stream);
    if (rc == NGR_OK && h) rc = launch_unpad_rows(Hp, M, F, F8, h, di.sms, stream);
    return rc;
}

int linear_residual_norm_any(int norm, const void *x, const void *W, const void *bias,
                             const void *residual, const void *gamma, const void *beta, float eps,
                             int64_t M, int64_t K, int64_t N, int dtype, void *h, void *y,
                             void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const int op = NGR_OP_LINEAR_RESIDUAL_NORM;
    if (!needs_pad(op, K, N))
        return linear_residual_norm(norm, x, W, bias, residual, gamma, beta, eps, M, K, N, dtype,
                                    h, y, ws, ws_bytes, stream);
    if (norm != kNormLayer && norm != kNormRms) return NGR_ERR_ARG;
    if (!x || !W || !gamma || !y || (norm == kNormLayer && !beta)) return NGR_ERR_NULL;
    size_t inner = 0;
    PadRegions R;
    DevInfo di;
    int rc = pad_prologue(op, M, K, N, dtype, h == nullptr, ws, ws_bytes,
                          {x, W, bias, residual, gamma, beta, h, y}, &inner, &R, &di);
    if (rc != NGR_OK || M == 0) return rc;
    char *w = static_cast<char *>(ws);
    const int64_t N8 = round8(N);
    const void *xp, *Wp, *biasp, *resp, *gp, *bp;
    rc = pad_in(x, M, K, M, w, R.x, &xp, di, stream);
    if (rc == NGR_OK) rc = pad_in(W, N, K, N8, w, R.w1, &Wp, di, stream);
    if (rc == NGR_OK) rc = pad_in(bias, 1, N, 1, w, R.b1, &biasp, di, stream);
    if (rc == NGR_OK) rc = pad_in(residual, M, N, M, w, R.res, &resp, di, stream);
    if (rc == NGR_OK) rc = pad_in(gamma, 1, N, 1, w, R.g, &gp, di, stream);
    if (rc == NGR_OK) rc = pad_in(beta, 1, N, 1, w, R.b, &bp, di, stream);
    if (rc != NGR_OK) return rc;
    void *Hp = h ? static_cast<void *>(w + R.h) : nullptr;
    rc = linear_residual_norm(norm, xp, Wp, biasp, resp, gp, bp, eps, M, round8(K), N8, dtype, Hp,
                              w + R.y, ws, inner, stream, N);
    if (rc == NGR_OK) rc = launch_unpad_rows(w + R.y, M, N, N8, y, di.sms, stream);
    if (rc == NGR_OK && h) rc = launch_unpad_rows(Hp, M, N, N8, h, di.sms, stream);
    return rc;
}

__global__ void bounded_wait_probe_kernel(int *err, unsigned long long timeout_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // Nothing ever arrives on `bar`: the wait must run out and record it.
    const WaitCtx wc{&abort_flag, err, timeout_ns};
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, wc);
    __syncthreads();
}

}  // namespace

int launch_bounded_wait_probe(int *err, unsigned long long timeout_ns, cudaStream_t stream)
{
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -7;
}

}  // namespace ngr

using namespace ngr;

extern "C" {

size_t ngr_workspace_bytes(int op, int64_t M, int64_t K, int64_t N, int ffn_h_in_workspace)
{
    if (op < NGR_OP_LAYERNORM_LINEAR || op > NGR_OP_LINEAR_RESIDUAL_NORM) return 0;
    if (M < 0 || K <= 0 || N <= 0 || M >= kMaxDim || K >= kMaxDim || N >= kMaxDim) return 0;
    return ws_total(op, M, K, N, ffn_h_in_workspace != 0);
}

int ngr_fused_layernorm_linear(const void *x, const void *gamma, const void *beta, const void *W,
                               const void *bias, float eps, int64_t M, int64_t K, int64_t N,
                               int dtype, void *y, void *workspace, size_t workspace_bytes,
                               ngr_stream_t stream)
{
    return norm_linear(NGR_OP_LAYERNORM_LINEAR, kNormLayer, kActNone, x, gamma, beta, W, bias, eps,
                       M, K, N, dtype, y, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_rmsnorm_linear(const void *x, const void *gamma, const void *W, const void *bias,
                             float eps, int64_t M, int64_t K, int64_t N, int dtype, void *y,
                             void *workspace, size_t workspace_bytes, ngr_stream_t stream)
{
    return norm_linear(NGR_OP_RMSNORM_LINEAR, kNormRms, kActNone, x, gamma, nullptr, W, bias, eps, M,
                       K, N, dtype, y, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_linear_silu(const void *x, const void *W, const void *bias, int64_t M, int64_t K,
                          int64_t N, int dtype, void *y, void *workspace, size_t workspace_bytes,
                          ngr_stream_t stream)
{
    return norm_linear(NGR_OP_LINEAR_SILU, kNormNone, kActSilu, x, nullptr, nullptr, W, bias, 0.f, M,
                       K, N, dtype, y, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int ngr_ffn_linear_silu_linear(const void *x, const void *W1, const void *W2, int64_t M,
                               int64_t K, int64_t F, int dtype, void *h, void *y, void *workspace,
                               size_t workspace_bytes, ngr_stream_t stream)
{
    return mlp_chain_any(NGR_OP_FFN, kNormNone, kActSilu, x, nullptr, nullptr, W1, nullptr, W2,
                         nullptr, 0.f, M, K, F, dtype, h, y, workspace, workspace_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_norm_linear_act(int norm, int act, const void *x, const void *gamma,
                              const void *beta, const void *W, const void *bias, float eps,
                              int64_t M, int64_t K, int64_t N, int dtype, void *y,
                              void *workspace, size_t workspace_bytes, ngr_stream_t stream)
{
    if (norm < kNormNone || norm > kNormRms || act < kActNone || act > kActGelu)
        return NGR_ERR_ARG;
    return norm_linear(NGR_OP_NORM_LINEAR, norm, act, x, gamma, norm == kNormLayer ? beta : nullptr,
                       W, bias, eps, M, K, N, dtype, y, workspace, workspace_bytes,
                       reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_mlp(int norm, int act, const void *x, const void *gamma, const void *beta,
                  const void *W1, const void *b1, const void *W2, const void *b2, float eps,
                  int64_t M, int64_t K, int64_t F, int dtype, void *h, void *y, void *workspace,
                  size_t workspace_bytes, ngr_stream_t stream)
{
    if (norm < kNormNone || norm > kNormRms || act < kActNone || act > kActGelu)
        return NGR_ERR_ARG;
    return mlp_chain_any(NGR_OP_MLP, norm, act, x, gamma, norm == kNormLayer ? beta : nullptr, W1,
                         b1, W2, b2, eps, M, K, F, dtype, h, y, workspace, workspace_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_norm_swiglu(int norm, const void *x, const void *gamma, const void *beta,
                          const void *Wg, const void *Wu, float eps, int64_t M, int64_t K,
                          int64_t F, int dtype, void *h, void *workspace, size_t workspace_bytes,
                          ngr_stream_t stream)
{
    if (norm < kNormNone || norm > kNormRms) return NGR_ERR_ARG;
    return swiglu_chain_any(NGR_OP_SWIGLU, norm, x, gamma, norm == kNormLayer ? beta : nullptr, Wg,
                            Wu, nullptr, eps, M, K, F, dtype, h, nullptr, workspace,
                            workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_mlp_swiglu(int norm, const void *x, const void *gamma, const void *beta,
                         const void *Wg, const void *Wu, const void *Wd, float eps, int64_t M,
                         int64_t K, int64_t F, int dtype, void *h, void *y, void *workspace,
                         size_t workspace_bytes, ngr_stream_t stream)
{
    if (norm < kNormNone || norm > kNormRms) return NGR_ERR_ARG;
    return swiglu_chain_any(NGR_OP_MLP_SWIGLU, norm, x, gamma, norm == kNormLayer ? beta : nullptr,
                            Wg, Wu, Wd, eps, M, K, F, dtype, h, y, workspace, workspace_bytes,
                            reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fused_linear_residual_norm(int norm, const void *x, const void *W, const void *bias,
                                   const void *residual, const void *gamma, const void *beta,
                                   float eps, int64_t M, int64_t K, int64_t N, int dtype,
                                   void *h, void *y, void *workspace, size_t workspace_bytes,
                                   ngr_stream_t stream)
{
    return linear_residual_norm_any(norm, x, W, bias, residual, gamma,
                                    norm == kNormLayer ? beta : nullptr, eps, M, K, N, dtype, h, y,
                                    workspace, workspace_bytes,
                                    reinterpret_cast<cudaStream_t>(stream));
}

int ngr_fold_prepare(int norm, const void *gamma, const void *beta, const void *W,
                     const void *bias, int64_t K, int64_t N, int dtype, void *Wf, float *cb,
                     ngr_stream_t stream)
{
    if (norm != kNormLayer && norm != kNormRms) return NGR_ERR_ARG;
    if (dtype != NGR_F16 && dtype != NGR_BF16) return NGR_ERR_DTYPE;
    if (K <= 0 || N <= 0 || K >= kMaxDim || N >= kMaxDim) return NGR_ERR_SHAPE;
    int rc = NGR_OK;
    if (!gamma || !W || !Wf || !cb || (norm == kNormLayer && !beta)) return NGR_ERR_NULL;
    if (norm == kNormRms) beta = nullptr;
    const bool aligned = K % 8 == 0 && N % 8 == 0 && aligned16(gamma) && aligned16(W) &&
                         (!beta || aligned16(beta)) && (!bias || aligned16(bias));
    if (!aligned16(Wf) || !aligned16(cb) || !aligned2(gamma) || !aligned2(W) ||
        (beta && !aligned2(beta)) || (bias && !aligned2(bias)))
        return NGR_ERR_ALIGN;
    DevInfo di;
    rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    auto launch = aligned ? launch_fold_prepare : launch_fold_prepare_any;
    rc = launch(norm, dtype == NGR_BF16, gamma, beta, W, bias, K, N, Wf, cb, di.sms,
                reinterpret_cast<cudaStream_t>(stream));
    return rc == 0 ? NGR_OK : rc;
}

int ngr_fused_norm_linear_folded(int norm, const void *x, const void *Wf, const float *cb,
                                 float eps, int64_t M, int64_t K, int64_t N, int dtype, void *y,
                                 void *workspace, size_t workspace_bytes, ngr_stream_t stream)
{
    return folded_linear(norm, x, Wf, cb, eps, M, K, N, dtype, y, workspace, workspace_bytes,
                         reinterpret_cast<cudaStream_t>(stream));
}

int ngr_row_stats(int norm, const void *x, float eps, int64_t M, int64_t K, int dtype,
                  float *stats, ngr_stream_t stream)
{
    if (norm != kNormLayer && norm != kNormRms) return NGR_ERR_ARG;
    int rc = check_sizes(M, K, 8, dtype);
    if (rc != NGR_OK) return rc;
    if (M == 0) return NGR_OK;
    if (!x || !stats) return NGR_ERR_NULL;
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(stats) & 7u) != 0) return NGR_ERR_ALIGN;
    DevInfo di;
    rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    rc = launch_rowstats(norm, dtype == NGR_BF16, x, M, K, eps, reinterpret_cast<float2 *>(stats),
                         nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, di.sms,
                         reinterpret_cast<cudaStream_t>(stream));
    if (rc != NGR_OK) return rc;
    return cudaGetLastError() == cudaSuccess ? NGR_OK : NGR_ERR_CUDA;
}

int ngr_workspace_error(void *workspace, ngr_stream_t stream)
{
    if (!workspace) return NGR_ERR_WORKSPACE;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NGR_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return NGR_ERR_CUDA;
    if (v != 0 && cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return NGR_ERR_CUDA;
    return v == 0 ? NGR_OK : NGR_ERR_TIMEOUT;
}

int ngr_debug_bounded_wait(void *workspace, uint32_t timeout_us, ngr_stream_t stream_)
{
    if (!workspace) return NGR_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return NGR_ERR_ALIGN;
    DevInfo di;
    int rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess) return NGR_ERR_CUDA;
    rc = launch_bounded_wait_probe(static_cast<int *>(workspace),
                                   static_cast<unsigned long long>(timeout_us) * 1000ull, stream);
    return rc == 0 ? NGR_OK : NGR_ERR_CUDA;
}

int ngr_tile_plan(int op, int64_t M, int64_t K, int64_t N, int *plan)
{
    if (!plan) return NGR_ERR_NULL;
    if (op < NGR_OP_LAYERNORM_LINEAR || op > NGR_OP_LINEAR_RESIDUAL_NORM ||
        op == NGR_OP_SWIGLU || M <= kDecodeMaxM || K <= 0 || N <= 0)
        return NGR_ERR_ARG;
    DevInfo di;
    const int rc = current_device_info(&di);
    if (rc != NGR_OK) return rc;
    const bool chain = op == NGR_OP_FFN || op == NGR_OP_MLP || op == NGR_OP_MLP_SWIGLU;
    const WsLayout L = ws_layout(op, M, K, N, false);
    const int64_t n_out = chain ? K : (L.padded ? round8(N) : N);
    const int64_t k_in = chain ? N : (L.padded ? round8(K) : K);
    // the products with a norm on their input: the single layers' (the
    // general layer's taken as normalized); the chains' second product and
    // the post-norm op's product have none
    const bool in_norm = op == NGR_OP_LAYERNORM_LINEAR || op == NGR_OP_RMSNORM_LINEAR ||
                         op == NGR_OP_NORM_LINEAR;
    const GemmPlan p = plan_gemm(M, n_out, k_in, di.sms, in_norm, L.split_cnt_bytes + L.split_part_bytes,
                                 !in_norm);
    plan[0] = p.mc ? 2 : (p.pair ? 1 : 0);
    plan[1] = p.bn;
    plan[2] = p.nsub;
    plan[3] = p.splits > 1 ? p.splits : 1;
    plan[4] = p.grid;
    plan[5] = p.stages;
    return NGR_OK;
}

int ngr_set_tile_config(int pair, int bn, int nsub)
{
    return set_tile_config(pair, bn, nsub) == 0 ? NGR_OK : NGR_ERR_ARG;
}

int ngr_kernel_timing_start(int n_calls)
{
    if (n_calls <= 0) return NGR_ERR_ARG;
    const size_t need = static_cast<size_t>(n_calls) * kSlots * 2;
    while (t_events.size() < need) {
        cudaEvent_t e;
        const cudaError_t err = cudaEventCreate(&e);
        if (err != cudaSuccess) return record_cuda_error("cudaEventCreate", err, cudaGetErrorString(err));
        t_events.push_back(e);
    }
    t_count.assign(static_cast<size_t>(n_calls), 0);
    t_calls = n_calls;
    t_call = 0;
    t_kernel = 0;
    t_armed = true;
    return NGR_OK;
}

int ngr_kernel_timing_stop(float *ms, int capacity)
{
    if (!t_armed) return 0;
    t_armed = false;
    int written = 0;
    for (int c = 0; c < t_call; ++c) {
        if (ms && (c + 1) * kSlots > capacity) break;
        for (int k = 0; k < kSlots; ++k) {
            float v = -1.f;
            if (k < t_count[c]) {
                cudaEvent_t b = t_events[2 * (c * kSlots + k)];
                cudaEvent_t e = t_events[2 * (c * kSlots + k) + 1];
                cudaError_t err = cudaEventSynchronize(e);
                if (err == cudaSuccess) err = cudaEventElapsedTime(&v, b, e);
                if (err != cudaSuccess)
                    return record_cuda_error("kernel timing", err, cudaGetErrorString(err));
            }
            if (ms) ms[c * kSlots + k] = v;
        }
        ++written;
    }
    return written;
}

const char *ngr_status_string(int status)
{
    switch (status) {
    case NGR_OK: return "NGR_OK";
    case NGR_ERR_NULL: return "NGR_ERR_NULL: a required pointer is NULL";
    case NGR_ERR_SHAPE: return "NGR_ERR_SHAPE: invalid M, K or N";
    case NGR_ERR_ALIGN: return "NGR_ERR_ALIGN: K or N not a multiple of 8, or a misaligned pointer";
    case NGR_ERR_DTYPE: return "NGR_ERR_DTYPE: dtype must be NGR_F16 or NGR_BF16";
    case NGR_ERR_WORKSPACE: return "NGR_ERR_WORKSPACE: workspace missing or too small";
    case NGR_ERR_ARCH: return "NGR_ERR_ARCH: the current device is not sm_103 (GB300)";
    case NGR_ERR_CUDA: return "NGR_ERR_CUDA: a CUDA call failed";
    case NGR_ERR_TIMEOUT: return "NGR_ERR_TIMEOUT: a kernel's bounded wait ran out";
    case NGR_ERR_ARG: return "NGR_ERR_ARG: invalid argument";
    default: return "unknown ngr status";
    }
}

int ngr_version(void) { return 100; }

const char *ngr_last_error(void) { return g_last_error; }

}  // extern "C"
