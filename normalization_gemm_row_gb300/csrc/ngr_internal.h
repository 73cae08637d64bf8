// ngr_internal.h -- declarations shared by the library's translation units
// (kernel launchers, argument blocks, workspace layout).  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace ngr {

enum { kNormNone = 0, kNormLayer = 1, kNormRms = 2, kNormFoldLayer = 3, kNormFoldRms = 4 };

// Epilogue activation, applied after the bias (a runtime argument).
enum { kActNone = 0, kActSilu = 1, kActRelu = 2, kActGelu = 3 };

// Folded (inference-mode) forms: the GEMM runs on raw x against
// W' = gamma o W and the row statistics are applied in the epilogue.
__host__ __device__ constexpr bool is_fold(int norm)
{
    return norm == kNormFoldLayer || norm == kNormFoldRms;
}

// Tile geometry shared by host and device.
constexpr int kBM = 128;        // rows of x per tile (UMMA M)
constexpr int kBK = 64;         // K per pipeline stage: 64 x 2 B = one 128-byte swizzle row
constexpr int kUmmaK = 16;      // K per tcgen05.mma (kind::f16)
// Tile kernel: 16 warps -- producer, MMA, TMEM, spare, 8 transform, 4 epilogue.
constexpr int kGemmThreads = 512;
constexpr int kTransformWarp0 = 4;
constexpr int kTransformThreads = 256;
constexpr int kEpilogueWarp0 = 12;
// The transform warps form groups that take turns on consecutive stages
// (2 groups of 4 warps), or all 8 normalize every stage (1 group).  With
// the transform's waits polling briefly and then sleeping with a time hint,
// two groups measured 4.4 % faster at LayerNorm 1024 x 8192 -> 8192, 2.3 %
// with RMSNorm there and about 1 % at RMSNorm 512 x 14336 -> 49152: while
// one group normalizes a stage the other is already waiting for the next.
// (With polling waits the single group had been 0.5-2 % faster.)
#ifndef NGR_TRANSFORM_GROUPS
#define NGR_TRANSFORM_GROUPS 2
#endif
constexpr int kTransformGroups = NGR_TRANSFORM_GROUPS;
constexpr int kGroupThreads = kTransformThreads / kTransformGroups;
constexpr int kGroupWarps = kGroupThreads / 32;

// Decode (swap-AB) path: weight rows on the UMMA M side, tokens on N.
constexpr int kDecodeMaxM = 32;      // M up to this uses the decode path
constexpr int kDecodeMaxGroups = 8;  // k groups (CTAs sharing one 128-row weight tile)
constexpr int kDecodeThreads = 384;
// k blocks of tokens one decode CTA holds in shared memory (its slice of x):
// 64 KB of [MN x 64] 16-bit boxes beside the weight ring.
__host__ __device__ constexpr int decode_max_kb(int mn) { return (64 * 1024) / (mn * kBK * 2); }

// Arguments of the persistent GEMM kernel (normal orientation: x rows on M).
struct alignas(128) GemmArgs {
    CUtensorMap map_a;      // activations [M, K], box {64, 128}, 128-byte swizzle
    CUtensorMap map_b;      // weights [N, K], box {64, BN}, 128-byte swizzle
    CUtensorMap map_gb;     // FP32 [2, K] = rows gamma, beta; box {64, 2}
    CUtensorMap map_b2;     // gated (SwiGLU) kernel: the up projection [N, K], like map_b
    const float2 *stats;    // [M] (mu, rstd); unused without a norm
    const float *gamma_f;   // [K] FP32 gamma (kernels that read it from global memory)
    const float *beta_f;    // [K] FP32 beta
    const void *bias;       // [N] or nullptr
    const float *fold_c;    // folded forms: c[n] = sum_k W'[n,k] (FP32)
    const float *fold_b;    // folded forms: b'[n] = beta . W[n,:] + bias[n] (FP32)
    const void *residual;   // [M, N] added last, or nullptr
    void *y;                // [M, N]
    int *err;               // device error word
    int zero_err;           // nonzero: this kernel is the call's first and clears *err
    int act;                // kAct*: activation after the bias (not used when gated)
    int M, N, K;
    int m_tiles, n_tiles, k_blocks, num_tiles;
    // Tile kernels (single CTA or CTA pair): K split into k_splits ranges of
    // kb_per_split k blocks (1 = no split).  Each (tile, range) unit writes
    // FP32 partials of its 32 x 32 accumulator chunks; the last of a chunk's
    // units (its counter) sums them in range order and finishes the chunk.
    int k_splits, kb_per_split;
    float *partials;        // [tiles][CTAs per tile][4][chunks][k_splits][32 cols][32 rows]
    int *split_counters;    // [tiles][CTAs per tile][4][chunks], zero at kernel start
    unsigned long long timeout_ns;
};

// Arguments of the decode kernel (swap-AB; CTA (kg, ng) of a k_groups x
// n_groups grid takes k blocks [kg kb_per_group, +kb_per_group) of the
// 128-row weight tiles of n group ng).
struct alignas(128) DecodeArgs {
    CUtensorMap map_w;      // weights [N, K], box {64, 128}, 128-byte swizzle
    CUtensorMap map_x;      // activations [M, K], box {64, MN}, 128-byte swizzle
    const float2 *stats;    // [M] (mu, rstd): a norm or a folded weight
    const float *gamma_f;   // [K] FP32 (a norm)
    const float *beta_f;    // [K] FP32 (LayerNorm)
    const void *bias;
    const float *fold_c;
    const float *fold_b;
    const void *residual;   // [M, N] added last, or nullptr
    void *y;
    float *partials;        // [n_tiles][kDecodeMaxGroups][MN][128] fp32
    int *counters;          // [n_tiles][4], zero at kernel start
    int *err;
    int zero_err;
    int act;                // kAct*
    int M, N, K;
    int n_tiles, k_blocks;
    int k_groups, kb_per_group, n_groups;
    unsigned long long timeout_ns;
};

// The decode grid: k groups of kb_per_group k blocks x n groups of tiles.
struct DecodePlan {
    int k_groups, kb_per_group, n_groups;
};

// GEMM tile variant selected by the host planner.
struct GemmPlan {
    int bn;          // N tile (UMMA N)
    int stages;      // pipeline depth
    int grid;        // persistent CTAs (a multiple of 2 for CTA pairs)
    size_t smem;     // dynamic shared memory bytes
    bool pair;       // CTA-pair kernel (tcgen05 cta_group::2, 256-row tiles)
    int bm;          // rows per output tile: 128, or 256 for a CTA pair
    int b_rows;      // rows of W in one TMA box (BN, or BN / 2 for a CTA pair)
    int nsub;        // N sub-tiles of BN columns per output tile (CTA pair: 1 or 2)
    int tw;          // output tile width in N: bn * nsub, or bn when gated
    bool gated;      // SwiGLU: sub-tile 0 multiplies the gate weight, 1 the up weight
    int splits;      // K ranges per output tile (1 = none)
    bool mc = false; // clusters of two CTA pairs sharing the weight boxes (multicast):
                     // 512 x 464 super-tiles, sub-tiles 224 + 240
};

// The multicast cluster kernel's super-tile and weight-box geometry, and
// the epilogue chunks of a CTA's 464 accumulator columns (14 of 32, one of
// 16), which are also the units of its K-split partials and counters.
constexpr int kMcRows = 512;
constexpr int kMcCols = 464;
constexpr int kMcChunks = 15;

// Bytes of FP32 partials and of counters a split plan needs (ctas: CTAs
// per output tile, 2 for the CTA pair, 1 for the single-CTA kernel).
size_t split_partial_bytes(int64_t num_tiles, int tw, int splits, int ctas = 2);
size_t split_counter_bytes(int64_t num_tiles, int tw, int ctas = 2);
// The multicast kernel's split partials and counters for `super` super-tiles.
size_t mc_split_partial_bytes(int64_t super, int splits);
size_t mc_split_counter_bytes(int64_t super);
// The single-CTA kernel splits K at most this many ways, into ranges of at
// least kMinKbPerSplitSingle k blocks.
constexpr int kMaxSplitsSingle = 4;
constexpr int kMinKbPerSplitSingle = 16;

// Record why a CUDA call failed (thread-local; read back through
// ngr_last_error).  Returns -7 (NGR_ERR_CUDA) for use in return statements.
int record_cuda_error(const char *what, int code, const char *detail);

// NGR_DEBUG set (and not "0"): every entry point synchronizes its stream
// after launching and reports the device error word.
bool debug_mode();
// Bound on every in-kernel barrier wait: NGR_WAIT_TIMEOUT_MS, default 2 s.
unsigned long long wait_timeout_ns();
// Tensor maps (record the reason in ngr_last_error on failure):
// row-major [rows, cols] 16-bit matrix, box {64 columns, box_rows rows},
// 128-byte swizzle;
bool map_2d(CUtensorMap *m, const void *ptr, bool bf16, int64_t rows, int64_t cols,
            uint32_t box_rows);
// FP32 gamma and beta as the two rows of a [2, K] matrix whose rows are
// `row_stride` bytes apart, box {64 columns, 2 rows}, no swizzle.
bool map_gb(CUtensorMap *m, const float *gamma_f, int64_t K, size_t row_stride);

// Launchers (return 0 or a negative ngr_status).
int launch_rowstats(int norm, bool bf16, const void *x, int64_t M, int64_t K,
                    float eps, float2 *stats, const void *gamma,
                    const void *beta, float *gamma_f, float *beta_f,
                    int *counters, int n_counters, int *err_to_clear,
                    int num_sms, cudaStream_t stream, void *xhat = nullptr,
                    int64_t k_valid = -1, bool pdl = false);

// Copies for shapes whose K or N is not a multiple of 8 (ngr_pad.cu):
// rows of `cols` 16-bit values (pitch `src_pitch`) into rows of `dst_cols`
// (a multiple of 8) with a zero tail, followed by zero rows up to
// `dst_rows` (default: none), and back.
int launch_pad_rows(const void *src, int64_t rows, int64_t cols, int64_t src_pitch, void *dst,
                    int64_t dst_cols, int num_sms, cudaStream_t stream, int64_t dst_rows = 0);
int launch_unpad_rows(const void *src, int64_t rows, int64_t cols, int64_t src_pitch, void *dst,
                      int num_sms, cudaStream_t stream);

int launch_gemm(int norm, bool bf16, const GemmPlan &plan, const GemmArgs &args, bool pdl,
                cudaStream_t stream);
int launch_gemm4(int norm, bool bf16, const GemmArgs &args, int grid, bool pdl, cudaStream_t stream);
int gemm4_clusters();           // resident clusters of four of the multicast kernel
size_t gemm4_smem_bytes();
// max_split_bytes: room for split-K partials and counters (0 = never split).
// norm: a LayerNorm or RMSNorm on x; plain: no transform of x (no norm, or
// a folded weight with the statistics applied in the epilogue).  The
// multicast kernel takes either.
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, bool norm,
                   size_t max_split_bytes = 0, bool plain = false);
// The SwiGLU variant: CTA-pair tiles of 256 x BN outputs, two BN-column
// accumulators (gate, up) per tile.
GemmPlan plan_gemm_gated(int64_t M, int64_t N, int num_sms);
int set_tile_config(int pair, int bn, int nsub);
size_t gemm_smem_bytes(int bn, int stages, bool norm);

int launch_decode(int norm, bool bf16, int mn, const DecodeArgs &args, bool pdl,
                  cudaStream_t stream);
DecodePlan plan_decode(int64_t n_tiles, int64_t k_blocks, int mn, int num_sms);
size_t decode_smem_bytes(int mn);

int launch_fold_prepare(int norm, bool bf16, const void *gamma, const void *beta,
                        const void *W, const void *bias, int64_t K, int64_t N, void *Wf,
                        float *cb, int num_sms, cudaStream_t stream);
// The fold for any K, N and 2-byte-aligned operands: Wf as [N, K8] rows, cb
// as [2, N8] (K8, N8: K, N rounded up to multiples of 8; zero padding).
int launch_fold_prepare_any(int norm, bool bf16, const void *gamma, const void *beta,
                            const void *W, const void *bias, int64_t K, int64_t N, void *Wf,
                            float *cb, int num_sms, cudaStream_t stream);

int launch_bounded_wait_probe(int *err, unsigned long long timeout_ns,
                              cudaStream_t stream);

}  // namespace ngr
