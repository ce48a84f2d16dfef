// Internal interface between the host API (api.cpp) and the kernel launchers.
// Plain structs of device pointers and sizes, passed to the kernels by value.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qkvp {

constexpr int kThreads = 256;         // threads per CTA for the GQA kernels
constexpr int kMaxHalf = 64;          // RoPE frequencies for head_dim 128
constexpr int kFwdChunksPerThread = 10;
constexpr int kBwdChunksPerThread = 6;
constexpr int kMaxBwdParts = 1024;    // cap on per-CTA weight-grad partial rows

enum Role : int { kRoleQ = 0, kRoleK = 1, kRoleV = 2 };

// Streaming (shared-memory staged) kernels.
// Shape of the pipelined kernels: consumer warps per CTA (+1 producer warp),
// the CTAs per SM the shared-memory budget is cut for, the most bytes to keep
// in flight in the ring, and the smallest stage worth a tile. Measured on
// GB300 (T = 16384, Muse Spark packing): one CTA of 10 consumer warps per SM
// is best for the forward (with and without the pre-norm save) and the
// backward (with 11 warps per SM the register cap is 168 per thread, enough
// for the pair-per-lane backward without spills). The bytes in flight pace
// the reads: the RoPE forwards and the backward run best with about 160 KB in
// flight per SM (8 stages of a 20 KB token, 4 of a 39 KB one), the NoPE
// forward, whose consumers finish a tile quickly, with half of that (deeper
// rings issue the reads in bursts that interleave worse with the writes).
// Tiles of at least 16 KB keep rows of small models (10-12 KB per token)
// from giving rings too shallow to cover the memory latency.
struct StreamShape {
  int warps;
  int ctas_per_sm;
  int max_inflight;     // bytes of stage data in flight per CTA (cap)
  int min_stage_bytes;  // smallest tile worth taking
};
constexpr StreamShape fwd_stream_shape(bool save_pre, bool rope = true) {
  return StreamShape{10, 1, (save_pre || rope) ? 160 * 1024 : 80 * 1024, 16 * 1024};
}
constexpr StreamShape bwd_stream_shape() { return StreamShape{10, 1, 160 * 1024, 16 * 1024}; }
constexpr int kMaxStages = 8;  // depth of the shared-memory ring (max)
constexpr int kStreamMaxSteps = 6;       // 16-byte chunks per consumer thread per tile (max)

#if defined(__CUDACC__)
#define QKVP_HD __host__ __device__
#else
#define QKVP_HD
#endif

// Shared-memory layout of a streaming CTA (byte offsets).
struct StreamSmem {
  static constexpr int kBarriers = 0;                  // uint64 full[kMaxStages], empty[kMaxStages]
  static constexpr int kWeights = 2 * kMaxStages * 8;  // float w_q[hd], w_k[hd]
  QKVP_HD static int tables(int hd) { return kWeights + 2 * hd * 4; }
  // per stage: float cos[tpt][hd/2], sin[tpt][hd/2], then int32 slot[tpt]
  QKVP_HD static int table_stride(int hd, int tpt) { return (tpt * hd * 4 + tpt * 4 + 15) & ~15; }
  // stage data, 128-byte aligned
  QKVP_HD static int data(int hd, int tpt, int stages) {
    return (tables(hd) + stages * table_stride(hd, tpt) + 127) & ~127;
  }
  // after the ring: float bias[row] of the GQAttention variant (when given)
  QKVP_HD static int bias(int hd, int tpt, int stages, int stage_bytes) {
    return data(hd, tpt, stages) + stages * stage_bytes;
  }
};

struct StreamGeom {
  int32_t tpt;          // tokens per tile
  int32_t stages;       // stages in the ring
  int32_t steps;        // chunks per consumer thread per tile
  int32_t stage_bytes;  // bytes of one stage's data
  int64_t n_tiles;
  int32_t dense;        // packed rows are contiguous: one bulk copy per tile
  int32_t pad_;
};

struct RopeTable {
  uint64_t turns[kMaxHalf];  // frac(inv_freq_i / 2pi) * 2^64
  float scale;               // factor on cos and sin (1 for plain RoPE)
  int32_t pad_;
};

// Bias gradient of the backward: at most this many chunk pairs per consumer
// thread (its running sums stay in registers).
constexpr int kBiasMaxSteps = 2;

// Forward (contiguous or paged-pool destination), GQA layouts.
struct FwdArgs {
  const uint4* packed;
  int64_t row_stride16;   // packed row stride, 16-byte chunks
  const int32_t* pos;
  const float* w_q;
  const float* w_k;
  float eps;
  float inv_head_dim;
  int64_t T;
  int32_t n_q, n_kv, group;
  int32_t cpt;            // 16-byte chunks per token = heads * head_dim / 8
  uint32_t cpt_magic;     // floor(2^32 / cpt) + 1
  uint32_t gs_magic;      // floor(2^32 / (group + 2)) + 1
  int64_t item_chunks;    // chunks per work item
  int64_t n_items;
  int32_t max_tok;        // tokens an item can touch (shared-memory table rows)
  uint4* q;
  uint4* k;
  uint4* v;
  uint4* q_pre;
  uint4* k_pre;
  const int32_t* page;
  const int32_t* offset;
  uint4* k_pool;
  uint4* v_pool;
  int32_t num_pages, page_size;
  int32_t* dev_status;
  int* err;               // library device error word
  const float* bias;      // [cpt * 8] in packed-row order, or null
  StreamGeom sg;
  RopeTable rope;
};

struct BwdArgs {
  const uint4* dq;
  const uint4* dk;
  const uint4* dv;
  const uint4* q_pre;
  const uint4* k_pre;
  const int32_t* pos;
  const float* w_q;
  const float* w_k;
  float eps;
  float inv_head_dim;
  int64_t T;
  int32_t n_q, n_kv, group;
  int32_t cpt;
  uint32_t cpt_magic;
  uint32_t gs_magic;
  int64_t item_chunks;
  int64_t n_items;
  int32_t max_tok;
  uint4* dpacked;
  int64_t row_stride16;
  float* partials;        // [grid][2][head_dim] (norm on)
  float* db_partials;     // [grid][cpt * 8] (bias given)
  // Weight-gradient fold of the pipelined kernel (norm on, no bias): the CTA
  // that finishes last adds the partial rows (fixed order) into dw_q / dw_k
  // itself, so no finalize kernel runs. null flags: the finalize kernel does it.
  uint32_t* flags;             // [grid] per-CTA arrival words, then the election word
  uint32_t call_id;            // this call's generation (never 0)
  int32_t accumulate;          // add to dw_q / dw_k instead of overwriting
  float* dw_q;
  float* dw_k;
  const float* bias;      // [cpt * 8] in packed-row order, or null
  int* err;
  StreamGeom sg;
  RopeTable rope;
};

struct LatentArgs {
  const uint4* rows;
  int64_t row_stride16;
  const int32_t* pos;
  const float* w;
  float eps;
  float inv_norm_dim;
  int64_t T;
  int32_t norm_chunks;    // norm_dim / 8
  int32_t row_chunks;     // (norm_dim + rope_dim) / 8
  uint4* out;             // contiguous destination [T, row_chunks] (or null)
  const int32_t* page;
  const int32_t* offset;
  uint4* pool;            // pool destination (or null)
  int32_t num_pages, page_size;
  int32_t* dev_status;
  int* err;               // library device error word (pipelined kernel)
  StreamGeom sg;          // pipelined kernel geometry
  RopeTable rope;
};

struct ScatterArgs {
  const uint4* src_a;     // [T, row_chunks]
  const uint4* src_b;     // optional second source (v), same shape
  uint4* pool_a;
  uint4* pool_b;
  int64_t T;
  int32_t row_chunks;
  const int32_t* page;
  const int32_t* offset;
  int32_t num_pages, page_size;
  int32_t* dev_status;
};

struct FwdVariant {
  int head_dim;       // 64 or 128
  bool sectioned;
  bool rope;
  bool save_pre;
  bool pool;
  bool norm;          // RMSNorm of q and k (off: split -> RoPE only)
  bool bias;          // qkv bias added first
};

struct BwdVariant {
  int head_dim;
  bool sectioned;
  bool rope;
  bool norm;
  bool bias;
  int steps;  // chunk pairs per consumer thread of the pipelined kernel (0: not known yet)
};

// Kernel entry points (host stubs for cudaLaunchKernel / occupancy queries).
// Each takes its argument struct by value as the only parameter.
// One getter per instance file (head_dim x norm on / off).
const void* fwd_kernel_d64_norm(const FwdVariant& v);
const void* fwd_kernel_d64_nonorm(const FwdVariant& v);
const void* fwd_kernel_d128_norm(const FwdVariant& v);
const void* fwd_kernel_d128_nonorm(const FwdVariant& v);
const void* bwd_kernel_norm(const BwdVariant& v);
const void* bwd_kernel_nonorm(const BwdVariant& v);
const void* fwd_stream_kernel_d64_norm(const FwdVariant& v);
const void* fwd_stream_kernel_d64_nonorm(const FwdVariant& v);
const void* fwd_stream_kernel_d128_norm(const FwdVariant& v);
const void* fwd_stream_kernel_d128_nonorm(const FwdVariant& v);
const void* bwd_stream_kernel_norm(const BwdVariant& v);
const void* bwd_stream_kernel_nonorm(const BwdVariant& v);

inline const void* fwd_kernel(const FwdVariant& v) {
  if (v.head_dim == 64) return v.norm ? fwd_kernel_d64_norm(v) : fwd_kernel_d64_nonorm(v);
  return v.norm ? fwd_kernel_d128_norm(v) : fwd_kernel_d128_nonorm(v);
}
inline const void* fwd_stream_kernel(const FwdVariant& v) {
  if (v.head_dim == 64) return v.norm ? fwd_stream_kernel_d64_norm(v) : fwd_stream_kernel_d64_nonorm(v);
  return v.norm ? fwd_stream_kernel_d128_norm(v) : fwd_stream_kernel_d128_nonorm(v);
}
inline const void* bwd_kernel(const BwdVariant& v) { return v.norm ? bwd_kernel_norm(v) : bwd_kernel_nonorm(v); }
inline const void* bwd_stream_kernel(const BwdVariant& v) {
  return v.norm ? bwd_stream_kernel_norm(v) : bwd_stream_kernel_nonorm(v);
}
const void* dw_finalize_kernel();
const void* latent_kernel(bool pool, bool rope, int norm_chunks_per_lane);
const void* scatter_kernel();
const void* latent_stream_kernel(bool pool, bool rope, int norm_chunks_per_lane);

// Address of the library's device error word on the current device (nullptr
// if it cannot be obtained), and its value (read and optionally cleared,
// synchronously).
int* device_error_word();
int read_device_error(bool clear, int* value);

// qkvp_dw_finalize_kernel arguments: outputs [dw_q | dw_k] (when dw_q is set)
// then db (when db is set), each the float64 sum of its column of partial rows.
struct FinalizeArgs {
  const float* partials;     // [nparts][2][head_dim]
  const float* db_partials;  // [nparts][n_bias]
  int32_t nparts;
  int32_t head_dim;
  int32_t n_bias;            // bias length (cpt * 8), 0 without a bias
  float* dw_q;               // null: no weight gradients (norm off)
  float* dw_k;
  float* db;                 // null: no bias gradient
  int32_t accumulate;
};
constexpr int kFinalizeOutputsPerCta = 32;
constexpr int kFinalizeThreads = 256;

// The wqkv projection with the prologue in its epilogue (tcgen05): tile of
// a CTA pair computes 2 kGemmBM tokens x kGemmBN packed columns (each CTA
// holds kGemmBM token rows of it), kGemmBK per pipeline stage.
constexpr int kGemmBM = 128, kGemmBN = 256, kGemmBK = 64;
struct GemmArgs {
  int64_t T;              // tokens (rows of x)
  int32_t hidden;         // K: columns of x and W
  int32_t n_q, n_kv, group, n_blocks;  // n_blocks = n_q + 2 n_kv head blocks of the packed row
  uint32_t gs_magic;      // floor(2^32 / (group + 2)) + 1
  int32_t m_tiles, n_tiles;  // M tiles of 2 kGemmBM tokens (one per CTA pair), N tiles of kGemmBN columns
  int64_t n_work;         // m_tiles * n_tiles
  const int32_t* pos;
  const float* w_q;
  const float* w_k;
  float eps;
  float inv_head_dim;
  uint4* q;
  uint4* k;
  uint4* v;
  uint4* q_pre;
  uint4* k_pre;
  int* err;
  RopeTable rope;
};
// Tensor maps of the projection kernel's outputs, each the 2-D view
// [T, heads * head_dim] bf16 read in boxes of 64 columns x 32 tokens with the
// 128-byte swizzle (the epilogue stores its tiles with TMA).
struct GemmOutMaps {
  CUtensorMap q, k, v, q_pre, k_pre;
};
const void* gemm_fwd_kernel(int head_dim, bool sectioned, bool rope, bool save);
int gemm_fwd_smem_bytes();
int gemm_fwd_threads();

// Per-head Newton-Schulz of a fused QKV update through the block Gram
// matrices: a Gram pass (split CTAs per unit of 128 weight rows, each a range
// of 64-column boxes), a polynomial pass (one CTA per unit) and an apply pass
// (persistent, boxes of 128 rows x 64 columns).
constexpr int kNsUnitRows = 128;
constexpr int kNsMaxSplit = 64;  // Gram CTAs per unit
struct NsArgs {
  int32_t rows;      // count (n_q + 2 n_kv) head_dim: rows of the (stacked) weight
  int32_t cols;      // in_features
  int32_t head_dim;  // 64 or 128
  int32_t units;     // ceil(rows / 128)
  int32_t nb;        // cols / 64
  int32_t split;     // Gram CTAs per unit, at most nb
  float scale;       // max(1, head_dim / cols) ** 0.5
  float eps;         // added to each block's Frobenius norm
  float* partial;    // workspace: [units * split][128][head_dim + 4] fp32 Gram partials
  uint4* mh;         // workspace: [units][2][128 x 128] bf16 hi, lo planes of M (swizzled box images)
  int* err;
};
// Row stride of a Gram partial, in floats: head_dim plus 4, so that the 32
// rows a warp reads from shared memory start in different banks.
QKVP_HD constexpr int ns_partial_stride(int head_dim) { return head_dim + 4; }
// Gram partials the polynomial kernel stages in shared memory at a time.
QKVP_HD constexpr int ns_poly_stage_parts(int head_dim) { return head_dim == 64 ? 6 : 3; }
const void* ns_gram_kernel();
const void* ns_poly_kernel(int head_dim);
const void* ns_apply_kernel();
int ns_gram_smem_bytes();
int ns_poly_smem_bytes(int head_dim);
int ns_apply_smem_bytes();
int ns_gram_threads();
int ns_poly_threads();
int ns_apply_threads();

// One thread whose only wait never completes (the bounded-wait self-test).
const void* wait_selftest_kernel();

constexpr int kLatentWarps = 8;        // warps per CTA of the latent kernel
constexpr int kLatentTokensPerWarp = 2;
constexpr int kLatentTileTokens = 16;     // rows per tile of the pipelined latent kernel
constexpr int kLatentStreamWarps = 4;     // its consumer warps (+1 producer); 4 rows per warp per tile
constexpr int kLatentStreamCtasPerSm = 4; // small tiles and many CTAs: the first rows arrive early

}  // namespace qkvp
