// Host side of the C ABI: argument checks, RoPE frequency tables, launch
// geometry and dispatch to the kernels. Nothing here allocates device memory
// or synchronises; every launch goes to the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <atomic>
#include <mutex>

#include "launch.h"
#include "qkv_prologue.h"

namespace qkvp {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxHeadsTimesChunks = 32768;  // keeps in-item chunk indices below 2^16

// ------------------------------------------------------------ device ----

struct DeviceInfo {
  bool probed = false;
  int status = QKVP_OK;
  int sms = 0;
  int smem_per_sm = 0;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

// The current device, checked once per device: it must be sm_103 (the only
// architecture the library is compiled for).
int current_device(int* sms, int* smem_per_sm = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return QKVP_ERR_ARCH;
  }
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    int major = 0, minor = 0, sms_ = 0, smem_ = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms_, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
      cudaGetLastError();
      return QKVP_ERR_ARCH;
    }
    d.status = (major == 10 && minor == 3) ? QKVP_OK : QKVP_ERR_ARCH;
    d.sms = sms_;
    d.smem_per_sm = smem_;
    d.probed = true;
  }
  *sms = d.sms;
  if (smem_per_sm) *smem_per_sm = d.smem_per_sm;
  return d.status;
}

// Resident CTAs per SM for (kernel, threads, smem) on the current device,
// queried once and cached (a launch then makes no query call). 0 means the
// kernel cannot be launched with these resources; callers then take another
// kernel.
int blocks_per_sm(const void* kernel, int threads, size_t smem) {
  struct Entry {
    int dev;
    const void* kernel;
    int threads;
    size_t smem;
    int blocks;
  };
  static std::mutex mu;
  static Entry cache[512];
  static int n_cached = 0;
  int dev = -1;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
      if (cache[i].dev == dev && cache[i].kernel == kernel && cache[i].threads == threads && cache[i].smem == smem)
        return cache[i].blocks;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (n_cached < 512) cache[n_cached++] = Entry{dev, kernel, threads, smem, n};
  return n;
}

// Opt a kernel in to `smem` bytes of dynamic shared memory (once per device
// and kernel; the attribute only ever grows).
bool allow_smem(const void* kernel, size_t smem) {
  if (smem <= 48 * 1024) return true;
  struct Entry {
    int dev;
    const void* kernel;
    size_t bytes;
  };
  static std::mutex mu;
  static Entry cache[256];
  static int n = 0;
  int dev = -1;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].dev == dev && cache[i].kernel == kernel && cache[i].bytes >= smem) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (n < 256) cache[n++] = Entry{dev, kernel, smem};
  return true;
}

// Tile geometry of the streaming kernels, or false when the layout does not
// fit them. A tile holds tpt tokens; each token's upt units (chunk pairs) are
// split over tpg = consumers / tpt threads taking steps = ceil(upt / tpg)
// units each (steps <= max_steps); lph = lanes per head. Among the tile sizes
// whose last step is at least kMinStepFill full, the smallest one of at least
// shape.min_stage_bytes is taken (else the largest), so a tile stays small
// and the ring deep; the ring holds up to shape.max_inflight bytes, at least
// two stages, in the shared memory left to each of the shape.ctas_per_sm CTAs
// of an SM. token_bytes = bytes staged per token. extra_dyn = dynamic shared
// memory after the ring (the bias copy); any_fill = take tile sizes whatever
// their last step's fill (the bias gradient, whose step cap is small).
bool stream_geometry(const StreamShape& shape, int upt, int lph, int hd, int64_t T, int64_t token_bytes,
                     int smem_per_sm, int static_smem, int extra_dyn, bool any_fill, int max_steps,
                     bool prefer_fill, StreamGeom* g, size_t* smem) {
  constexpr double kMinStepFill = 0.8;  // useful chunks / (steps * tpg)
  const int nct = shape.warps * 32;
  const int budget = smem_per_sm / shape.ctas_per_sm - 1024 - static_smem - extra_dyn;
  // Tiles of tpt tokens, tpt dividing the consumer threads into token groups of
  // whole heads. Larger tiles only add steps and stage bytes, so a scan stops
  // at the first that needs more than max_steps steps or no longer fits two
  // stages.
  //  * prefer_fill: any such tpt; among them, preferring tiles of at least
  //    min_stage_bytes, the highest fill of the steps times the share of
  //    shape.max_inflight the ring can hold, then the smallest tile (the
  //    backward and the norm-off forward at head_dim 128: 4-token tiles, 96 %
  //    full, against 2-token tiles, 80 % full: Qwen3 backward 111 -> 99 us,
  //    Llama 3 forward 78 -> 69 us on GB300);
  //  * else tpt = 1, 2, 4, ...: the first of at least min_stage_bytes whose
  //    steps are at least kMinStepFill full (the norm-on forward, whose
  //    4-token tiles measured slower: Qwen3 forward 94 -> 98 us).
  int pick = 0;
  if (prefer_fill) {
    double pick_score = -1.0;
    bool pick_big = false;
    for (int tpt = 1; tpt <= nct / lph; ++tpt) {
      if (nct % tpt != 0 || (nct / tpt) % lph != 0) continue;
      const int tpg = nct / tpt;
      const int steps = (upt + tpg - 1) / tpg;
      if (steps > max_steps) break;
      const int64_t stage = (int64_t)tpt * token_bytes;
      const int64_t per_stage = stage + StreamSmem::table_stride(hd, tpt);
      const int64_t fit = (budget - StreamSmem::tables(hd) - 128) / per_stage;
      if (fit < 2) break;
      const double fill = (double)upt / ((double)steps * tpg);
      if (!any_fill && fill < kMinStepFill) continue;
      const int64_t stages = std::min<int64_t>(
          std::min<int64_t>(fit, std::max<int64_t>(2, shape.max_inflight / stage)), kMaxStages);
      const double held = std::min(1.0, (double)(stages * stage) / (double)shape.max_inflight);
      const double score = fill * held;
      const bool big = stage >= shape.min_stage_bytes;
      if (pick == 0 || (big && !pick_big) || (big == pick_big && score > pick_score + 1e-9)) {
        pick = tpt;
        pick_score = score;
        pick_big = big;
      }
    }
  } else {
    for (int tpt = 1; nct / tpt >= lph && (nct / tpt) % lph == 0; tpt *= 2) {
      const int tpg = nct / tpt;
      const int steps = (upt + tpg - 1) / tpg;
      if (steps > max_steps) break;
      if (!any_fill && (double)upt / ((double)steps * tpg) < kMinStepFill) continue;
      const int64_t per_stage = (int64_t)tpt * token_bytes + StreamSmem::table_stride(hd, tpt);
      if ((budget - StreamSmem::tables(hd) - 128) / per_stage < 2) break;
      pick = tpt;
      if ((int64_t)tpt * token_bytes >= shape.min_stage_bytes) break;
    }
  }
  if (pick == 0) return false;
  const int tpt = pick;
  const int64_t stage = (int64_t)tpt * token_bytes;
  const int64_t per_stage = stage + StreamSmem::table_stride(hd, tpt);
  int64_t stages = (budget - StreamSmem::tables(hd) - 128) / per_stage;
  int64_t by_bytes = shape.max_inflight / stage;
  if (by_bytes < 2) by_bytes = 2;
  if (stages > by_bytes) stages = by_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  g->tpt = tpt;
  g->stages = (int32_t)stages;
  g->steps = (upt + nct / tpt - 1) / (nct / tpt);
  g->stage_bytes = (int32_t)stage;
  g->n_tiles = (T + tpt - 1) / tpt;
  *smem = (size_t)StreamSmem::data(hd, tpt, (int)stages) + (size_t)stages * stage + (size_t)extra_dyn;
  return true;
}

// Launch with programmatic stream serialization: the kernel may be launched
// while the previous kernel in the stream is still running; every kernel of the
// library waits (griddepcontrol.wait) for it before touching memory.
int launch(const void* kernel, int64_t grid, int threads, size_t smem, cudaStream_t s, void* arg) {
  void* args[] = {arg};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelExC(&cfg, kernel, args);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return err == cudaErrorNoKernelImageForDevice || err == cudaErrorInvalidDeviceFunction
               ? QKVP_ERR_ARCH
               : QKVP_ERR_LAUNCH;
  }
  return QKVP_OK;
}

// Launch with several kernel parameters (same attributes as launch()), in
// clusters of `cluster` CTAs along x when cluster > 1, or always when
// explicit_cluster (a kernel that uses cluster-only instructions such as
// st.async needs an explicit cluster launch even for one CTA).
int launch_args(const void* kernel, int64_t grid, int threads, size_t smem, cudaStream_t s, void** args,
                int cluster = 1, bool pdl = true, bool explicit_cluster = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n_attr = 0;
  if (pdl) {
    attr[n_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n_attr++].val.programmaticStreamSerializationAllowed = 1;
  }
  if (cluster > 1 || explicit_cluster) {
    attr[n_attr].id = cudaLaunchAttributeClusterDimension;
    attr[n_attr].val.clusterDim.x = (unsigned)cluster;
    attr[n_attr].val.clusterDim.y = 1;
    attr[n_attr++].val.clusterDim.z = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n_attr;
  const cudaError_t err = cudaLaunchKernelExC(&cfg, kernel, args);
  if (err != cudaSuccess) {
    cudaGetLastError();
    return err == cudaErrorNoKernelImageForDevice || err == cudaErrorInvalidDeviceFunction ? QKVP_ERR_ARCH
                                                                                            : QKVP_ERR_LAUNCH;
  }
  return QKVP_OK;
}

// Clusters of two CTAs of (kernel, threads, smem) that can be resident at
// once on the current device (cached per device and kernel), or 0.
int max_clusters_of_2(const void* kernel, int threads, size_t smem) {
  struct Entry {
    int dev;
    const void* kernel;
    size_t smem;
    int n;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n_cached = 0;
  int dev = -1;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_cached; ++i)
      if (cache[i].dev == dev && cache[i].kernel == kernel && cache[i].smem == smem) return cache[i].n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (n_cached < 64) cache[n_cached++] = Entry{dev, kernel, smem, n};
  return n;
}

// cuTensorMapEncodeTiled, fetched from the driver once (the library does not
// link libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Tensor map of a row-major bf16 matrix [rows, cols] (cols contiguous, a
// multiple of 8) read in boxes of 64 columns x box_rows rows with the 128-byte
// swizzle the tcgen05 descriptors expect; outside the matrix a box reads 0.
bool bf16_tile_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols, int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, elem,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// -------------------------------------------------------------- RoPE ----

// turns_i = frac(inv_freq_i / 2pi) * 2^64 with inv_freq_i = base^(-2i/D), or
// the caller's table: the angle per unit position as a 0.64 fixed-point
// fraction of one turn. The kernels multiply it by the position modulo 2^64,
// which reduces the angle exactly. Double precision leaves < 2^-56 turn of
// error per unit position (about 2^-37 turn at position 2^19).
uint64_t turns_of(double inv_freq) {
  const double two_pi = 6.283185307179586476925286766559;
  const double v = inv_freq / two_pi;
  const double frac = v - std::floor(v);  // in [0, 1), exact
  const double scaled = std::ldexp(frac, 64);
  return scaled >= 18446744073709551616.0 ? 0 : (uint64_t)scaled;
}

void rope_table(double base, int dim, const double* inv_freq, float scale, RopeTable* out) {
  if (inv_freq) {
    std::memset(out, 0, sizeof(*out));
    for (int i = 0; i < dim / 2; ++i) out->turns[i] = turns_of(inv_freq[i]);
    out->scale = scale;
    return;
  }
  static thread_local double last_base = -1.0;
  static thread_local int last_dim = 0;
  static thread_local RopeTable last;
  if (base != last_base || dim != last_dim) {
    std::memset(&last, 0, sizeof(last));
    for (int i = 0; i < dim / 2; ++i) last.turns[i] = turns_of(std::pow(base, -2.0 * i / dim));
    last_base = base;
    last_dim = dim;
  }
  *out = last;
  out->scale = scale;
}

// ------------------------------------------------------------ checks ----

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// True when p points into device memory of the current device (not host,
// managed-on-host or another GPU's memory reached through peer access).
bool on_current_device(const void* p) {
  int dev = -1;
  cudaPointerAttributes attr;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeDevice && attr.device == dev;
}
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Gqa {
  int heads = 0;          // n_q + 2 n_kv
  int64_t row = 0;        // elements per row (heads * head_dim)
  int64_t stride = 0;     // row stride in elements
};

int check_gqa(const qkvp_layout* L, int64_t T, Gqa* g) {
  if (!L) return QKVP_ERR_NULL;
  if (L->kind != QKVP_INTERLEAVED && L->kind != QKVP_SECTIONED) return QKVP_ERR_SHAPE;
  if (T < 0 || L->n_q <= 0 || L->n_kv <= 0 || L->n_q % L->n_kv != 0) return QKVP_ERR_SHAPE;
  if (L->head_dim != 64 && L->head_dim != 128) return QKVP_ERR_SHAPE;
  const int64_t heads = (int64_t)L->n_q + 2 * (int64_t)L->n_kv;
  if (heads * (L->head_dim / 8) > kMaxHeadsTimesChunks) return QKVP_ERR_SHAPE;
  g->heads = (int)heads;
  g->row = heads * L->head_dim;
  g->stride = L->row_stride == 0 ? g->row : L->row_stride;
  if (g->stride < g->row || g->stride % 8 != 0) return QKVP_ERR_SHAPE;
  return QKVP_OK;
}

struct Latent {
  int64_t row = 0;
  int64_t stride = 0;
};

int check_latent(const qkvp_layout* L, int64_t T, Latent* g) {
  if (!L) return QKVP_ERR_NULL;
  if (L->kind != QKVP_LATENT || T < 0) return QKVP_ERR_SHAPE;
  if (L->norm_dim < 8 || L->norm_dim > 1024 || L->norm_dim % 8 != 0 || L->rope_dim != 64)
    return QKVP_ERR_SHAPE;
  g->row = (int64_t)L->norm_dim + L->rope_dim;
  g->stride = L->row_stride == 0 ? g->row : L->row_stride;
  if (g->stride < g->row || g->stride % 8 != 0) return QKVP_ERR_SHAPE;
  return QKVP_OK;
}

int check_scalars(float eps, double rope_base, bool rope) {
  if (!(eps >= 0.f) || !std::isfinite(eps)) return QKVP_ERR_VALUE;
  if (rope && (!(rope_base > 0.0) || !std::isfinite(rope_base))) return QKVP_ERR_VALUE;
  return QKVP_OK;
}

int check_pool(int32_t num_pages, int32_t page_size) {
  if (num_pages <= 0 || page_size <= 0) return QKVP_ERR_VALUE;
  if ((int64_t)num_pages * page_size > INT32_MAX) return QKVP_ERR_VALUE;
  return QKVP_OK;
}

uint32_t magic(uint32_t d) { return (uint32_t)((1ull << 32) / d + 1); }

// Work items of the GQA kernels: `chunks_per_thread * kThreads` consecutive
// (token, chunk) pairs.
void gqa_items(int64_t T, int cpt, int chunks_per_thread, int64_t* item_chunks, int64_t* n_items,
               int* max_tok) {
  const int64_t L = (int64_t)chunks_per_thread * kThreads;
  *item_chunks = L;
  *n_items = (T * cpt + L - 1) / L;
  *max_tok = (int)((cpt + L - 2) / cpt + 1);
}

int64_t bwd_parts(int64_t n_items) { return n_items < kMaxBwdParts ? n_items : kMaxBwdParts; }

// The GQAttention variant options of a call, checked.
struct Variant {
  const double* inv_freq = nullptr;
  float scale = 1.f;
  const float* bias = nullptr;
};

int check_variant(const qkvp_variant* v, int rope_dim, bool gqa, Variant* out) {
  *out = Variant();
  if (!v) return QKVP_OK;
  if (v->inv_freq) {
    for (int i = 0; i < rope_dim / 2; ++i)
      if (!std::isfinite(v->inv_freq[i])) return QKVP_ERR_VALUE;
    out->inv_freq = v->inv_freq;
  }
  if (!std::isfinite(v->rope_scale) || v->rope_scale < 0.0) return QKVP_ERR_VALUE;
  out->scale = v->rope_scale == 0.0 ? 1.f : (float)v->rope_scale;
  if (v->bias) {
    if (!gqa) return QKVP_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(v->bias) & 15u) != 0) return QKVP_ERR_ALIGN;
    out->bias = v->bias;
  }
  return QKVP_OK;
}

// Bias gradient limits: the pipelined backward keeps at most kBiasMaxSteps
// chunk pairs per thread; the general backward takes one-token work items of
// at most kThreads * kBwdChunksPerThread chunks.
constexpr int kBiasMaxChunks = kThreads * kBwdChunksPerThread;

#define QKVP_TRY(expr)          \
  do {                          \
    const int _st = (expr);     \
    if (_st != QKVP_OK) return _st; \
  } while (0)

// ------------------------------------------- per-head Newton-Schulz ----

// Gram CTAs per 128-row unit: `want` when given, else enough for about two
// Gram CTAs per SM over all units (they are small: three fit on one SM),
// keeping at least four 64-column boxes (64 KiB of the weight) per CTA.
int ns_split(int64_t units, int nb, int want, int sms) {
  if (want > 0) return want;
  int64_t s = (2 * (int64_t)sms + units - 1) / units;
  const int64_t cap = nb / 4 > 1 ? nb / 4 : 1;
  if (s > cap) s = cap;
  if (s > kNsMaxSplit) s = kNsMaxSplit;
  return s < 1 ? 1 : (int)s;
}

// Workspace: the fp32 Gram partials, then each unit's M image (64 KiB).
size_t ns_partial_bytes(int64_t units, int split, int head_dim) {
  return (size_t)units * (size_t)split * kNsUnitRows * (size_t)ns_partial_stride(head_dim) * 4;
}
size_t ns_workspace_bytes(int64_t units, int split, int head_dim) {
  return ns_partial_bytes(units, split, head_dim) + (size_t)units * 65536;
}

// Shape checks shared by the Newton-Schulz entry points; *rows = the rows of
// `count` fused weights stacked along dim 0.
int check_ns(const qkvp_layout* layout, int64_t count, int64_t cols, int32_t split, int64_t* rows) {
  if (!layout) return QKVP_ERR_NULL;
  if (layout->kind != QKVP_INTERLEAVED && layout->kind != QKVP_SECTIONED) return QKVP_ERR_SHAPE;
  if (layout->n_q <= 0 || layout->n_kv <= 0 || layout->n_q % layout->n_kv) return QKVP_ERR_SHAPE;
  if (layout->head_dim != 64 && layout->head_dim != 128) return QKVP_ERR_SHAPE;
  if (count < 0 || count > (1 << 20)) return QKVP_ERR_SHAPE;
  *rows = ((int64_t)layout->n_q + 2 * (int64_t)layout->n_kv) * layout->head_dim * count;
  if (*rows > (1 << 30)) return QKVP_ERR_SHAPE;
  if (cols < 64 || cols % 64 != 0 || cols > (1 << 20)) return QKVP_ERR_SHAPE;
  if (split < 0 || split > kNsMaxSplit || split > cols / 64) return QKVP_ERR_SHAPE;
  return QKVP_OK;
}

bool overlaps(const void* p, size_t pn, const void* q, size_t qn) {
  const uintptr_t a = (uintptr_t)p, b = (uintptr_t)q;
  return a < b + qn && b < a + pn;
}

}  // namespace
}  // namespace qkvp

using namespace qkvp;

extern "C" {

int qkv_prologue_version(void) { return QKVP_VERSION; }

const char* qkv_prologue_status_string(int status) {
  switch (status) {
    case QKVP_OK: return "ok";
    case QKVP_ERR_NULL: return "a required pointer is NULL";
    case QKVP_ERR_SHAPE: return "invalid shape (T, head counts, head_dim, row_stride or layout kind)";
    case QKVP_ERR_ALIGN: return "a tensor is not 16-byte aligned (index tensors: 4-byte)";
    case QKVP_ERR_ARCH: return "no usable CUDA device, or the device is not sm_103";
    case QKVP_ERR_WORKSPACE: return "workspace missing or smaller than its size query gives";
    case QKVP_ERR_LAUNCH: return "CUDA launch failed";
    case QKVP_ERR_FLAGS: return "unknown or unsupported flag bits for this call";
    case QKVP_ERR_VALUE: return "invalid scalar (eps, rope_base, num_pages or page_size)";
    default: return "unknown status";
  }
}

// ------------------------------------------------------------- forward ----

static int gqa_forward(const qkvp_layout* L, const qkvp_variant* variant, int64_t T, const void* packed,
                       const int32_t* pos, const float* w_q, const float* w_k, float eps, double rope_base,
                       uint32_t flags, void* q, void* k, void* v, void* q_pre, void* k_pre,
                       const int32_t* page, const int32_t* offset, void* k_pool, void* v_pool,
                       int32_t num_pages, int32_t page_size, int32_t* dev_status, bool pool,
                       cudaStream_t stream) {
  Gqa g;
  QKVP_TRY(check_gqa(L, T, &g));
  const uint32_t allowed = (pool ? (uint32_t)QKVP_NOPE : (uint32_t)(QKVP_NOPE | QKVP_SAVE_PRE)) |
                           (uint32_t)(QKVP_FORCE_GENERIC | QKVP_NORM_OFF);
  if (flags & ~allowed) return QKVP_ERR_FLAGS;
  const bool rope = !(flags & QKVP_NOPE);
  const bool save = (flags & QKVP_SAVE_PRE) != 0;
  const bool norm = !(flags & QKVP_NORM_OFF);
  Variant vr;
  QKVP_TRY(check_variant(variant, L->head_dim, true, &vr));
  QKVP_TRY(check_scalars(eps, rope_base, rope && !vr.inv_freq));
  if (!packed || (norm && (!w_q || !w_k)) || !q || (rope && !pos)) return QKVP_ERR_NULL;
  if (pool) {
    if (!page || !offset || !k_pool || !v_pool) return QKVP_ERR_NULL;
    QKVP_TRY(check_pool(num_pages, page_size));
  } else {
    if (!k || !v) return QKVP_ERR_NULL;
    if (save && (!q_pre || !k_pre)) return QKVP_ERR_NULL;
  }
  const void* vec[] = {packed, norm ? w_q : nullptr, norm ? w_k : nullptr, q, pool ? k_pool : k,
                       pool ? v_pool : v, save ? q_pre : nullptr, save ? k_pre : nullptr};
  for (const void* p : vec)
    if (p && !aligned16(p)) return QKVP_ERR_ALIGN;
  if ((pos && !aligned4(pos)) || (page && !aligned4(page)) || (offset && !aligned4(offset)) ||
      (dev_status && !aligned4(dev_status)))
    return QKVP_ERR_ALIGN;
  if (T == 0) return QKVP_OK;

  int sms = 0, smem_per_sm = 0;
  QKVP_TRY(current_device(&sms, &smem_per_sm));
  FwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.packed = static_cast<const uint4*>(packed);
  a.row_stride16 = g.stride / 8;
  a.pos = pos;
  a.w_q = w_q;
  a.w_k = w_k;
  a.eps = eps;
  a.inv_head_dim = 1.0f / (float)L->head_dim;
  a.T = T;
  a.n_q = L->n_q;
  a.n_kv = L->n_kv;
  a.group = L->n_q / L->n_kv;
  a.cpt = g.heads * (L->head_dim / 8);
  a.cpt_magic = magic((uint32_t)a.cpt);
  a.gs_magic = magic((uint32_t)(a.group + 2));
  gqa_items(T, a.cpt, kFwdChunksPerThread, &a.item_chunks, &a.n_items, &a.max_tok);
  a.q = static_cast<uint4*>(q);
  a.k = static_cast<uint4*>(k);
  a.v = static_cast<uint4*>(v);
  a.q_pre = static_cast<uint4*>(q_pre);
  a.k_pre = static_cast<uint4*>(k_pre);
  a.page = page;
  a.offset = offset;
  a.k_pool = static_cast<uint4*>(k_pool);
  a.v_pool = static_cast<uint4*>(v_pool);
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.dev_status = dev_status;
  a.bias = vr.bias;
  if (rope) rope_table(rope_base, L->head_dim, vr.inv_freq, vr.scale, &a.rope);

  const FwdVariant var{L->head_dim, L->kind == QKVP_SECTIONED, rope, save, pool, norm, vr.bias != nullptr};
  const int bias_bytes = vr.bias ? a.cpt * 8 * (int)sizeof(float) : 0;
  size_t smem = 0;
  if (!(flags & QKVP_FORCE_GENERIC) &&
      stream_geometry(fwd_stream_shape(save, rope), a.cpt / 2, L->head_dim / 16, L->head_dim, T,
                      (int64_t)a.cpt * 16, smem_per_sm, 0, bias_bytes, false, kStreamMaxSteps, !norm, &a.sg, &smem) &&
      (a.err = device_error_word()) != nullptr) {
    a.sg.dense = g.stride == g.row;
    const void* kern = fwd_stream_kernel(var);
    const int threads = (fwd_stream_shape(save).warps + 1) * 32;
    const int bps = allow_smem(kern, smem) ? blocks_per_sm(kern, threads, smem) : 0;
    if (bps > 0) {
      const int64_t cap = (int64_t)sms * bps;
      return launch(kern, a.sg.n_tiles < cap ? a.sg.n_tiles : cap, threads, smem, stream, &a);
    }
  }
  const void* kern = fwd_kernel(var);
  smem = (size_t)a.max_tok * (L->head_dim / 2) * 2 * sizeof(float) + (size_t)a.max_tok * sizeof(int32_t);
  const int64_t cap = (int64_t)sms * std::max(1, blocks_per_sm(kern, kThreads, smem));
  const int64_t grid = a.n_items < cap ? a.n_items : cap;
  return launch(kern, grid, kThreads, smem, stream, &a);
}

static int latent_forward(const qkvp_layout* L, const qkvp_variant* variant, int64_t T, const void* rows,
                          const int32_t* pos, const float* w, float eps, double rope_base, uint32_t flags,
                          void* out, const int32_t* page, const int32_t* offset, void* pool,
                          int32_t num_pages, int32_t page_size, int32_t* dev_status,
                          bool to_pool, cudaStream_t stream) {
  Latent g;
  QKVP_TRY(check_latent(L, T, &g));
  if (flags & ~(uint32_t)(QKVP_NOPE | QKVP_FORCE_GENERIC)) return QKVP_ERR_FLAGS;
  const bool rope = !(flags & QKVP_NOPE);
  Variant vr;
  QKVP_TRY(check_variant(variant, L->rope_dim, false, &vr));
  QKVP_TRY(check_scalars(eps, rope_base, rope && !vr.inv_freq));
  if (!rows || !w || (rope && !pos)) return QKVP_ERR_NULL;
  if (to_pool) {
    if (!page || !offset || !pool) return QKVP_ERR_NULL;
    QKVP_TRY(check_pool(num_pages, page_size));
  } else if (!out) {
    return QKVP_ERR_NULL;
  }
  if (!aligned16(rows) || !aligned16(w) || (out && !aligned16(out)) || (pool && !aligned16(pool)))
    return QKVP_ERR_ALIGN;
  if ((pos && !aligned4(pos)) || (page && !aligned4(page)) || (offset && !aligned4(offset)) ||
      (dev_status && !aligned4(dev_status)))
    return QKVP_ERR_ALIGN;
  if (T == 0) return QKVP_OK;

  int sms = 0, smem_per_sm = 0;
  QKVP_TRY(current_device(&sms, &smem_per_sm));
  LatentArgs a;
  std::memset(&a, 0, sizeof(a));
  a.rows = static_cast<const uint4*>(rows);
  a.row_stride16 = g.stride / 8;
  a.pos = pos;
  a.w = w;
  a.eps = eps;
  a.inv_norm_dim = 1.0f / (float)L->norm_dim;
  a.T = T;
  a.norm_chunks = L->norm_dim / 8;
  a.row_chunks = (int32_t)(g.row / 8);
  a.out = static_cast<uint4*>(out);
  a.page = page;
  a.offset = offset;
  a.pool = static_cast<uint4*>(pool);
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.dev_status = dev_status;
  if (rope) rope_table(rope_base, L->rope_dim, vr.inv_freq, vr.scale, &a.rope);
  const int ncl = a.norm_chunks <= 32 ? 1 : (a.norm_chunks <= 64 ? 2 : 4);

  // Pipelined kernel: tiles of kLatentTileTokens rows, kLatentStreamCtasPerSm
  // CTAs per SM, each ring as deep as the shared memory allows (>= 2 stages).
  // Its table per stage holds the positions and the pool slots (layout of a
  // 2-wide "head": one int per row each).
  if (!(flags & QKVP_FORCE_GENERIC) && (a.err = device_error_word()) != nullptr) {
    const int tpt = kLatentTileTokens, thd = 2;
    const int64_t stage = (int64_t)tpt * a.row_chunks * 16;
    const int budget = smem_per_sm / kLatentStreamCtasPerSm - 1024;
    const int64_t per_stage = stage + StreamSmem::table_stride(thd, tpt);
    int64_t stages = (budget - StreamSmem::tables(thd) - 128) / per_stage;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages >= 2) {
      a.sg.tpt = tpt;
      a.sg.stages = (int32_t)stages;
      a.sg.steps = 1;
      a.sg.stage_bytes = (int32_t)stage;
      a.sg.n_tiles = (T + tpt - 1) / tpt;
      a.sg.dense = g.stride == g.row;
      const size_t smem = (size_t)StreamSmem::data(thd, tpt, (int)stages) + (size_t)stages * stage;
      const void* kern = latent_stream_kernel(to_pool, rope, ncl);
      const int threads = (kLatentStreamWarps + 1) * 32;
      const int bps = allow_smem(kern, smem) ? blocks_per_sm(kern, threads, smem) : 0;
      if (bps > 0) {
        const int64_t cap = (int64_t)sms * bps;
        return launch(kern, a.sg.n_tiles < cap ? a.sg.n_tiles : cap, threads, smem, stream, &a);
      }
    }
  }
  const void* kern = latent_kernel(to_pool, rope, ncl);
  const int threads = kLatentWarps * 32;
  const int64_t per_cta = (int64_t)kLatentWarps * kLatentTokensPerWarp;
  const int64_t need = (T + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)sms * std::max(1, blocks_per_sm(kern, threads, 0));
  return launch(kern, need < cap ? need : cap, threads, 0, stream, &a);
}

int qkv_prologue_fwd_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T, const void* packed,
                        const int32_t* pos, const float* w_q, const float* w_k, float eps, double rope_base,
                        uint32_t flags, void* q, void* k, void* v, void* q_pre, void* k_pre, void* stream) {
  if (!layout) return QKVP_ERR_NULL;
  if (layout->kind == QKVP_LATENT)
    return latent_forward(layout, variant, T, packed, pos, w_k, eps, rope_base, flags, k, nullptr, nullptr,
                          nullptr, 0, 0, nullptr, false, static_cast<cudaStream_t>(stream));
  return gqa_forward(layout, variant, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, k, v, q_pre, k_pre,
                     nullptr, nullptr, nullptr, nullptr, 0, 0, nullptr, false, static_cast<cudaStream_t>(stream));
}

int qkv_prologue_fwd(const qkvp_layout* layout, int64_t T, const void* packed, const int32_t* pos,
                     const float* w_q, const float* w_k, float eps, double rope_base,
                     uint32_t flags, void* q, void* k, void* v, void* q_pre, void* k_pre,
                     void* stream) {
  return qkv_prologue_fwd_ex(layout, nullptr, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, k, v, q_pre,
                             k_pre, stream);
}

int qkv_prologue_pool_write_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T,
                               const void* packed, const int32_t* pos, const float* w_q, const float* w_k,
                               float eps, double rope_base, uint32_t flags, void* q, const int32_t* page,
                               const int32_t* offset, void* k_pool, void* v_pool, int32_t num_pages,
                               int32_t page_size, int32_t* dev_status, void* stream) {
  if (!layout) return QKVP_ERR_NULL;
  if (layout->kind == QKVP_LATENT)
    return latent_forward(layout, variant, T, packed, pos, w_k, eps, rope_base, flags, nullptr, page, offset,
                          k_pool, num_pages, page_size, dev_status, true, static_cast<cudaStream_t>(stream));
  return gqa_forward(layout, variant, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, nullptr, nullptr,
                     nullptr, nullptr, page, offset, k_pool, v_pool, num_pages, page_size, dev_status, true,
                     static_cast<cudaStream_t>(stream));
}

int qkv_prologue_pool_write(const qkvp_layout* layout, int64_t T, const void* packed,
                            const int32_t* pos, const float* w_q, const float* w_k, float eps,
                            double rope_base, uint32_t flags, void* q, const int32_t* page,
                            const int32_t* offset, void* k_pool, void* v_pool, int32_t num_pages,
                            int32_t page_size, int32_t* dev_status, void* stream) {
  return qkv_prologue_pool_write_ex(layout, nullptr, T, packed, pos, w_q, w_k, eps, rope_base, flags, q, page,
                                    offset, k_pool, v_pool, num_pages, page_size, dev_status, stream);
}

int qkv_prologue_pool_scatter(const qkvp_layout* layout, int64_t T, const void* k_rows,
                              const void* v_rows, const int32_t* page, const int32_t* offset,
                              void* k_pool, void* v_pool, int32_t num_pages, int32_t page_size,
                              int32_t* dev_status, void* stream) {
  if (!layout) return QKVP_ERR_NULL;
  int64_t row = 0;
  const bool latent = layout->kind == QKVP_LATENT;
  if (latent) {
    Latent g;
    QKVP_TRY(check_latent(layout, T, &g));
    row = g.row;
  } else {
    Gqa g;
    QKVP_TRY(check_gqa(layout, T, &g));
    row = (int64_t)layout->n_kv * layout->head_dim;
  }
  if (!k_rows || !k_pool || !page || !offset) return QKVP_ERR_NULL;
  if (!latent && (!v_rows || !v_pool)) return QKVP_ERR_NULL;
  QKVP_TRY(check_pool(num_pages, page_size));
  if (!aligned16(k_rows) || !aligned16(k_pool) || (!latent && (!aligned16(v_rows) || !aligned16(v_pool))))
    return QKVP_ERR_ALIGN;
  if (!aligned4(page) || !aligned4(offset) || (dev_status && !aligned4(dev_status)))
    return QKVP_ERR_ALIGN;
  if (T == 0) return QKVP_OK;
  int sms = 0;
  QKVP_TRY(current_device(&sms));
  ScatterArgs a;
  std::memset(&a, 0, sizeof(a));
  a.src_a = static_cast<const uint4*>(k_rows);
  a.src_b = latent ? nullptr : static_cast<const uint4*>(v_rows);
  a.pool_a = static_cast<uint4*>(k_pool);
  a.pool_b = latent ? nullptr : static_cast<uint4*>(v_pool);
  a.T = T;
  a.row_chunks = (int32_t)(row / 8);
  a.page = page;
  a.offset = offset;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.dev_status = dev_status;
  const void* kern = scatter_kernel();
  const int64_t need = (T * a.row_chunks + 255) / 256;
  const int64_t cap = (int64_t)sms * std::max(1, blocks_per_sm(kern, 256, 0));
  return launch(kern, need < cap ? need : cap, 256, 0, static_cast<cudaStream_t>(stream), &a);
}

// ------------------------------------------------------------ backward ----

// Backward partial rows: one per CTA, at most max(work items, tokens), capped;
// each row holds [dw_q | dw_k] (norm on) then the bias row (bias given).
static int64_t bwd_row_floats(const qkvp_layout* layout, bool norm, bool bias) {
  const int64_t heads = (int64_t)layout->n_q + 2 * (int64_t)layout->n_kv;
  return (norm ? 2 * layout->head_dim : 0) + (bias ? heads * layout->head_dim : 0);
}

// Bytes of the partial rows; the workspace is these rows followed by
// kFoldBytes for the weight-gradient fold's arrival words (one per CTA, at
// most kMaxBwdParts) and its election word.
static size_t bwd_rows_bytes(const qkvp_layout* layout, const Variant& vr, bool norm, int64_t T) {
  Gqa g;
  if (check_gqa(layout, T, &g) != QKVP_OK || T == 0) return 0;
  int64_t item_chunks = 0, n_items = 0;
  int max_tok = 0;
  gqa_items(T, g.heads * (layout->head_dim / 8), kBwdChunksPerThread, &item_chunks, &n_items, &max_tok);
  return (size_t)bwd_parts(n_items > T ? n_items : T) * (size_t)bwd_row_floats(layout, norm, vr.bias != nullptr) *
         sizeof(float);
}

constexpr size_t kFoldBytes = 4 * (kMaxBwdParts + 4);

static size_t bwd_workspace(const qkvp_layout* layout, const Variant& vr, bool norm, int64_t T) {
  const size_t rows = bwd_rows_bytes(layout, vr, norm, T);
  return rows ? rows + kFoldBytes : 0;
}

// A new generation for the fold's arrival word on every call (never 0).
static uint32_t next_call_id() {
  static std::atomic<uint32_t> counter{0x9e3779b9u};
  uint32_t id = counter.fetch_add(1, std::memory_order_relaxed) + 1;
  return id ? id : counter.fetch_add(1, std::memory_order_relaxed) + 1;
}

size_t qkv_prologue_bwd_workspace_size(const qkvp_layout* layout, int64_t T) {
  return bwd_workspace(layout, Variant(), true, T);
}

size_t qkv_prologue_bwd_workspace_size_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T) {
  Variant vr;
  if (!layout || check_variant(variant, layout->head_dim, true, &vr) != QKVP_OK) return 0;
  // The size does not depend on the norm flag: a norm-off call needs less.
  return bwd_workspace(layout, vr, true, T);
}

int qkv_prologue_bwd_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T, const void* dq,
                        const void* dk, const void* dv, const void* q_pre, const void* k_pre, const int32_t* pos,
                        const float* w_q, const float* w_k, float eps, double rope_base, uint32_t flags,
                        void* dpacked, float* dw_q, float* dw_k, float* dbias, void* workspace,
                        size_t workspace_bytes, void* stream) {
  Gqa g;
  QKVP_TRY(check_gqa(layout, T, &g));
  if (flags & ~(uint32_t)(QKVP_NOPE | QKVP_ACCUMULATE_DW | QKVP_FORCE_GENERIC | QKVP_NORM_OFF))
    return QKVP_ERR_FLAGS;
  const bool rope = !(flags & QKVP_NOPE);
  const bool accumulate = (flags & QKVP_ACCUMULATE_DW) != 0;
  const bool norm = !(flags & QKVP_NORM_OFF);
  Variant vr;
  QKVP_TRY(check_variant(variant, layout->head_dim, true, &vr));
  const bool bias = vr.bias != nullptr;
  QKVP_TRY(check_scalars(eps, rope_base, rope && !vr.inv_freq));
  if (!dq || !dk || !dv || !dpacked || (rope && !pos)) return QKVP_ERR_NULL;
  if (norm && (!q_pre || !k_pre || !w_q || !w_k || !dw_q || !dw_k)) return QKVP_ERR_NULL;
  if (bias && !dbias) return QKVP_ERR_NULL;
  const void* vec[] = {dq, dk, dv, dpacked, norm ? q_pre : nullptr, norm ? k_pre : nullptr,
                       norm ? w_q : nullptr, norm ? w_k : nullptr, norm ? dw_q : nullptr,
                       norm ? dw_k : nullptr, bias ? dbias : nullptr};
  for (const void* p : vec)
    if (p && !aligned16(p)) return QKVP_ERR_ALIGN;
  if (pos && !aligned4(pos)) return QKVP_ERR_ALIGN;
  const int hd = layout->head_dim;
  const int cpt = g.heads * (hd / 8);
  if (bias && cpt > kBiasMaxChunks) return QKVP_ERR_SHAPE;
  const size_t need = bwd_workspace(layout, vr, norm, T);
  if (need > 0 && (!workspace || workspace_bytes < need)) return workspace ? QKVP_ERR_WORKSPACE : QKVP_ERR_NULL;
  if (workspace && !aligned16(workspace)) return QKVP_ERR_ALIGN;

  int sms = 0, smem_per_sm = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (T == 0) {
    if (accumulate || (!norm && !bias)) return QKVP_OK;
    QKVP_TRY(current_device(&sms));
    const size_t wbytes = (size_t)hd * sizeof(float), bbytes = (size_t)cpt * 8 * sizeof(float);
    if ((norm && (cudaMemsetAsync(dw_q, 0, wbytes, s) != cudaSuccess ||
                  cudaMemsetAsync(dw_k, 0, wbytes, s) != cudaSuccess)) ||
        (bias && cudaMemsetAsync(dbias, 0, bbytes, s) != cudaSuccess)) {
      cudaGetLastError();
      return QKVP_ERR_LAUNCH;
    }
    return QKVP_OK;
  }
  QKVP_TRY(current_device(&sms, &smem_per_sm));

  BwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.dq = static_cast<const uint4*>(dq);
  a.dk = static_cast<const uint4*>(dk);
  a.dv = static_cast<const uint4*>(dv);
  a.q_pre = static_cast<const uint4*>(q_pre);
  a.k_pre = static_cast<const uint4*>(k_pre);
  a.pos = pos;
  a.w_q = w_q;
  a.w_k = w_k;
  a.eps = eps;
  a.inv_head_dim = 1.0f / (float)hd;
  a.T = T;
  a.n_q = layout->n_q;
  a.n_kv = layout->n_kv;
  a.group = layout->n_q / layout->n_kv;
  a.cpt = cpt;
  a.cpt_magic = magic((uint32_t)a.cpt);
  a.gs_magic = magic((uint32_t)(a.group + 2));
  gqa_items(T, a.cpt, kBwdChunksPerThread, &a.item_chunks, &a.n_items, &a.max_tok);
  a.dpacked = static_cast<uint4*>(dpacked);
  a.row_stride16 = g.stride / 8;
  a.bias = vr.bias;
  if (rope) rope_table(rope_base, hd, vr.inv_freq, vr.scale, &a.rope);

  BwdVariant var{hd, layout->kind == QKVP_SECTIONED, rope, norm, bias, 0};
  const int64_t heads_qkv = norm ? (2 * layout->n_q + 3 * layout->n_kv) : (layout->n_q + 2 * layout->n_kv);
  const int64_t token_bytes = heads_qkv * hd * 2;
  const StreamShape shape = bwd_stream_shape();
  const int static_smem = (norm ? shape.warps : 1) * 2 * hd * (int)sizeof(float);
  const int bias_bytes = (norm && bias) ? cpt * 8 * (int)sizeof(float) : 0;
  size_t smem = 0;
  int64_t grid = 0;
  bool streamed = false;
  if (!(flags & QKVP_FORCE_GENERIC) &&
      stream_geometry(shape, a.cpt / 2, hd / 16, hd, T, token_bytes, smem_per_sm, static_smem, bias_bytes, bias,
                      bias ? kBiasMaxSteps : kStreamMaxSteps, true, &a.sg, &smem) &&
      (a.err = device_error_word()) != nullptr) {
    a.sg.dense = 1;
    var.steps = a.sg.steps;
    const void* kern = bwd_stream_kernel(var);
    const int threads = (shape.warps + 1) * 32;
    const int bps = allow_smem(kern, smem) ? blocks_per_sm(kern, threads, smem) : 0;
    if (bps > 0) {
      grid = (int64_t)sms * bps;
      if (grid > a.sg.n_tiles) grid = a.sg.n_tiles;
      if (grid > kMaxBwdParts) grid = kMaxBwdParts;
      streamed = true;
    }
  }
  const void* kern = nullptr;
  int threads = kThreads;
  if (streamed) {
    kern = bwd_stream_kernel(var);
    threads = (shape.warps + 1) * 32;
  } else {
    if (bias) {  // one token per work item: every thread keeps the same chunks
      a.item_chunks = a.cpt;
      a.n_items = T;
      a.max_tok = 1;
    }
    kern = bwd_kernel(var);
    smem = (size_t)a.max_tok * (hd / 2) * 2 * sizeof(float) + (bias ? (size_t)a.cpt * 8 * sizeof(float) : 0);
    if (!allow_smem(kern, smem)) return QKVP_ERR_LAUNCH;
    grid = (int64_t)sms * std::max(1, blocks_per_sm(kern, kThreads, smem));
    if (grid > a.n_items) grid = a.n_items;
    if (grid > kMaxBwdParts) grid = kMaxBwdParts;
  }
  float* ws = static_cast<float*>(workspace);
  a.partials = ws;
  a.db_partials = ws + (norm ? grid * 2 * hd : 0);
  // The pipelined kernel with the norm and no bias adds its own partial rows
  // (the last CTA to finish); otherwise the finalize kernel does.
  const bool fold = streamed && norm && !bias;
  if (fold) {
    a.flags = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(workspace) + bwd_rows_bytes(layout, vr, norm, T));
    a.call_id = next_call_id();
    a.accumulate = accumulate ? 1 : 0;
    a.dw_q = dw_q;
    a.dw_k = dw_k;
  }
  QKVP_TRY(launch(kern, grid, threads, smem, s, &a));
  if (fold || (!norm && !bias)) return QKVP_OK;

  FinalizeArgs f;
  std::memset(&f, 0, sizeof(f));
  f.partials = a.partials;
  f.db_partials = a.db_partials;
  f.nparts = (int32_t)grid;
  f.head_dim = hd;
  f.n_bias = bias ? cpt * 8 : 0;
  f.dw_q = norm ? dw_q : nullptr;
  f.dw_k = norm ? dw_k : nullptr;
  f.db = bias ? dbias : nullptr;
  f.accumulate = accumulate ? 1 : 0;
  const int n_out = (norm ? 2 * hd : 0) + f.n_bias;
  const int fgrid = (n_out + kFinalizeOutputsPerCta - 1) / kFinalizeOutputsPerCta;
  return launch(dw_finalize_kernel(), fgrid, kFinalizeThreads, 0, s, &f);
}

int qkv_prologue_bwd(const qkvp_layout* layout, int64_t T, const void* dq, const void* dk,
                     const void* dv, const void* q_pre, const void* k_pre, const int32_t* pos,
                     const float* w_q, const float* w_k, float eps, double rope_base,
                     uint32_t flags, void* dpacked, float* dw_q, float* dw_k, void* workspace,
                     size_t workspace_bytes, void* stream) {
  return qkv_prologue_bwd_ex(layout, nullptr, T, dq, dk, dv, q_pre, k_pre, pos, w_q, w_k, eps, rope_base, flags,
                             dpacked, dw_q, dw_k, nullptr, workspace, workspace_bytes, stream);
}

// ------------------------------------------- projection + prologue ----

int qkv_prologue_gemm_fwd(const qkvp_layout* layout, int64_t T, int32_t hidden, const void* x, const void* w_qkv,
                          const int32_t* pos, const float* w_q, const float* w_k, float eps, double rope_base,
                          uint32_t flags, void* q, void* k, void* v, void* q_pre, void* k_pre, void* stream) {
  Gqa g;
  QKVP_TRY(check_gqa(layout, T, &g));
  if (g.stride != g.row) return QKVP_ERR_SHAPE;  // W is [row width, hidden], dense
  if (hidden < 8 || hidden % 8 != 0 || T > INT32_MAX) return QKVP_ERR_SHAPE;
  if (flags & ~(uint32_t)(QKVP_NOPE | QKVP_SAVE_PRE)) return QKVP_ERR_FLAGS;
  const bool rope = !(flags & QKVP_NOPE), save = (flags & QKVP_SAVE_PRE) != 0;
  QKVP_TRY(check_scalars(eps, rope_base, rope));
  if (!x || !w_qkv || !w_q || !w_k || !q || !k || !v || (rope && !pos) || (save && (!q_pre || !k_pre)))
    return QKVP_ERR_NULL;
  const void* vec[] = {x, w_qkv, w_q, w_k, q, k, v, save ? q_pre : nullptr, save ? k_pre : nullptr};
  for (const void* p : vec)
    if (p && !aligned16(p)) return QKVP_ERR_ALIGN;
  if (pos && !aligned4(pos)) return QKVP_ERR_ALIGN;
  if (T == 0) return QKVP_OK;

  int sms = 0;
  QKVP_TRY(current_device(&sms));
  // The tensor maps must cover this GPU's own memory: x and w_qkv are read and
  // the outputs written by this GPU's tensor-memory-access (TMA) unit only.
  const void* dev_ptrs[] = {x, w_qkv, q, k, v, save ? q_pre : nullptr, save ? k_pre : nullptr};
  for (const void* ptr : dev_ptrs)
    if (ptr && !on_current_device(ptr)) return QKVP_ERR_VALUE;
  CUtensorMap tx, tw;
  if (!bf16_tile_map(&tx, x, T, hidden, kGemmBM) || !bf16_tile_map(&tw, w_qkv, g.heads * (int64_t)layout->head_dim,
                                                                    hidden, kGemmBN / 2))
    return QKVP_ERR_LAUNCH;
  GemmOutMaps om;
  const int64_t qcols = (int64_t)layout->n_q * layout->head_dim, kcols = (int64_t)layout->n_kv * layout->head_dim;
  if (!bf16_tile_map(&om.q, q, T, qcols, 32) || !bf16_tile_map(&om.k, k, T, kcols, 32) ||
      !bf16_tile_map(&om.v, v, T, kcols, 32) || !bf16_tile_map(&om.q_pre, save ? q_pre : q, T, qcols, 32) ||
      !bf16_tile_map(&om.k_pre, save ? k_pre : k, T, kcols, 32))
    return QKVP_ERR_LAUNCH;
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = T;
  a.hidden = hidden;
  a.n_q = layout->n_q;
  a.n_kv = layout->n_kv;
  a.group = layout->n_q / layout->n_kv;
  a.n_blocks = g.heads;
  a.gs_magic = magic((uint32_t)(a.group + 2));
  a.m_tiles = (int32_t)((T + 2 * kGemmBM - 1) / (2 * kGemmBM));
  a.n_tiles = (int32_t)((g.row + kGemmBN - 1) / kGemmBN);
  a.n_work = (int64_t)a.m_tiles * a.n_tiles;
  a.pos = pos;
  a.w_q = w_q;
  a.w_k = w_k;
  a.eps = eps;
  a.inv_head_dim = 1.0f / (float)layout->head_dim;
  a.q = static_cast<uint4*>(q);
  a.k = static_cast<uint4*>(k);
  a.v = static_cast<uint4*>(v);
  a.q_pre = static_cast<uint4*>(q_pre);
  a.k_pre = static_cast<uint4*>(k_pre);
  if ((a.err = device_error_word()) == nullptr) return QKVP_ERR_LAUNCH;
  if (rope) rope_table(rope_base, layout->head_dim, nullptr, 1.f, &a.rope);
  const void* kern = gemm_fwd_kernel(layout->head_dim, layout->kind == QKVP_SECTIONED, rope, save);
  const size_t smem = (size_t)gemm_fwd_smem_bytes();
  if (!allow_smem(kern, smem)) return QKVP_ERR_LAUNCH;
  const int threads = gemm_fwd_threads();
  const int clusters = max_clusters_of_2(kern, threads, smem);
  if (clusters < 1) return QKVP_ERR_LAUNCH;
  const int64_t grid = 2 * (a.n_work < clusters ? a.n_work : clusters);
  void* args[] = {&tx, &tw, &om, &a};
  return launch_args(kern, grid, threads, smem, static_cast<cudaStream_t>(stream), args, 2);
}

int qkv_newton_schulz_workspace(const qkvp_layout* layout, int64_t count, int64_t cols, int32_t split,
                                size_t* bytes) {
  using namespace qkvp;
  int64_t rows = 0;
  QKVP_TRY(check_ns(layout, count, cols, split, &rows));
  if (!bytes) return QKVP_ERR_NULL;
  if (count == 0) {
    *bytes = 0;
    return QKVP_OK;
  }
  const int64_t units = (rows + kNsUnitRows - 1) / kNsUnitRows;
  int sp = split;
  if (sp == 0) {
    int sms = 0;
    QKVP_TRY(current_device(&sms));
    sp = ns_split(units, (int)(cols / 64), 0, sms);
  }
  *bytes = ns_workspace_bytes(units, sp, layout->head_dim);
  return QKVP_OK;
}

int qkv_newton_schulz_batch(const qkvp_layout* layout, int64_t count, int64_t cols, const void* m, void* out,
                            int32_t split, void* workspace, size_t workspace_bytes, void* stream) {
  using namespace qkvp;
  int64_t rows = 0;
  QKVP_TRY(check_ns(layout, count, cols, split, &rows));
  if (!m || !out) return QKVP_ERR_NULL;
  if (!aligned16(m) || !aligned16(out)) return QKVP_ERR_ALIGN;
  const size_t bytes = (size_t)(rows * cols * 2);
  if (overlaps(m, bytes, out, bytes)) return QKVP_ERR_VALUE;

  if (count == 0) return QKVP_OK;
  int sms = 0;
  if (split == 0) QKVP_TRY(current_device(&sms));  // the planned split depends on the device
  const int64_t units = (rows + kNsUnitRows - 1) / kNsUnitRows;
  const int nb = (int)(cols / 64);
  const int sp = ns_split(units, nb, split, sms);
  const size_t need = ns_workspace_bytes(units, sp, layout->head_dim);
  if (!workspace || workspace_bytes < need) return QKVP_ERR_WORKSPACE;
  if (!aligned16(workspace)) return QKVP_ERR_ALIGN;
  if (overlaps(workspace, need, m, bytes) || overlaps(workspace, need, out, bytes)) return QKVP_ERR_VALUE;
  if (sms == 0) QKVP_TRY(current_device(&sms));

  CUtensorMap tm, to;
  if (!bf16_tile_map(&tm, m, rows, cols, kNsUnitRows) || !bf16_tile_map(&to, out, rows, cols, 32))
    return QKVP_ERR_LAUNCH;
  NsArgs a;
  std::memset(&a, 0, sizeof(a));
  a.rows = (int32_t)rows;
  a.cols = (int32_t)cols;
  a.head_dim = layout->head_dim;
  a.units = (int32_t)units;
  a.nb = nb;
  a.split = sp;
  a.scale = (float)std::sqrt(std::max(1.0, (double)layout->head_dim / (double)cols));
  a.eps = 1e-7f;
  a.partial = static_cast<float*>(workspace);
  a.mh = reinterpret_cast<uint4*>(static_cast<unsigned char*>(workspace) +
                                  ns_partial_bytes(units, sp, layout->head_dim));
  if ((a.err = device_error_word()) == nullptr) return QKVP_ERR_LAUNCH;
  const void* kg = ns_gram_kernel();
  const void* kp = ns_poly_kernel(layout->head_dim);
  const void* ky = ns_apply_kernel();
  if (!allow_smem(kg, ns_gram_smem_bytes()) || !allow_smem(kp, ns_poly_smem_bytes(layout->head_dim)) ||
      !allow_smem(ky, ns_apply_smem_bytes()))
    return QKVP_ERR_LAUNCH;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* gargs[] = {&tm, &a};
  QKVP_TRY(launch_args(kg, units * sp, ns_gram_threads(), ns_gram_smem_bytes(), st, gargs));
  void* pargs[] = {&a};
  QKVP_TRY(launch_args(kp, units, ns_poly_threads(), ns_poly_smem_bytes(layout->head_dim), st, pargs));
  const int64_t boxes = units * nb;
  void* yargs[] = {&tm, &to, &a};
  return launch_args(ky, boxes < sms ? boxes : sms, ns_apply_threads(), ns_apply_smem_bytes(), st, yargs);
}

int qkv_newton_schulz(const qkvp_layout* layout, int64_t cols, const void* m, void* out, int32_t split,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return qkv_newton_schulz_batch(layout, 1, cols, m, out, split, workspace, workspace_bytes, stream);
}

int qkv_newton_schulz_plan(const qkvp_layout* layout, int64_t count, int64_t cols, int32_t split,
                           int32_t* split_out, int32_t* grid_out) {
  using namespace qkvp;
  int64_t rows = 0;
  QKVP_TRY(check_ns(layout, count, cols, split, &rows));
  if (!split_out || !grid_out) return QKVP_ERR_NULL;
  if (count == 0) {
    *split_out = *grid_out = 0;
    return QKVP_OK;
  }
  int sms = 0;
  QKVP_TRY(current_device(&sms));
  const int64_t units = (rows + kNsUnitRows - 1) / kNsUnitRows;
  const int sp = ns_split(units, (int)(cols / 64), split, sms);
  *split_out = sp;
  *grid_out = (int32_t)(units * sp);
  return QKVP_OK;
}

int qkv_prologue_wait_selftest(void* stream) {
  using namespace qkvp;
  int sms = 0;
  QKVP_TRY(current_device(&sms));
  int* err = device_error_word();
  if (err == nullptr) return QKVP_ERR_LAUNCH;
  return launch(wait_selftest_kernel(), 1, 32, 0, static_cast<cudaStream_t>(stream), &err);
}

int qkv_prologue_device_error(int clear, int* value) {
  if (!value) return QKVP_ERR_NULL;
  int sms = 0;
  QKVP_TRY(current_device(&sms));
  return read_device_error(clear != 0, value) == 0 ? QKVP_OK : QKVP_ERR_LAUNCH;
}

}  // extern "C"
