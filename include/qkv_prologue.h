/*
 * qkv_prologue.h -- C ABI of the packed-QKV attention prologue for GB300 (sm_103a).
 *
 * The operation (sources: three pull-request pages; each entry point below
 * names the page and section that define it):
 *
 *   forward   packed projection row of one token
 *               -> split into heads (interleaved per KV group, or sectioned)
 *               -> per-head RMSNorm of q and k:  y = x / sqrt(mean(x^2) + eps) * w
 *               -> rotate-half RoPE of q and k (skipped on NoPE layers)
 *               -> contiguous q, k, v   (v is a bit copy)
 *                  or q contiguous + k, v written into a paged KV pool
 *   backward  gradients of q, k, v -> gradient of the packed row, written
 *             once in the packed layout, plus the two RMSNorm weight grads.
 *
 * RoPE convention: for i < D/2, inv_freq_i = rope_base^(-2 i / D),
 * theta = pos * inv_freq_i, and
 *     o_i       = y_i cos(theta) - y_{i+D/2} sin(theta)
 *     o_{i+D/2} = y_{i+D/2} cos(theta) + y_i sin(theta).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer except `layout` and `workspace_bytes`-style scalars is a
 *    DEVICE pointer. The caller owns every buffer; the library allocates no
 *    memory and never synchronises. Work is enqueued asynchronously on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) on the
 *    current CUDA device.
 *  - bf16 tensors are passed as `void*` (IEEE bfloat16 bit patterns),
 *    row-major, and must start on a 16-byte boundary. `row_stride` (in
 *    elements) must be a multiple of 8. Index tensors are int32, weights and
 *    weight gradients float32, 16-byte aligned.
 *  - Arguments are checked on the host before anything touches the device.
 *    On error nothing is enqueued and a negative qkvp_status is returned.
 *  - T == 0 is valid and enqueues nothing.
 *  - Outputs must not overlap inputs (results are undefined if they do).
 *  - Results are deterministic: the same inputs on the same device give the
 *    same bits, including the weight gradients (no float atomics).
 */
#ifndef QKV_PROLOGUE_H_
#define QKV_PROLOGUE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QKVP_API __attribute__((visibility("default")))
#else
#define QKVP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define QKVP_VERSION 3

/* Status codes (return values). */
typedef enum {
  QKVP_OK = 0,
  QKVP_ERR_NULL = -1,      /* a required pointer is NULL                       */
  QKVP_ERR_SHAPE = -2,     /* bad T / head counts / head_dim / row_stride       */
  QKVP_ERR_ALIGN = -3,     /* a tensor is not 16-byte aligned                   */
  QKVP_ERR_ARCH = -4,      /* no CUDA device, or the device is not sm_103       */
  QKVP_ERR_WORKSPACE = -5, /* workspace missing or smaller than required         */
  QKVP_ERR_LAUNCH = -6,    /* the CUDA runtime reported an error at launch      */
  QKVP_ERR_FLAGS = -7,     /* unknown or contradictory flag bits                */
  QKVP_ERR_VALUE = -8      /* eps < 0, rope_base <= 0, non-finite, pool sizes   */
} qkvp_status;

/* Packed layouts.
 *
 * QKVP_INTERLEAVED: a row is [n_kv groups][G + 2 slots][head_dim] with
 *   G = n_q / n_kv: slots 0..G-1 of group g are q heads g*G .. g*G+G-1, slot G
 *   is k head g, slot G+1 is v head g ("[muse_spark][perf] Split the packed
 *   qkv inside the q/k region", Problem 1: [T, 16 kv heads, 10, 64]).
 * QKVP_SECTIONED: a row is [n_q q heads | n_kv k heads | n_kv v heads], each
 *   head_dim wide ("[muon] Per-head Newton-Schulz for fused QKV projections",
 *   What this PR does).
 * Both hold exactly (n_q + 2 n_kv) * head_dim values per row, at row_stride.
 *
 * QKVP_LATENT: an MLA kv latent row of norm_dim + rope_dim values: the first
 *   norm_dim are RMSNorm-ed with one weight, the last rope_dim are rotated by
 *   rotate-half RoPE with no norm and no weight ("MLA DSpark: run each drafter
 *   layer's kv path beside its q path", Description). n_q, n_kv, head_dim are
 *   ignored; norm_dim must be a multiple of 8 and at most 1024, rope_dim 64.
 */
typedef enum { QKVP_INTERLEAVED = 0, QKVP_SECTIONED = 1, QKVP_LATENT = 2 } qkvp_layout_kind;

typedef struct {
  int32_t kind;       /* qkvp_layout_kind                                     */
  int32_t n_q;        /* query heads; a positive multiple of n_kv              */
  int32_t n_kv;       /* key/value heads (KV groups)                           */
  int32_t head_dim;   /* 64 or 128                                             */
  int64_t row_stride; /* elements between consecutive tokens' rows; 0 = dense  */
  int32_t norm_dim;   /* LATENT only (512 for the DSpark drafter)              */
  int32_t rope_dim;   /* LATENT only (64)                                      */
} qkvp_layout;

/* Flags. */
enum {
  QKVP_NOPE = 1,           /* NoPE layer: RMSNorm only, no rotation            */
  QKVP_SAVE_PRE = 2,       /* forward also writes the split pre-norm q and k   */
  QKVP_ACCUMULATE_DW = 4,  /* backward adds into dw_q / dw_k instead of writing */
  QKVP_FORCE_GENERIC = 8,  /* use the general kernels even where the
                              shared-memory pipelined ones apply (same output
                              bits; for A/B checks). The backward's weight-grad
                              sums may differ in rounding. */
  QKVP_NORM_OFF = 16       /* GQA layouts: no RMSNorm of q and k (split ->
                              RoPE only, the GQAttention variant of Llama 3 and
                              GPT-OSS). w_q / w_k may be NULL; the backward
                              reads neither q_pre nor k_pre and has no weight
                              gradients (dw_q / dw_k may be NULL, untouched). */
};

/* Options of the GQAttention variant (the *_ex entry points; NULL = none).
 *
 * "[muse_spark][perf] Split the packed qkv inside the q/k region" names the
 * follow-up: a split -> norm -> RoPE region in GQAttention for Llama 3, Qwen3
 * and GPT-OSS (GPT-OSS with a qkv bias). Those models scale their RoPE
 * frequencies (Llama 3's and YaRN's scalings) and YaRN multiplies cos and sin
 * by a factor; both only change the inputs below, the rotation is the same.
 *
 * inv_freq    HOST array of head_dim / 2 (LATENT: rope_dim / 2) float64
 *             frequencies replacing rope_base^(-2 i / D), or NULL. Finite.
 * rope_scale  factor on cos and sin (o = scale * R(theta) y); 0 means 1.
 * bias        DEVICE float32 [(n_q + 2 n_kv) * head_dim], 16-byte aligned, in
 *             the packed row's own order (the fused linear's output bias), or
 *             NULL. Added to every token's row before anything else: the norm
 *             (if on) sees x + b, and v becomes round(x + b) instead of a bit
 *             copy. q_pre / k_pre stay the input heads WITHOUT the bias; the
 *             backward adds it back. GQA layouts only.
 */
typedef struct {
  const double* inv_freq;
  double rope_scale;
  const float* bias;
} qkvp_variant;

/* Device-side status bits (pool writes): set with an atomic OR in
 * *dev_status when a token's page or offset is out of range; that token's
 * pool store is skipped, nothing traps. */
enum { QKVP_DEV_BAD_PAGE = 1, QKVP_DEV_BAD_OFFSET = 2 };

/* ---------------------------------------------------------------------------
 * qkv_prologue_fwd -- split + per-head RMSNorm + RoPE, contiguous outputs.
 *
 * Defines: "[muse_spark][perf] Split the packed qkv inside the q/k region",
 * Solution 1-3 and the after-diagram (split -> norm -> RoPE, copy v), and the
 * training note on the q norm kernel (it also writes the split q).
 *
 * layout      host pointer. INTERLEAVED or SECTIONED (GQA), or LATENT.
 * T           tokens (>= 0).
 * packed      bf16 [T, row_stride] (GQA) or [T, row_stride] latent rows.
 * pos         int32 [T] positions (any int32; ignored with QKVP_NOPE).
 * w_q, w_k    float32 [head_dim] RMSNorm weights of q and k heads. LATENT:
 *             w_k is the float32 [norm_dim] latent weight, w_q is ignored.
 * eps         RMSNorm epsilon (>= 0, added inside the square root).
 * rope_base   RoPE base (> 0).
 * flags       QKVP_NOPE | QKVP_SAVE_PRE (SAVE_PRE: GQA only) | QKVP_FORCE_GENERIC.
 * q           bf16 [T, n_q, head_dim] out.           LATENT: ignored.
 * k           bf16 [T, n_kv, head_dim] out.          LATENT: [T, norm_dim+rope_dim] out.
 * v           bf16 [T, n_kv, head_dim] out (copy).   LATENT: ignored.
 * q_pre,k_pre bf16 [T, n_q | n_kv, head_dim] out, only with QKVP_SAVE_PRE
 *             (bit copies of the input heads, for the backward).
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_fwd(const qkvp_layout* layout, int64_t T, const void* packed,
                     const int32_t* pos, const float* w_q, const float* w_k, float eps,
                     double rope_base, uint32_t flags, void* q, void* k, void* v,
                     void* q_pre, void* k_pre, void* stream);

/* ---------------------------------------------------------------------------
 * qkv_prologue_pool_write -- the forward with a paged-pool destination.
 *
 * Defines: "MLA DSpark: run each drafter layer's kv path beside its q path",
 * Description (the norm/RoPE kernel stores rows straight into the pool at
 * the given pages / offsets, with no staging buffer and no scatter) and Test
 * Coverage (the direct write equals the staged path + scatter, bit for bit:
 * qkv_prologue_fwd followed by qkv_prologue_pool_scatter).
 *
 * GQA layouts: q is written contiguous [T, n_q, head_dim]; the normed (+roped)
 *   k heads of token t go to k_pool[page[t], offset[t]] and its raw v heads to
 *   v_pool[page[t], offset[t]]; pools are bf16 [num_pages, page_size, n_kv,
 *   head_dim].
 * LATENT: the normed/roped row of token t goes to k_pool[page[t], offset[t]]
 *   of a bf16 [num_pages, page_size, norm_dim + rope_dim] pool; q, v_pool and
 *   w_q are ignored (may be NULL).
 * page, offset  int32 [T]. A token whose page is outside [0, num_pages) or
 *   offset outside [0, page_size) is not stored; the matching QKVP_DEV_* bit
 *   is OR-ed into *dev_status when dev_status (int32, device) is not NULL.
 * Two tokens naming the same slot race; the caller must not do that.
 * flags: QKVP_NOPE, QKVP_FORCE_GENERIC.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_pool_write(const qkvp_layout* layout, int64_t T, const void* packed,
                            const int32_t* pos, const float* w_q, const float* w_k, float eps,
                            double rope_base, uint32_t flags, void* q, const int32_t* page,
                            const int32_t* offset, void* k_pool, void* v_pool,
                            int32_t num_pages, int32_t page_size, int32_t* dev_status,
                            void* stream);

/* ---------------------------------------------------------------------------
 * qkv_prologue_pool_scatter -- the staged write's scatter step.
 *
 * Defines the "staged scatter write" that "MLA DSpark: run each drafter
 * layer's kv path beside its q path" (Test Coverage) compares the direct pool
 * write against. Copies contiguous rows into pool slots, bit for bit:
 * GQA: k_rows, v_rows bf16 [T, n_kv, head_dim] -> k_pool, v_pool slots.
 * LATENT: k_rows bf16 [T, norm_dim + rope_dim] -> k_pool slots (v ignored).
 * Index checks and dev_status as for qkv_prologue_pool_write.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_pool_scatter(const qkvp_layout* layout, int64_t T, const void* k_rows,
                              const void* v_rows, const int32_t* page, const int32_t* offset,
                              void* k_pool, void* v_pool, int32_t num_pages, int32_t page_size,
                              int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------
 * qkv_prologue_bwd_workspace_size -- bytes of device workspace that
 * qkv_prologue_bwd needs for this layout and T on the CURRENT device
 * (0 when T == 0; returns 0 for an invalid layout).
 * ------------------------------------------------------------------------- */
QKVP_API size_t qkv_prologue_bwd_workspace_size(const qkvp_layout* layout, int64_t T);

/* ---------------------------------------------------------------------------
 * qkv_prologue_bwd -- one-pass backward writing the packed gradient.
 *
 * Defines: "[muse_spark][perf] Split the packed qkv inside the q/k region",
 * TLDR and Solution 3 (the norm-backward kernels write the packed grad; no
 * cat) and Results / Numerics (weight grads unchanged by the fusion).
 *
 * dq      bf16 [T, n_q, head_dim]   gradient of the forward's q output.
 * dk, dv  bf16 [T, n_kv, head_dim]  gradients of k and v.
 * q_pre, k_pre  bf16 split pre-norm heads saved by the forward (QKVP_SAVE_PRE).
 * pos, w_q, w_k, eps, rope_base, flags(QKVP_NOPE) as in the forward.
 * dpacked bf16 [T, row_stride] out, in the layout's packing: q/k slots get
 *         the RMSNorm+RoPE input gradient, v slots get dv unchanged.
 * dw_q, dw_k  float32 [head_dim] out: sum over tokens and heads of the weight
 *         gradient. Overwritten, or added to with QKVP_ACCUMULATE_DW.
 * workspace   device scratch of at least qkv_prologue_bwd_workspace_size
 *         bytes (any contents; 16-byte aligned); QKVP_ERR_WORKSPACE if smaller.
 *         It holds per-CTA partial sums of the weight gradients and, at its
 *         end, one arrival word per CTA and an election word: the CTA of the
 *         backward kernel that finishes last adds the partial rows (fixed
 *         order: deterministic) into dw_q, dw_k itself. The words need no
 *         clearing (each call tags them with its own generation). Two calls
 *         whose work can overlap on the GPU must not share a workspace.
 * GQA layouts only.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_bwd(const qkvp_layout* layout, int64_t T, const void* dq, const void* dk,
                     const void* dv, const void* q_pre, const void* k_pre, const int32_t* pos,
                     const float* w_q, const float* w_k, float eps, double rope_base,
                     uint32_t flags, void* dpacked, float* dw_q, float* dw_k, void* workspace,
                     size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * qkv_prologue_bwd_noalloc -- qkv_prologue_bwd without a caller workspace.
 *
 * The pages have no counterpart to this call: it exists for callers of this
 * library that may not allocate device memory and have no buffer to lend,
 * e.g. a plugin in an engine that owns all device memory through its own
 * pool, or a latency-critical loop where cudaMalloc (which can synchronise
 * the device) is not allowed. Same arguments, results and errors as
 * qkv_prologue_bwd, minus the workspace: the weight-gradient partial sums go
 * to a fixed 520 KiB array inside the library's device memory, which every
 * GPU that loads the library holds until the process exits.
 *  - Limit: with the norm on, qkv_prologue_bwd_workspace_size(layout, T)
 *    must be <= 520 KiB, otherwise QKVP_ERR_WORKSPACE is returned and nothing
 *    is enqueued. That size is min(1024, max(T, n_items)) partial rows of
 *    2 * head_dim floats plus 4112 bytes of arrival words, n_items =
 *    ceil(T * (n_q + 2 n_kv) * head_dim / 8 / 1536): head_dim 64 always fits
 *    (at most 1024 rows of 512 B); head_dim 128 fits while max(T, n_items)
 *    <= 515 (e.g. n_q 32, n_kv 8: 515 tokens; n_q 128, n_kv 16: 309 tokens).
 *    With QKVP_NORM_OFF no scratch is needed and every T is accepted.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture. The cache outlives a cudaDeviceReset: do not use this
 *    call on a device after resetting it in the same process.
 *  - All calls share the array and it keeps the last call's contents (nothing
 *    in it needs to start at zero). Calls whose work can overlap on the GPU
 *    (different streams without ordering) race on it: order them.
 *  - Allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_bwd_noalloc(const qkvp_layout* layout, int64_t T, const void* dq,
                                      const void* dk, const void* dv, const void* q_pre,
                                      const void* k_pre, const int32_t* pos, const float* w_q,
                                      const float* w_k, float eps, double rope_base, uint32_t flags,
                                      void* dpacked, float* dw_q, float* dw_k, void* stream);

/* ---------------------------------------------------------------------------
 * The *_ex entry points: the calls above with a qkvp_variant (may be NULL,
 * which gives exactly the plain call). Same arguments, errors and results
 * otherwise; flags may also hold QKVP_NORM_OFF (GQA layouts).
 *
 * qkv_prologue_bwd_ex also takes
 * dbias   float32 [(n_q + 2 n_kv) * head_dim] out, required when the variant
 *         has a bias (else ignored): the bias gradient, dpacked's values (in
 *         float32, before rounding to bf16) summed over tokens in float32 in a
 *         fixed order. Overwritten, or added to with QKVP_ACCUMULATE_DW.
 *         With a bias the backward needs (n_q + 2 n_kv) * head_dim <= 12288
 *         (QKVP_ERR_SHAPE beyond).
 * Its workspace size is qkv_prologue_bwd_workspace_size_ex (larger with a
 * bias: one float row of the bias length per CTA).
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_fwd_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T,
                                 const void* packed, const int32_t* pos, const float* w_q,
                                 const float* w_k, float eps, double rope_base, uint32_t flags,
                                 void* q, void* k, void* v, void* q_pre, void* k_pre, void* stream);

QKVP_API int qkv_prologue_pool_write_ex(const qkvp_layout* layout, const qkvp_variant* variant,
                                        int64_t T, const void* packed, const int32_t* pos,
                                        const float* w_q, const float* w_k, float eps,
                                        double rope_base, uint32_t flags, void* q,
                                        const int32_t* page, const int32_t* offset, void* k_pool,
                                        void* v_pool, int32_t num_pages, int32_t page_size,
                                        int32_t* dev_status, void* stream);

QKVP_API size_t qkv_prologue_bwd_workspace_size_ex(const qkvp_layout* layout,
                                                   const qkvp_variant* variant, int64_t T);

QKVP_API int qkv_prologue_bwd_ex(const qkvp_layout* layout, const qkvp_variant* variant, int64_t T,
                                 const void* dq, const void* dk, const void* dv, const void* q_pre,
                                 const void* k_pre, const int32_t* pos, const float* w_q,
                                 const float* w_k, float eps, double rope_base, uint32_t flags,
                                 void* dpacked, float* dw_q, float* dw_k, float* dbias,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * qkv_prologue_gemm_fwd -- the wqkv projection with the prologue fused into its
 * epilogue: packed = x . w_qkv^T (bf16 inputs, fp32 accumulation on the tensor
 * cores), rounded to bf16 exactly as the packed tensor of the unfused path,
 * then split, normed and roped into q, k, v (and q_pre, k_pre) as
 * qkv_prologue_fwd does; the packed tensor itself is never written.
 *
 * Defines: the step just before the prologue, "[muse_spark][perf] Split the
 * packed qkv inside the q/k region", Problem 1 (the packed tensor is the wqkv
 * projection's output) and Solution 1 (the region starts at that output).
 *
 * layout   GQA layout (INTERLEAVED or SECTIONED), row_stride 0 (dense). Its
 *          packed row order is the row order of w_qkv.
 * hidden   K: columns of x and of w_qkv, a multiple of 8.
 * x        bf16 [T, hidden] row-major (the input of the projection).
 * w_qkv    bf16 [(n_q + 2 n_kv) * head_dim, hidden] row-major (nn.Linear's
 *          weight layout).
 * pos, w_q, w_k, eps, rope_base: as qkv_prologue_fwd.
 * flags    QKVP_NOPE, QKVP_SAVE_PRE (q_pre, k_pre = the bf16 packed heads).
 * q, k, v, q_pre, k_pre: as qkv_prologue_fwd (contiguous outputs).
 * x and w_qkv must be device memory of the current device (cudaMalloc or a
 * caching allocator on it): the kernel reads them through tensor maps of this
 * GPU's memory, so another GPU's memory (peer access), host or managed memory
 * gives QKVP_ERR_VALUE. The call is for one-GPU use: each GPU of a multi-GPU
 * job calls it on its own data.
 * The summation order of the projection differs from other GEMM libraries,
 * so a packed value sitting on a bf16 rounding boundary can round the other
 * way than in an unfused cuBLAS + qkv_prologue_fwd pair.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_gemm_fwd(const qkvp_layout* layout, int64_t T, int32_t hidden, const void* x,
                                   const void* w_qkv, const int32_t* pos, const float* w_q, const float* w_k,
                                   float eps, double rope_base, uint32_t flags, void* q, void* k, void* v,
                                   void* q_pre, void* k_pre, void* stream);

/* ---------------------------------------------------------------------------
 * qkv_newton_schulz -- per-head Newton-Schulz of a fused QKV weight's update.
 *
 * Defines: "[muon] Per-head Newton-Schulz for fused QKV projections"
 * (DeepSpeed), What this PR does: dim 0 of a fused weight
 * [(n_q + 2 n_kv) * head_dim, in_features] is cut into head_dim-row blocks,
 * which are the same blocks in the sectioned and the interleaved packing (so
 * `layout->kind` does not change the result, only the row count is taken from
 * it); every block G is replaced by NS(G) * max(1, head_dim / in_features)^0.5,
 * where NS is Muon's published quintic Newton-Schulz iteration:
 *     X = G / (||G||_F + 1e-7);  5 times:  A = X X^T,  X = a X + (b A + c A A) X
 * with (a, b, c) = (3.4445, -4.7750, 2.0315).
 *
 * Evaluation: every matrix of the iteration is a polynomial in the block's
 * Gram matrix A_0 = X X^T (P_k = a I + b A_k + c A_k^2, A_{k+1} = P_k A_k P_k),
 * so the result is M X with M = P_4 P_3 P_2 P_1 P_0: three kernels, one pass
 * over m for the Gram matrices, the five steps on head_dim x head_dim
 * matrices, one pass over m to apply M. The same function of G as the
 * iteration; only the rounding differs.
 * Arithmetic: tensor-core products with fp32 accumulation whose matrix
 * operands are each held as the sum of two bf16 numbers (about 16 significant
 * bits; three bf16 MMAs per product), norms and sums in fp32. The result is
 * much closer to the exact iteration than the published bf16 iteration (whose
 * own distance from it is 1-2 % in relative Frobenius norm per block).
 * Deterministic: the same inputs and split give the same bits.
 *
 * layout     INTERLEAVED or SECTIONED; n_q, n_kv, head_dim (64 or 128) give
 *            the rows; row_stride is not used.
 * cols       in_features: a multiple of 64, at most 2^20.
 * m          bf16 [rows, cols] row-major (the update: gradient or momentum).
 * out        bf16 [rows, cols] row-major; must not overlap m (QKVP_ERR_VALUE).
 * split      0: the library picks how many CTAs share the Gram pass of one
 *            128-row unit (each a contiguous range of 64-column boxes; the
 *            fp32 partials are summed in a fixed order); else that number,
 *            at most min(64, cols / 64) (QKVP_ERR_SHAPE otherwise). The bits
 *            of the result depend on it.
 * workspace  device memory of at least qkv_newton_schulz_workspace() bytes
 *            for the same arguments, 16-byte aligned, any contents, not
 *            overlapping m or out (QKVP_ERR_WORKSPACE if missing or smaller,
 *            QKVP_ERR_ALIGN, QKVP_ERR_VALUE). Owned by the caller; it must not
 *            be used by anything else until the launches are done.
 * The three kernels are queued on `stream` and return at once. A wait that
 * times out inside a kernel sets bit 1 of the device error word
 * (qkv_prologue_device_error); the output is then invalid.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_newton_schulz(const qkvp_layout* layout, int64_t cols, const void* m, void* out,
                               int32_t split, void* workspace, size_t workspace_bytes, void* stream);

/* The same for `count` fused updates of one shape stacked along dim 0
 * (m and out: bf16 [count, rows, cols], contiguous), in one set of launches:
 * the optimizer step of every layer at once. Head blocks are independent and
 * the factor depends only on head_dim and cols, so the stack is one taller
 * weight of count * (n_q + 2 n_kv) blocks. count 0 enqueues nothing;
 * otherwise as qkv_newton_schulz (count * rows at most 2^30). */
QKVP_API int qkv_newton_schulz_batch(const qkvp_layout* layout, int64_t count, int64_t cols, const void* m,
                                     void* out, int32_t split, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* Workspace bytes qkv_newton_schulz_batch needs for these arguments (count 0:
 * 0): ceil(count rows / 128) * (split * 128 * (head_dim + 4) * 4 + 65536). Host
 * only; with split 0 it plans the split for the current device. */
QKVP_API int qkv_newton_schulz_workspace(const qkvp_layout* layout, int64_t count, int64_t cols, int32_t split,
                                         size_t* bytes);

/* The split and the Gram pass's grid qkv_newton_schulz_batch would use for
 * these arguments (host only, nothing is launched; count 0 gives 0, 0). */
QKVP_API int qkv_newton_schulz_plan(const qkvp_layout* layout, int64_t count, int64_t cols, int32_t split,
                                    int32_t* split_out, int32_t* grid_out);

/* ---------------------------------------------------------------------------
 * qkv_prologue_device_error -- read (and with clear != 0, reset) the
 * library's device error word on the current device. Bit 1 means a
 * pipelined kernel's bounded wait on its shared-memory pipeline gave up
 * (after 2 s) and the kernel returned early: the results of that launch are
 * invalid. Synchronises with the device (it copies the word to the host).
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_device_error(int clear, int* value);

/* ---------------------------------------------------------------------------
 * qkv_prologue_wait_selftest -- exercises the library's bounded wait on the
 * current device: enqueues on `stream` one single-thread kernel whose only wait
 * (an mbarrier phase that nothing completes) gives up after the library's limit
 * (2 s), sets bit 1 of the device error word (qkv_prologue_device_error) and
 * returns. Every pipelined kernel waits the same way; this lets a test make a
 * wait run out without faulting or hanging the GPU. Not an operation of the
 * pages. Returns when the kernel is enqueued.
 * ------------------------------------------------------------------------- */
QKVP_API int qkv_prologue_wait_selftest(void* stream);

/* Static, human-readable text for a qkvp_status value. */
QKVP_API const char* qkv_prologue_status_string(int status);

/* QKVP_VERSION of the compiled library. */
QKVP_API int qkv_prologue_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QKV_PROLOGUE_H_ */
