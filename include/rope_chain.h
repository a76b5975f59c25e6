/*
 * rope_chain.h -- C ABI of librope_chain.so: the speculative draft's context
 * K/V chain (MuseSparkDSparkModel.precompute_and_store_context_kv) on one
 * GB300 GPU (sm_103a).
 *
 * The chain, per context row t of width D = 8192 and draft layer l < L:
 *   1. hidden RMSNorm of x[t], rounded to bf16                 rc_context_norms
 *   2. layer l's input RMSNorm of that, stacked into [L, T, D]  rc_context_norms
 *   3. K/V projection [L, T, D] x [L, D, 2*H*64]                rc_kv_project
 *   4. weightless K-norm of every 64-wide key head, GPT-J RoPE,
 *      and the slot-mapped insert of K and V into paged caches  rc_kv_store
 *
 * Sources, cited by web page title and symbol:
 *   [ctx] "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.draft.context"
 *   [rt]  "vllm.models.muse_spark.nvidia.specialized_decode.runtime.draft"
 *   [bnd] "vllm.models.muse_spark.nvidia.specialized_decode.cutedsl.common.draft_boundary"
 *
 * Conventions for every call:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never frees or retains them.  Pointer ARRAYS (slots, caches) are HOST
 *     arrays of device pointers, read during the call only.  A pointer
 *     to an INPUT may also be the device address of page-locked host memory
 *     (rc_device_address): the kernels then read it over the host link
 *     (NVLink-C2C on GB300) with no staging copy.  The host memory must
 *     stay allocated and unchanged until the stream has passed the call.
 *   - bf16 values travel as uint16_t bit patterns.
 *   - Work is enqueued on `stream`; calls do not synchronise and do not
 *     allocate device memory, so they can be issued inside CUDA graph
 *     capture.  Outputs are valid once the stream reaches that point.
 *   - Arguments are checked on the host before anything is launched; a
 *     rejected call returns RC_ERR_INVALID_ARG or RC_ERR_UNSUPPORTED, leaves
 *     every buffer untouched, and rc_last_error() says why.
 *   - Floating point: FP32 arithmetic with the rounding points of [ctx]
 *     (each product, sum and fma rounded to nearest even; nothing fused
 *     beyond the fma the pages write); 1/sqrt is the correctly rounded
 *     IEEE sqrt then divide (the pages use a hardware approximation).
 *     Subnormals are kept.
 */
#ifndef ROPE_CHAIN_H
#define ROPE_CHAIN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RC_OK = 0,
    RC_ERR_INVALID_ARG = 1,   /* malformed argument: null, misaligned, out of range */
    RC_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels cover */
    RC_ERR_CUDA = 3           /* a CUDA runtime call or launch failed */
} rc_status;

/* Weight layouts accepted by rc_kv_project. */
typedef enum {
    RC_W_KN = 0,   /* W[L, D, N]: N contiguous (the projection as x @ W) */
    RC_W_NK = 1    /* W[L, N, D]: D contiguous (nn.Linear layout; [rt]
                      ContextKV._project multiplies by its transpose) */
} rc_weight_layout;

/* Message of the last failed call on this host thread ("" if none). */
const char *rc_last_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int32_t rc_version(void);

/*
 * rc_context_norms -- steps 1 and 2.  [ctx] ContextNorms / _ContextNormsKernel,
 * [rt] ContextKV._project (the stack), [bnd] boundary_fragments (norm order).
 *
 *   z[t]      = bf16( hidden_norm(x[t]) )
 *   out[l, t] = bf16( pre_norm_l(z[t]) )         for l < L
 * with norm(v)_c = (v_c * r) * gamma_c (or v_c * r when the weight is NULL),
 * r = 1 / sqrt(fma(sum_c v_c^2, 1/D, eps)), the sum in a fixed documented
 * order (thread t of 256 holds columns 2048k + 8t + i; in-thread (k, i)
 * order; xor butterfly over each warp; the 8 warp sums left to right).
 *
 *   x         bf16 [T, D] row-major, contiguous, 16-byte aligned
 *   T         rows, 0 <= T < 2^31 (T == 0: nothing is launched)
 *   D         must be 8192 (the single-tile row norm); else RC_ERR_UNSUPPORTED
 *   hidden_w  bf16 [D] hidden-norm weight, 16-byte aligned, or NULL (weightless)
 *   pre_w     bf16 [L, D] layer input-norm weights, 16-byte aligned, or NULL
 *   L         layers, 1 <= L <= 64
 *   eps       shared by both norms
 *   out       bf16 [L, T, D] contiguous, 16-byte aligned; must not overlap x
 */
rc_status rc_context_norms(const uint16_t *x, int64_t T, int32_t D,
                           const uint16_t *hidden_w, const uint16_t *pre_w,
                           int32_t L, float eps, uint16_t *out,
                           cudaStream_t stream);

/*
 * rc_context_norms_ex -- steps 1 and 2 with every option of [ctx]
 * ContextNormConstants and ContextNorms: each norm's weight absent, bf16 or
 * FP32; the weight scaling the norm's input (before the sum of squares) or
 * its output; a gain center added to each weight element; and each norm's
 * own eps ([ctx] ContextNorms takes hidden_eps and pre_eps).
 *
 * For one norm with weight w, gamma_c = w_c + center (w_c itself when the
 * center is 0, so a -0.0 weight keeps its sign), and
 *   input scale:   u_c = gamma_c * v_c,  y_c = u_c * r(u)
 *   output scale:  y_c = (v_c * r(v)) * gamma_c
 *   no weight:     y_c = v_c * r(v)
 * with r(u) = 1 / sqrt(fma(sum_c u_c^2, 1/D, eps)) in the order of
 * rc_context_norms ([bnd] boundary_fragments writes both scale sides in this
 * order).  z = bf16(hidden norm of x); out[l, t] = bf16(layer l's norm of z),
 * an input-scale layer weight giving each layer its own r.
 *
 *   x, T, D, L, out   as rc_context_norms
 *   hidden, pre       HOST pointers to the two norms' parameters, read during
 *                     the call; hidden->weight is [D], pre->weight [L, D]
 *                     (device, 16-byte aligned, NULL exactly when
 *                     weight_dtype is RC_NORM_NONE; input_scale and
 *                     gain_center of a weightless norm are ignored)
 * Errors: RC_ERR_INVALID_ARG for a NULL or misaligned pointer, an unknown
 * weight_dtype or a weight/dtype mismatch; RC_ERR_UNSUPPORTED for D != 8192.
 */
typedef enum {
    RC_NORM_NONE = 0,   /* weightless norm */
    RC_NORM_BF16 = 1,   /* bf16 weight (uint16_t bit patterns) */
    RC_NORM_F32 = 2     /* FP32 weight */
} rc_norm_weight;

typedef struct {
    const void *weight;     /* device pointer, or NULL with RC_NORM_NONE */
    int32_t weight_dtype;   /* rc_norm_weight */
    int32_t input_scale;    /* non-zero: the weight scales the norm's input */
    float gain_center;      /* added to each weight element when non-zero */
    float eps;              /* this norm's eps */
} rc_norm_params;

rc_status rc_context_norms_ex(const uint16_t *x, int64_t T, int32_t D,
                              const rc_norm_params *hidden, const rc_norm_params *pre,
                              int32_t L, uint16_t *out, cudaStream_t stream);

/*
 * rc_kv_project -- step 3.  [rt] ContextKV._project
 * (torch.bmm(per_layer, stacked_kv_weight.transpose(1, 2))).
 *
 *   out[l, t, n] = bf16( sum_k normed[l, t, k] * W_l[k, n] )
 * BF16 inputs, FP32 accumulation on the tensor cores (tcgen05), one
 * rounding to bf16 at the end.  The summation order is the kernel's, so
 * results agree with an exact sum to within bf16 rounding plus FP32
 * accumulation error, not bit for bit.
 *
 *   normed     bf16 [L, T, D] contiguous, 16-byte aligned
 *   W          bf16 weights in `w_layout`, contiguous, 16-byte aligned
 *   w_layout   RC_W_KN or RC_W_NK
 *   out        bf16 [L, T, N] contiguous, 16-byte aligned
 *   L          1 <= L <= 4096;  T: 0 <= T <= 8388480 (T == 0: no launch)
 *   D          multiple of 64, >= 64;  N: multiple of 128, >= 128
 *   workspace  optional device scratch for split-K (16-byte aligned) and its
 *              size in bytes; NULL/0 runs without split-K.  For few output
 *              tiles the K dimension is split across CTAs and the FP32
 *              partial sums are added in split order by a second kernel
 *              (deterministic for a given workspace size).  With many
 *              tiles whose last round would leave most SMs idle, the last
 *              layer's final row blocks are split the same way in a launch
 *              of their own.  From eight rounds of tiles the persistent
 *              kernel's CTA pairs take their tiles in order from a 4-byte
 *              counter in the workspace (zeroed by the call), so the pairs
 *              that read the same rows of `normed` stay in step and share
 *              them in L2 (with a fixed tile order they drift apart and read
 *              them from DRAM again).  The tile order does not change the
 *              results.  The bytes that give all of this are
 *              rc_kv_project_workspace_size(); calls sharing one workspace
 *              must not overlap on the GPU.
 */
rc_status rc_kv_project(const uint16_t *normed, const uint16_t *W,
                        int32_t w_layout, uint16_t *out, int32_t L, int64_t T,
                        int32_t D, int32_t N, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes rc_kv_project uses at most for these sizes on the current
   device (0 when it would split nothing).  Host-only apart from one device
   attribute query; returns 0 for invalid sizes. */
size_t rc_kv_project_workspace_size(int32_t L, int64_t T, int32_t D, int32_t N);

/* The same figure for a GPU with num_sms streaming multiprocessors, with no
   device involved (plan allocations ahead of time, or for another GPU).
   Host-only; returns 0 for invalid sizes or num_sms < 1. */
size_t rc_kv_project_workspace_size_sms(int32_t L, int64_t T, int32_t D, int32_t N,
                                        int32_t num_sms);

/* How rc_kv_project (and rc_kv_project_store) run these sizes on a GPU with
   num_sms SMs given workspace_bytes of workspace.  Host-only.
     kernel          0: single CTAs (128-row tiles), 1: CTA pairs, one tile
                     each (256 x 256), 2: persistent CTA pairs walking the tiles
     splits          K splits of the main launch (1: none; > 1: FP32 partials
                     in the workspace, then a reduction launch)
     tail_splits     persistent plans: 0 without a tail launch; else the K
                     splits of the last layer's final row blocks, run as a
                     launch of their own (plus their reduction)
     tail_row0       the first of those rows (T without a tail launch)
     dynamic_tiles   persistent plans: 1 when the pairs take tiles in order
                     from a counter in the workspace (so pairs that share rows
                     of `normed` stay in step), 0 for a fixed tile sequence
     workspace_bytes the part of the workspace used
   T = 0 launches nothing: the plan reads single CTAs, 1 split, no
   workspace.  RC_ERR_INVALID_ARG / RC_ERR_UNSUPPORTED for sizes
   rc_kv_project refuses or num_sms < 1; *plan untouched then. */
typedef struct {
    int32_t kernel;
    int32_t splits;
    int32_t tail_splits;
    int32_t dynamic_tiles;
    int64_t tail_row0;
    size_t workspace_bytes;
} rc_project_plan;

rc_status rc_kv_project_plan(int32_t L, int64_t T, int32_t D, int32_t N, int32_t num_sms,
                             size_t workspace_bytes, rc_project_plan *plan);

/*
 * rc_kv_store -- step 4.  [ctx] ContextKvStore / _ContextKvStoreKernel,
 * _sum_squares_64, _rope; [rt] ContextKV.store.
 *
 * For every layer l < L whose slots[l] is not NULL and every row t < rows,
 * with s = slots[l][t]:
 *   s < 0                                      row skipped (nothing read or written)
 *   s >= num_blocks*block_size, or (cos_sin != NULL) positions[t] outside
 *   [0, max_position)                          row skipped and counted in *err
 *   otherwise, for each head h < H:
 *     key   = bf16(k_h * r), r = 1/sqrt(fma(sum k_h^2, 1/64, eps)),
 *             the sum folded as lane j holding the pair (2j, 2j+1): even and
 *             odd squares each by an xor butterfly, then even + odd;
 *     key   = GPT-J RoPE of each pair (2j, 2j+1) with c = cos_sin[pos, j],
 *             s = cos_sin[pos, 32 + j]: (fma(x, c, -(y*s)), fma(y, c, x*s)),
 *             rounded to bf16 (skipped when cos_sin is NULL);
 *     caches[l][s / block_size, h, s % block_size, 0:64]   = key
 *     caches[l][s / block_size, h, s % block_size, 64:128] = v[l, t, h, :]
 *   No other cache element is written.
 *
 *   k, v          bf16 views [L, >=rows, H, 64]: element (l, t, h, e) at
 *                 base + l*layer_stride + t*row_stride + h*64 + e; 4-byte
 *                 aligned, strides even and >= 0.  For a projection output
 *                 kv [L, T, 2*H*64]: k = kv, v = kv + 64*H, row stride
 *                 128*H, layer stride T*128*H.
 *   positions     int64 [rows] (read only with cos_sin), 8-byte aligned
 *   slots         host array of L device pointers to int64 [rows]; NULL
 *                 entries skip their layer
 *   cos_sin       bf16 [max_position, 64] (cos in 0..31, sin in 32..63) or NULL
 *   caches        host array of L device pointers to contiguous bf16
 *                 [num_blocks, H, block_size, 128], 4-byte aligned
 *   num_blocks, block_size   >= 1, num_blocks*block_size < 2^31
 *   H             KV heads: 1, 2, 4, 8, 16 or 32
 *   L             1 <= L <= 4096; layers go to the GPU 8 per launch
 *   rows          rows to insert, 0 <= rows < 2^31 (0: nothing launched)
 *   err           device int32 counter, incremented once per skipped
 *                 (row, layer) as above; may be NULL
 * Two non-negative slots of one layer that are equal write the same cache
 * entry in an unspecified order (a precondition violation).
 */
rc_status rc_kv_store(const uint16_t *k, const uint16_t *v,
                      int64_t k_layer_stride, int64_t k_row_stride,
                      int64_t v_layer_stride, int64_t v_row_stride,
                      const int64_t *positions, const int64_t *const *slots,
                      const uint16_t *cos_sin, int64_t max_position,
                      uint16_t *const *caches, int32_t num_blocks,
                      int32_t block_size, int32_t H, int32_t L, float eps,
                      int64_t rows, int32_t *err, cudaStream_t stream);

/*
 * rc_kv_store_rows -- rc_kv_store with a row count per layer ([rt]
 * _slot_groups: each layer's slot mapping has its own length and layer l
 * inserts its first len(slots[l]) rows; the pages issue one store call per
 * run of consecutive layers of equal length, here one launch takes up to 8
 * layers of any lengths).
 *
 *   layer_rows    HOST array of L row counts, each 0 <= layer_rows[l] < 2^31;
 *                 slots[l] and k, v hold at least layer_rows[l] rows
 *   other arguments as rc_kv_store (positions holds max_l layer_rows[l] rows)
 */
rc_status rc_kv_store_rows(const uint16_t *k, const uint16_t *v,
                           int64_t k_layer_stride, int64_t k_row_stride,
                           int64_t v_layer_stride, int64_t v_row_stride,
                           const int64_t *positions, const int64_t *const *slots,
                           const uint16_t *cos_sin, int64_t max_position,
                           uint16_t *const *caches, int32_t num_blocks,
                           int32_t block_size, int32_t H, int32_t L, float eps,
                           const int64_t *layer_rows, int32_t *err, cudaStream_t stream);

/*
 * rc_kv_project_store -- steps 3 and 4 fused (the projection and the store
 * of [rt] ContextKV.store in one pass; the scope's "store fused into the
 * GEMM epilogue").  The caches receive exactly the bits that
 *   rc_kv_project(normed, W, w_layout, kv, ...) followed by
 *   rc_kv_store(k = kv, v = kv + 64*H, row stride 128*H, layer stride
 *               T*128*H, positions, slots, cos_sin, caches, ..., rows, err)
 * would write with the same workspace, without the [L, T, 128*H] round trip:
 * the key is normed from the bf16-rounded projection exactly as
 * rc_kv_store norms it.  Where the projection is not split, CTA-pair tiles
 * store from the GEMM epilogue; split plans store from the pass that adds
 * the FP32 partials.
 *
 *   normed, W, w_layout, D        as rc_kv_project; N = 128*H
 *   L                             1 <= L <= 64 (one launch for all layers)
 *   T                             rows of the projection, as rc_kv_project
 *   positions, slots, cos_sin, max_position, caches, num_blocks,
 *   block_size, H, eps, err       as rc_kv_store (caches and cos_sin
 *                                 16-byte aligned)
 *   rows                          rows stored, 0 <= rows <= T
 *   kv_out                        optional bf16 [L, T, 128*H]: also write the
 *                                 projection; required when the plan neither
 *                                 splits nor uses CTA pairs (T <= 128 or
 *                                 N = 128, without a workspace)
 *   workspace                     as rc_kv_project
 */
rc_status rc_kv_project_store(const uint16_t *normed, const uint16_t *W,
                              int32_t w_layout, int32_t L, int64_t T, int32_t D,
                              int32_t H, const int64_t *positions,
                              const int64_t *const *slots,
                              const uint16_t *cos_sin, int64_t max_position,
                              uint16_t *const *caches, int32_t num_blocks,
                              int32_t block_size, float eps, int64_t rows,
                              int32_t *err, uint16_t *kv_out, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * rc_kv_project_store_rows -- rc_kv_project_store with a row count per
 * layer, as rc_kv_store_rows: layer l stores its first layer_rows[l] rows.
 *
 *   layer_rows    HOST array of L row counts, each 0 <= layer_rows[l] <= T
 *   other arguments as rc_kv_project_store
 */
rc_status rc_kv_project_store_rows(const uint16_t *normed, const uint16_t *W,
                                   int32_t w_layout, int32_t L, int64_t T, int32_t D,
                                   int32_t H, const int64_t *positions,
                                   const int64_t *const *slots,
                                   const uint16_t *cos_sin, int64_t max_position,
                                   uint16_t *const *caches, int32_t num_blocks,
                                   int32_t block_size, float eps, const int64_t *layer_rows,
                                   int32_t *err, uint16_t *kv_out, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream);

/*
 * rc_context_kv -- the whole chain in one call (steps 1 to 4; [rt]
 * ContextKV.store / MuseSparkDSparkModel.precompute_and_store_context_kv),
 * with the norms fused into the projection (the scope's "norms fused into
 * the GEMM producer"): a row pass writes the hidden-norm output
 * z = bf16(hidden_norm(x)) and each row's layer-norm inverse RMS r once; the
 * projection forms each layer's operand bf16((z * r) * pre_w[l]) in shared
 * memory (bit-identical to rc_context_norms' output) and stores as
 * rc_kv_project_store does.  The [L, T, D] normed rows never reach memory.
 * The caches receive exactly the bits of rc_context_norms +
 * rc_kv_project_store with an equally split projection.
 *
 *   x, T, D, hidden_w, pre_w, L, eps      as rc_context_norms (D = 8192,
 *                                         L <= 64)
 *   W, w_layout, H                        as rc_kv_project (N = 128*H)
 *   positions ... err, kv_out             as rc_kv_project_store
 *   workspace   device scratch, 256-byte aligned, required: the row pass's
 *               z and r (T*D*2 + T*4 bytes, rounded up) — or, for T <= 128
 *               or H = 1, the normed rows [L, T, D] — followed by the split-K
 *               partials; rc_context_kv_workspace_size() gives the bytes of
 *               the full plan, and less space splits K less.
 */
rc_status rc_context_kv(const uint16_t *x, int64_t T, int32_t D,
                        const uint16_t *hidden_w, const uint16_t *pre_w,
                        int32_t L, float eps, const uint16_t *W,
                        int32_t w_layout, int32_t H, const int64_t *positions,
                        const int64_t *const *slots, const uint16_t *cos_sin,
                        int64_t max_position, uint16_t *const *caches,
                        int32_t num_blocks, int32_t block_size, int64_t rows,
                        int32_t *err, uint16_t *kv_out, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream);

/* Workspace bytes of rc_context_kv for these sizes on the current device
   (0 for unsupported sizes). */
size_t rc_context_kv_workspace_size(int32_t L, int64_t T, int32_t D, int32_t H);

/*
 * rc_context_kv_chunked -- steps 1 to 4 ([rt] ContextKV.store /
 * MuseSparkDSparkModel.precompute_and_store_context_kv) as
 * rc_context_norms followed by rc_kv_project_store, by row chunks: the
 * norms of chunk c + 1 run on the GPU beside the projection + store of
 * chunk c (each SM holds one persistent projection CTA and one norms CTA),
 * so that the norms' HBM traffic overlaps the tensor-bound projection.  The
 * caches receive exactly the bits of rc_context_norms + rc_kv_project_store
 * (the normed rows, each projection sum and each stored bit are the same;
 * only the order in which rows are stored differs, so two rows sharing a
 * slot may leave either row's values, as in rc_kv_project_store).
 *
 *   x, T, D, hidden_w, pre_w, L, eps   as rc_context_norms (D = 8192,
 *                                      L <= 64)
 *   W, w_layout, H                     as rc_kv_project (N = 128*H)
 *   positions ... err                  as rc_kv_project_store (no kv_out)
 *   chunks      row chunks wanted (<= 0: chosen for the sizes and for where
 *               x lives); fewer are used where a chunk's projection would
 *               not run as persistent CTA pairs without workspace
 *               (rc_context_kv_chunks says how many); x may be page-locked
 *               host memory (its device address, rc_device_address), which
 *               the norms of each chunk read over the host link
 *   workspace   device scratch, 256-byte aligned, required, not
 *               overlapping x or W: the normed rows [L, T, D] (chunk by
 *               chunk), then a 256-byte tile counter per chunk (or, with one
 *               chunk, the projection's workspace, or where single CTAs
 *               project without a K split a bf16 copy of the projection
 *               that the store reads); rc_context_kv_chunked_workspace_size()
 *               gives enough bytes
 * The call ends with the last chunk's projection, which starts after every
 * earlier kernel of the call has completed; a later kernel or copy in the
 * stream sees all of the call's writes.  Errors as rc_kv_project_store
 * (RC_ERR_INVALID_ARG for a workspace too small for the plan).
 */
rc_status rc_context_kv_chunked(const uint16_t *x, int64_t T, int32_t D,
                                const uint16_t *hidden_w, const uint16_t *pre_w,
                                int32_t L, float eps, const uint16_t *W,
                                int32_t w_layout, int32_t H, const int64_t *positions,
                                const int64_t *const *slots, const uint16_t *cos_sin,
                                int64_t max_position, uint16_t *const *caches,
                                int32_t num_blocks, int32_t block_size, int64_t rows,
                                int32_t *err, int32_t chunks, void *workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * rc_context_kv_chunked_ex -- rc_context_kv_chunked with every norm option
 * of rc_context_norms_ex and a row count per layer: the caches receive
 * exactly the bits of rc_context_norms_ex + rc_kv_project_store_rows.
 *
 *   x, T, D, hidden, pre, L       as rc_context_norms_ex (D = 8192)
 *   W, w_layout, H                as rc_kv_project (N = 128*H)
 *   positions ... block_size      as rc_kv_project_store
 *   eps                           the K-norm's eps (the norms carry their
 *                                 own in hidden and pre)
 *   layer_rows                    HOST array of L row counts, each in
 *                                 [0, T] (layer l stores its first
 *                                 layer_rows[l] rows), or NULL for T rows
 *                                 in every layer
 *   err, chunks, workspace, ...   as rc_context_kv_chunked (the same
 *                                 workspace size); with x in device memory
 *                                 and a norm option beyond bf16 output-scale
 *                                 weights without a centre, chunks <= 0
 *                                 means one chunk (the option kernel beside
 *                                 the projection costs more than the overlap
 *                                 gains), while x in host memory is chunked
 *                                 as rc_context_kv_chunks says
 * Errors as rc_context_norms_ex and rc_context_kv_chunked.
 */
rc_status rc_context_kv_chunked_ex(const uint16_t *x, int64_t T, int32_t D,
                                   const rc_norm_params *hidden, const rc_norm_params *pre,
                                   int32_t L, const uint16_t *W, int32_t w_layout, int32_t H,
                                   const int64_t *positions, const int64_t *const *slots,
                                   const uint16_t *cos_sin, int64_t max_position,
                                   uint16_t *const *caches, int32_t num_blocks, int32_t block_size,
                                   float eps, const int64_t *layer_rows, int32_t *err,
                                   int32_t chunks, void *workspace, size_t workspace_bytes,
                                   cudaStream_t stream);

/* Workspace bytes of rc_context_kv_chunked for these sizes on the current
   device, enough for any chunk request and for x in device or host memory
   (0 for unsupported sizes; `chunks` is accepted for symmetry). */
size_t rc_context_kv_chunked_workspace_size(int32_t L, int64_t T, int32_t D, int32_t H,
                                            int32_t chunks);

/* Host only: the number of row chunks rc_context_kv_chunked uses for these
   sizes and chunk request on a GPU of num_sms SMs, with x in device memory
   (x_on_host = 0) or page-locked host memory read over the host link
   (x_on_host != 0; the call tells the two apart itself); 0 for unsupported
   sizes.  row0, when not NULL, receives the chunks' first rows and T
   (count + 1 entries; room for 17). */
int32_t rc_context_kv_chunks(int32_t L, int64_t T, int32_t D, int32_t H, int32_t chunks,
                             int32_t x_on_host, int32_t num_sms, int64_t *row0);

/*
 * rc_context_kv in two calls.  rc_context_rows is the row pass: per row t,
 *   z[t]  = bf16(hidden_norm(x[t]))          bf16 [T, 8192], 16-byte aligned
 *   r2[t] = 1/sqrt(fma(sum z[t]^2, 1/D, eps)) FP32 [T] (the layer norms'
 *                                            inverse RMS, shared by all layers)
 * in the order and roundings of rc_context_norms.  rc_context_kv_from_rows
 * then projects and stores from (z, r2, pre_w): each layer's operand
 * bf16((z * r2) * pre_w[l]) is formed in shared memory.  It takes
 * T > 128 and H >= 2 (CTA-pair tiles) only; `workspace` holds the split-K
 * partials (rc_kv_project_workspace_size() bytes; may be NULL).
 */
rc_status rc_context_rows(const uint16_t *x, int64_t T, int32_t D,
                          const uint16_t *hidden_w, float eps, uint16_t *z,
                          float *r2, cudaStream_t stream);
rc_status rc_context_kv_from_rows(const uint16_t *z, const float *r2, int64_t T,
                                  int32_t D, const uint16_t *pre_w, int32_t L,
                                  float eps, const uint16_t *W, int32_t w_layout,
                                  int32_t H, const int64_t *positions,
                                  const int64_t *const *slots,
                                  const uint16_t *cos_sin, int64_t max_position,
                                  uint16_t *const *caches, int32_t num_blocks,
                                  int32_t block_size, int64_t rows, int32_t *err,
                                  uint16_t *kv_out, void *workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * rc_kv_project_no_alloc -- rc_kv_project for callers that cannot allocate.
 * The pages have no counterpart: it is an addition of this library.
 *
 * Some callers cannot call cudaMalloc or provide a workspace (code running
 * inside an allocator or memory-pool callback, plug-ins whose host framework
 * owns every device allocation, serving paths that must not touch the
 * allocator once running).  This call takes the same operands as
 * rc_kv_project minus the workspace and allocates nothing: its split-K
 * scratch is an array of RC_NO_ALLOC_SCRATCH_BYTES (24 MiB) inside the
 * library, held on every GPU that loads the library until the process
 * exits.  Arguments are checked as rc_kv_project checks them (sizes, layout,
 * NULL and 16-byte alignment, out overlapping normed or W); out, normed or
 * W overlapping the array itself is refused too.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.
 *   - Sizes whose split-K plan needs more than 24 MiB are refused with
 *     RC_ERR_UNSUPPORTED (on a 152-SM GB300 no size needs more than 20 MB).
 *   - All calls share the array and it keeps the last call's contents; two
 *     calls whose work overlaps on the GPU (e.g. on different streams) race
 *     on it, so order them on one stream.  Nothing in it needs clearing:
 *     each call writes every partial it reads and zeroes the tile counter
 *     it uses (an asynchronous memset on `stream`, which allocates nothing).
 * Results are bit-identical to rc_kv_project's given a workspace of
 * rc_kv_project_workspace_size() bytes (the same plan, the same kernels).
 */
#define RC_NO_ALLOC_SCRATCH_BYTES ((size_t)24 << 20)
rc_status rc_kv_project_no_alloc(const uint16_t *normed, const uint16_t *W,
                                 int32_t w_layout, uint16_t *out, int32_t L,
                                 int64_t T, int32_t D, int32_t N,
                                 cudaStream_t stream);

/*
 * rc_qkv_front -- the decode QKV front of one draft layer on 1 to 16 tokens:
 * QKV projection, QK-norm, GPT-J RoPE and KV insert in one kernel ([rt]
 * _fused_qkv_projection, _attention, may_fuse_qkv_front; the pages' kernel
 * source is not among them, so its arithmetic is read from what they state).
 *
 *   proj[m, n] = bf16(sum_k hidden[m, k] * W[n, k])   FP32 accumulation
 * Each output row is [Q | K | V | O-gate]: q_size = 64*num_heads columns of
 * Q, kv_size = 64*num_kv_heads of K, kv_size of V, q_size of the gate
 * (_attention's split).  Then, per token m:
 *   out[m, Q and K heads] = per 64-wide head: bf16(head * r) with r the
 *       weightless inverse RMS 1/sqrt(fma(sum e^2, 1/64, eps)) (the context
 *       K-norm's lane-pair order), then GPT-J RoPE at positions[m] from
 *       cos_sin (cos_sin may be NULL: no rotation), rounded to bf16;
 *   out[m, V and gate]    = proj;
 *   cache[s/bs, h, s%bs, 0:64] = out[m, K head h] and [64:128] = V head h,
 *       for s = slots[m] >= 0.
 * A token whose slot is >= num_blocks*block_size, or (with a table) whose
 * position is outside [0, max_position), adds one to *err and inserts
 * nothing; with a bad position its Q and K are normed but not rotated.
 *
 *   hidden      bf16 [M, D] contiguous, 16-byte aligned
 *   M           tokens, 0 <= M <= 16 (0: nothing launched); else RC_ERR_UNSUPPORTED
 *   D           a positive multiple of 64
 *   W           bf16 [Nqkv, D] (the nn.Linear weight), Nqkv = 64*(2*num_heads +
 *               2*num_kv_heads), 16-byte aligned
 *   positions   int64 [M] (read with a table), 8-byte aligned
 *   slots       int64 [M] slot mapping, or NULL (nothing inserted)
 *   cache       bf16 [num_blocks, num_kv_heads, block_size, 128], 4-byte
 *               aligned; num_blocks*block_size < 2^31
 *   out         bf16 [M, Nqkv], 16-byte aligned, overlapping no input
 *   raw_out     optional bf16 [M, Nqkv]: also write the projection itself
 *   err         optional device int32 counter
 * Bit 8 and up of rc_read_device_faults are this kernel's fault bits.
 */
rc_status rc_qkv_front(const uint16_t *hidden, int32_t M, int32_t D, const uint16_t *W,
                       int32_t num_heads, int32_t num_kv_heads, const int64_t *positions,
                       const uint16_t *cos_sin, int64_t max_position, const int64_t *slots,
                       uint16_t *cache, int32_t num_blocks, int32_t block_size, float eps,
                       uint16_t *out, uint16_t *raw_out, int32_t *err, cudaStream_t stream);

/* rc_device_address -- the address at which the current device reads p:
   p itself for device or managed memory; for page-locked host memory
   mapped into the device's address space (cudaHostAlloc, or
   cudaHostRegister with mapping), its device address (the same value under
   unified addressing).  Pass the start of the page-locked allocation; the
   device address of a byte inside it is the result plus that byte's offset
   (the Python binding maps slices of pinned tensors this way).
   RC_ERR_INVALID_ARG when the device cannot address p through the CUDA
   runtime (pageable host memory, NULL); dev untouched then.  Host-only; no
   page counterpart. */
rc_status rc_device_address(const void *p, const void **dev);

/* Sticky fault bits raised on the device when a bounded wait gives up: bits
   0-3 by the projection kernels, bits 8-11 by the QKV front (per kernel:
   load pipeline, tensor-core pipeline, accumulator, drain).  A kernel that
   sees a raised bit of its own kind skips its work, so after a fault its
   outputs are wrong until the bits are cleared.  Reads (and with clear != 0
   resets) the bits of the current device; synchronises the device.  No
   page counterpart. */
rc_status rc_read_device_faults(uint32_t *flags, int32_t clear);

#ifdef __cplusplus
}
#endif

#endif /* ROPE_CHAIN_H */
