/*
 * spark_attn.h -- C ABI of the spark2_5 single-token decode attention block
 * for NVIDIA GB300 (sm_103a).
 *
 * The block (turbospark-runtime 0.3.0, src/families/spark/mod.rs, module doc
 * "One decoder layer, transcribed", and src/families/spark/attn.rs,
 * encode_attention_block) computes, for every sequence b of a batch:
 *
 *   x      = h / sqrt(mean(h^2) + eps) * input_layernorm     (plain w)
 *   qkv    = q_k_v_proj @ x           rows: q (n_q*d) | k (n_kv*d) | v (n_kv*d)
 *   g      = g_proj @ x               one logit per query head
 *   q, k   = NeoX rope at the token's position, per layer class:
 *              full    -> leading full_rotary_dim dims at full_theta
 *              sliding -> all head_dim dims at sliding_theta
 *   k, v   -> written into the cache row of the token's position
 *   a      = GQA attention (query head h reads KV head h / (n_q/n_kv)),
 *            scale `scale`, over the whole history (full layer) or the last
 *            `window` positions through the ring (sliding layer)
 *   a      = a * sigmoid(g) broadcast over head_dim       (before o_proj)
 *   out    = h + o_proj @ a                                (raw residual)
 *
 * Conventions shared by every entry point:
 *   - Device pointers are CUDA device addresses owned by the caller; the
 *     library never allocates or frees memory and never synchronises a stream
 *     unless the entry point says so.  All device pointers must be 16-byte
 *     aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued on it in order; a non-zero return means nothing was enqueued,
 *     except SPARK_ERR_CUDA from a failed launch.
 *   - Matrices are row-major: a [rows x cols] weight has out[r] = sum_c W[r,c] in[c].
 *   - Host arrays (`positions`) are read during the call only.
 *   - Return value: SPARK_OK (0) or a negative spark_status.
 */
#ifndef SPARK_ATTN_H
#define SPARK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPARK_ATTN_ABI_VERSION 4
/* largest batch one call accepts */
#define SPARK_MAX_BATCH 1024

/* Status codes.  INVALID_ARG / POSITION / BAD_RING / WORKSPACE / UNSUPPORTED
 * are detected on the host before anything is enqueued (the counterpart of
 * the pages' RealForwardError::Unsupported); CUDA is a launch error reported
 * by the runtime (RealForwardError::Gpu); DEVICE is a failure a kernel
 * recorded in the workspace error word. */
typedef enum spark_status {
  SPARK_OK = 0,
  SPARK_ERR_INVALID_ARG = -1,  /* null pointer, batch out of range, bad enum, misaligned pointer */
  SPARK_ERR_POSITION = -2,     /* position < 0, or its cache row lies outside the layer's capacity */
  SPARK_ERR_BAD_RING = -3,     /* ring capacity that would evict a row still inside the window */
  SPARK_ERR_WORKSPACE = -4,    /* workspace null, too small or misaligned */
  SPARK_ERR_UNSUPPORTED = -5,  /* geometry the kernels are not built for */
  SPARK_ERR_CUDA = -6,         /* a CUDA runtime call failed */
  SPARK_ERR_DEVICE = -7        /* a kernel set the workspace error word */
} spark_status;

typedef enum spark_dtype { SPARK_F32 = 0, SPARK_BF16 = 1 } spark_dtype;

/* Layer class: an entry of 1 in the model's full_attention_layer_mask marks a
 * full layer (src/families/spark/attn.rs, encode_attention_block, the rope
 * and window set-up). */
typedef enum spark_layer_class { SPARK_SLIDING = 0, SPARK_FULL = 1 } spark_layer_class;

/* Block geometry.  spark_geom_default() fills spark2_5's values: hidden 2560,
 * 16 query heads over 4 KV heads at head_dim 256, full layers rotate 64 dims
 * at theta 5e6, sliding layers all 256 at theta 1e4, window 512, eps 1e-6,
 * scale 256^-0.5 (mod.rs module doc; attn.rs module doc item 2).
 * Supported: head_dim == 256, n_q == 4 * n_kv with 1 <= n_kv <= 8,
 * hidden a multiple of 8 in [8, 8192], full_rotary_dim even in [2, 256],
 * window >= 1, thetas > 0, eps >= 0, finite scale. */
typedef struct spark_geom {
  int32_t hidden;
  int32_t n_q;
  int32_t n_kv;
  int32_t head_dim;
  int32_t full_rotary_dim;
  int32_t window;
  float full_theta;
  float sliding_theta;
  float eps;
  float scale;
} spark_geom;

/* One layer's weights (device, caller-owned), all of element type `dtype`:
 *   norm_w [hidden]                       input_layernorm.weight
 *   qkv_w  [n_q*d + 2*n_kv*d][hidden]     q_k_v_proj.weight (rows q | k | v)
 *   g_w    [n_q][hidden]                  g_proj.weight
 *   o_w    [hidden][n_q*d]                o_proj.weight                     */
typedef struct spark_layer_weights {
  const void* norm_w;
  const void* qkv_w;
  const void* g_w;
  const void* o_w;
  int32_t dtype; /* spark_dtype */
} spark_layer_weights;

/* One layer's KV cache (device, caller-owned): K and V are two buffers of
 * [batch][capacity][n_kv][head_dim] elements of `dtype`.
 * ring_capacity == 0: linear addressing, position p lives in row p
 *   (needs p < capacity).
 * ring_capacity  > 0: a ring of that many rows (sliding layers only;
 *   ring_capacity <= capacity and ring_capacity >= window): position p lives
 *   in row p mod ring_capacity, and attention addresses rows through the ring
 *   once seq_len = p + 1 exceeds it (attn.rs, encode_attention_block, the
 *   window set-up; kv_write.rs, kv_write_target). */
typedef struct spark_kv_layer {
  void* k;
  void* v;
  int64_t capacity;
  int32_t ring_capacity;
  int32_t dtype; /* spark_dtype */
} spark_kv_layer;

/* Fill `g` with spark2_5's geometry. */
void spark_geom_default(spark_geom* g);

/* Bytes of device workspace spark_attn_decode / spark_dbg_attention need for
 * `batch` sequences (0 for invalid arguments).  The workspace holds the fused
 * projection outputs, the rotated queries, the attention output, the split-K
 * partial results, the merge tickets and a device error word. */
size_t spark_attn_workspace_bytes(const spark_geom* g, int32_t batch);

/* Zero a workspace (enqueued on `stream`).  Required once after allocation:
 * the split-K merge tickets must start at zero; every call leaves them at
 * zero again. */
int spark_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Read and clear the workspace's device error word.  SYNCHRONISES `stream`.
 * Bits: 1 = a pipeline wait ran out of time, 2 = an index outside its buffer
 * was skipped. */
int spark_attn_error_word(void* workspace, size_t workspace_bytes, uint32_t* word, void* stream);

/* One decode step of the attention block for `batch` independent sequences
 * (attn.rs, encode_attention_block, plus the input RMSNorm and the raw
 * residual add of mod.rs's layer loop).
 *   h          [batch][hidden] fp32 device: residual stream in.
 *   (the projections take SPARK_PATH_AUTO's kernels, see below)
 *   w          the layer's weights.
 *   kv         the layer's cache; row slot(positions[b]) of K and V of each
 *              sequence b is overwritten with the token's rope'd k and its v,
 *              rounded to the cache's element type; nothing else is written.
 *   layer_class SPARK_FULL / SPARK_SLIDING.
 *   positions  [batch] HOST int32: the token's position in each sequence;
 *              the token attends to positions [kv_start, positions[b]].
 *   out        [batch][hidden] fp32 device: h + o_proj(...).  May equal h.
 *   workspace  >= spark_attn_workspace_bytes(g, batch) bytes, 256-byte
 *              aligned, initialised once by spark_attn_workspace_init.  Calls
 *              sharing a workspace must be ordered on one stream.
 * Errors: INVALID_ARG, POSITION, BAD_RING, WORKSPACE, UNSUPPORTED before any
 * work is enqueued; CUDA if a launch fails. */
int spark_attn_decode(const spark_geom* g, const float* h, const spark_layer_weights* w,
                      const spark_kv_layer* kv, int32_t layer_class,
                      const int32_t* positions, int32_t batch, float* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* A chunk of m consecutive tokens of ONE sequence through one layer, at
 * positions p0 .. p0+m-1: prefill, or verifying drafted tokens.  The result
 * is that of m calls of spark_attn_decode in position order (kv_write.rs,
 * module doc: chunked prefill reuses the per-token attention block, only the
 * K/V projections being batched): token t attends, causally, to the rows of
 * the tokens before it in the chunk and to the history inside its window,
 * even where a ring wraps inside the chunk (its k and v are staged in the
 * workspace and reach the cache only after attention).  The projections of
 * the m tokens run as one batch (tensor cores for m > 4, bf16 weights).
 *   h     [m][hidden] fp32 device; out [m][hidden], may equal h.
 *   kv    the sequence's cache: [1][capacity][n_kv][head_dim].  Rows
 *         slot(p0+t) receive the tokens' k and v (on a ring with m > its
 *         capacity, the last `capacity` tokens' rows).
 *   p0    position of the first token (>= 0); a linear cache needs
 *         p0 + m <= capacity.
 *   m     1 .. SPARK_MAX_BATCH.
 *   workspace  >= spark_attn_workspace_bytes(g, m), as for spark_attn_decode.
 * Errors as spark_attn_decode. */
int spark_attn_prefill(const spark_geom* g, const float* h, const spark_layer_weights* w,
                       const spark_kv_layer* kv, int32_t layer_class, int32_t p0, int32_t m,
                       float* out, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step through a stack of n_layers attention blocks (mod.rs's
 * layer loop with the MLP left out: the output of layer l is the input of
 * layer l+1).  The same result as calling spark_attn_decode layer by layer,
 * with h -> out, then out -> out; for bf16 weights and caches, batch <= 4,
 * n_kv <= 4, hidden <= 4096 and full_rotary_dim a multiple of 4 it runs as
 * one persistent kernel per 40 layers (cooperative launch, one CTA per SM)
 * whose weight and KV streams run ahead across layer boundaries; otherwise it
 * falls back to the per-layer path.
 *   w, kv, layer_class  arrays of n_layers entries (host arrays of device
 *                       pointers), positions as for spark_attn_decode.
 *   out may equal h.  workspace as for spark_attn_decode. */
int spark_attn_decode_stack(const spark_geom* g, const float* h, int32_t n_layers,
                            const spark_layer_weights* w, const spark_kv_layer* kv,
                            const int32_t* layer_class, const int32_t* positions,
                            int32_t batch, float* out, void* workspace,
                            size_t workspace_bytes, void* stream);

/* ---- the block's stages (same conventions) ------------------------------ */

/* Which kernels compute the two projections (the `path` argument below).
 * AUTO picks what spark_attn_decode runs: for batch <= 4, or fp32 weights,
 * the GEMV kernels, which read each weight once for up to 4 sequences; for
 * larger batches with bf16 weights, a GEMM on the tensor cores (tcgen05,
 * tensor-memory accumulator) that reads each weight from HBM once for the
 * whole batch (one launch; chunks of 128 sequences after the first find the
 * weight rows in L2), its fp32 activations carried as two bf16 halves
 * (x = hi + lo).
 * GEMV and MMA force one; MMA needs bf16 weights, hidden % 64 == 0 and, for
 * q_k_v_proj, a rotary dim <= 128 or == head_dim (else UNSUPPORTED). */
#define SPARK_PATH_AUTO 0
#define SPARK_PATH_GEMV 1
#define SPARK_PATH_MMA 2

/* Input RMSNorm + q_k_v_proj + g_proj + split + per-class NeoX rope + the
 * cache-row write (attn.rs, encode_attention_block: the fused projection,
 * the gate's projection reading the same normed x, encode_split_qkv with k
 * and v landing in their slots, encode_rope_neox_subdim on q and on k).
 *   q_rot    [batch][n_q*d] fp32 device: rotated queries.
 *   g_logits [batch][n_q] fp32 device: gate logits (before the sigmoid).
 *   kv       row slot(p) of K receives rope(k), of V receives v.
 *   path     SPARK_PATH_*.
 *   workspace as for spark_attn_decode (the MMA path keeps its activation
 *            rows, rope tables and split-K partial results there). */
int spark_dbg_qkv_rope(const spark_geom* g, const float* h, const spark_layer_weights* w,
                       const spark_kv_layer* kv, int32_t layer_class, const int32_t* positions,
                       int32_t batch, float* q_rot, float* g_logits, int32_t path,
                       void* workspace, size_t workspace_bytes, void* stream);

/* GQA decode attention over each sequence's window (attn.rs,
 * encode_attention_block -> kv_write.rs, encode_attention_any), split over
 * the GPU with a log-sum-exp merge.
 *   q_rot [batch][n_q*d] fp32 device.
 *   a     [batch][n_q*d] fp32 device: un-gated attention output.
 *   n_ctas number of thread blocks sharing the work (0 = automatic); the
 *          result does not depend on it beyond floating-point reassociation.
 *   workspace as for spark_attn_decode. */
int spark_dbg_attention(const spark_geom* g, const float* q_rot, const spark_kv_layer* kv,
                        int32_t layer_class, const int32_t* positions, int32_t batch,
                        float* a, int32_t n_ctas, void* workspace, size_t workspace_bytes,
                        void* stream);

/* The same attention for callers that cannot allocate device memory: hosts
 * whose own memory pool owns the whole device and forbids allocations by
 * plug-ins, and latency-critical loops that must not allocate mid-run.  It
 * takes no workspace: its scratch -- the split-K partial results, the merge
 * tickets and an error word -- is a fixed array of about 2.4 MiB inside the
 * library, which every GPU that loads the library holds until the process
 * exits.  No counterpart on the source pages: this entry point is this
 * library's own.
 *   Arguments, checks and results as spark_dbg_attention, without n_ctas
 *   and the workspace; the grid is the one spark_dbg_attention chooses by
 *   itself, at most 320 CTAs.  Limit: batch * n_kv <= 256, else
 *   SPARK_ERR_WORKSPACE (nothing enqueued).  Allocates nothing (no
 *   cudaMalloc, no cudaFree, no allocating library call).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  Every call clears the array's merge tickets
 *   and then shares the array: calls that overlap on the GPU (on different
 *   streams, or on one stream without ordering) race and must not be
 *   issued.  Failures a kernel records (bits as spark_attn_error_word) stay
 *   in the array's error word until spark_dbg_attention_noalloc_error_word
 *   reads it. */
int spark_dbg_attention_noalloc(const spark_geom* g, const float* q_rot,
                                const spark_kv_layer* kv, int32_t layer_class,
                                const int32_t* positions, int32_t batch, float* a,
                                void* stream);

/* Read and clear the error word of spark_dbg_attention_noalloc's fixed array
 * on the current device (the bits of every call since the last read).
 * SYNCHRONISES `stream`; allocates nothing.  No counterpart on the source
 * pages. */
int spark_dbg_attention_noalloc_error_word(uint32_t* word, void* stream);

/* Head gate + o_proj + raw residual (attn.rs: encode_sigmoid_head_gate_mul
 * and the o_proj GEMV; mod.rs: encode_residual_add).
 *   a        [batch][n_q*d] fp32 device, un-gated attention output.
 *   g_logits [batch][n_q] fp32 device gate logits.
 *   h        [batch][hidden] fp32 device; out [batch][hidden], may equal h.
 *   path, workspace as for spark_dbg_qkv_rope. */
int spark_dbg_gate_oproj(const spark_geom* g, const float* a, const float* g_logits,
                         const float* h, const spark_layer_weights* w, int32_t batch,
                         float* out, int32_t path, void* workspace, size_t workspace_bytes,
                         void* stream);

/* The failure path of the kernels' bounded waits, on purpose: one thread
 * waits for an mbarrier phase that nothing completes, gives up after
 * limit_ns (1 .. 2e9), sets bit 1 of the workspace error word and returns,
 * leaving the context usable.  For tests of the error reporting; the pages
 * have no counterpart. */
int spark_dbg_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns, void* stream);

/* Human-readable text of a status code (static storage). */
const char* spark_attn_status_string(int status);

/* SPARK_ATTN_ABI_VERSION of the loaded library. */
int32_t spark_attn_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPARK_ATTN_H */
