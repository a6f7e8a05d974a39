// launch.h -- host launchers of the block's kernels (internal to the library).
#pragma once

#include "common.cuh"

namespace spark {

// Input RMSNorm + q_k_v_proj + g_proj + NeoX rope + cache-row write:
// q_rot[b] = rope(W_q x_b), cache rows of k and v at slot(pos[b]), g[b] = W_g x_b.
cudaError_t launch_qkv_rope(int wdtype, int cdtype, const float* h, const void* norm_w,
                            const void* qkv_w, const void* g_w, float* q_rot, void* kc, void* vc,
                            float* g_out, uint32_t* err, int hidden, int n_q, int n_kv, int batch,
                            int64_t capacity, int ring_capacity, int rotary_dim, double theta,
                            float eps, const int32_t* positions, cudaStream_t st);

// Head gate + o_proj + raw residual: out[b] = h[b] + W_o (a[b] * sigmoid(g[b])).
// free_sms > 0: SMs the previous kernel leaves free while it runs (one
// sequence: the grid is shaped so that most rows are requested on them).
cudaError_t launch_oproj(int wdtype, const float* a, const float* g, const float* h,
                         const void* o_w, float* out, uint32_t* err, int hidden, int n_q, int batch,
                         cudaStream_t st, int free_sms = -1);

// The rows a chunk of consecutive tokens of one sequence produces, staged
// ([tokens][n_kv][head_dim] in the cache type) until attention has run.
// p0 < 0: a decode step (no chunk).
struct ChunkSrc {
  int64_t p0 = -1;
  const void* k = nullptr;
  const void* v = nullptr;
};

// Split-K GQA decode attention with the log-sum-exp merge.  With a chunk,
// `positions` are the tokens' positions, the cache is one sequence's, and
// rows at positions >= chunk.p0 come from the staged rows.  The grid never
// exceeds max_ctas CTAs (`part` holds max_ctas + batch * n_kv partials).
// sms_held (optional): the SMs the launch's CTAs hold until it ends.
cudaError_t launch_attention(int cdtype, const float* q_rot, const void* kc, const void* vc,
                             int n_kv, int64_t capacity, int ring_capacity, bool full,
                             int window, float scale, const int32_t* positions, int batch,
                             float* a, float* part, uint32_t* counters, uint32_t* err,
                             int n_ctas, const void* l2_prefetch, size_t l2_prefetch_bytes,
                             cudaStream_t st, const ChunkSrc& chunk = ChunkSrc(),
                             int max_ctas = kMaxAttnCtas, int* sms_held = nullptr);

// The same attention for a chunk, grouped by query (attn_chunk.cu): one CTA
// per (group of consecutive tokens, KV head) reads the union of the tokens'
// windows once.  Applies to bf16 caches when the groups cover the GPU.
bool attention_chunk_grouped_applies(int cdtype, int m, int n_kv);
cudaError_t launch_attention_chunk_grouped(const float* q_rot, const void* kc, const void* vc, int n_kv,
                                           int64_t capacity, int ring_capacity, bool full, int window,
                                           float scale, int64_t p0, int m, const void* ks, const void* vs,
                                           float* a, uint32_t* err, cudaStream_t st);

// Copy a chunk's staged rows into their cache slots (after attention).
cudaError_t launch_commit_rows(int cdtype, const void* ks, const void* vs, void* kc, void* vc,
                               int n_kv, int64_t p0, int m, int ring_capacity, cudaStream_t st);

// The two projections for a batch on the tensor cores (mma.cu): same results
// as launch_qkv_rope / launch_oproj, for bf16 weights.
struct MmaWorkspace {
  __nv_bfloat16* x;    // [chunk][2][bpad][max(hidden, q_dim)] activation rows (hi, lo)
  float2* cs;          // [batch][head_dim / 2] rope (cos, sin)
  float* part;         // split-K partial results
  uint32_t* tickets;   // [kMmaMaxCtas] split-K tickets, zero between launches
  uint64_t* trace;     // [kTraceWords] opt-in phase stamps
};

bool mma_projections_supported(int wdtype, int hidden, int n_q, int rotary_dim);

cudaError_t launch_qkv_mma(int cdtype, const float* h, const void* norm_w, const void* qkv_w,
                           const void* g_w, float* q_rot, void* kc, void* vc, float* g_out,
                           uint32_t* err, int hidden, int n_q, int n_kv, int batch, int64_t capacity,
                           int ring_capacity, int rotary_dim, double theta, float eps,
                           const int32_t* positions, const MmaWorkspace& ws, cudaStream_t st);

cudaError_t launch_oproj_mma(const float* a, const float* g, const float* h, const void* o_w,
                             float* out, uint32_t* err, int hidden, int n_q, int batch,
                             const MmaWorkspace& ws, cudaStream_t st);

// The MLP half of a decoder layer and the head (mlp.cu: GEMV kernels for
// small batches, any weight type; mma.cu: tensor-core GEMMs, bf16 weights).
//   mlp:  out[b] = h[b] + W_down (gelu(W_gate x_b) * (W_up x_b)), x_b = rms(h_b) * norm_w
//   head: logits[b] = E rms(h_b) * norm_w
// m ([batch][inter] fp32) holds the GELU products of the GEMV path; xd
// ([chunk][2][bpad][inter] bf16) the (hi, lo) rows of the tensor-core path.
cudaError_t launch_mlp_gemv(int wdtype, const float* h, const void* norm_w, const void* gate_w,
                            const void* up_w, const void* down_w, float* m, float* out, uint32_t* err,
                            int hidden, int inter, int batch, float eps, cudaStream_t st);
cudaError_t launch_head_gemv(int wdtype, const float* h, const void* norm_w, const void* embed,
                             float* logits, uint32_t* err, int hidden, int vocab, int batch, float eps,
                             cudaStream_t st);
bool mma_mlp_supported(int wdtype, int hidden, int inter);
cudaError_t launch_mlp_mma(const float* h, const void* norm_w, const void* gate_w, const void* up_w,
                           const void* down_w, float* out, uint32_t* err, int hidden, int inter, int batch,
                           float eps, const MmaWorkspace& ws, __nv_bfloat16* xd, cudaStream_t st);
cudaError_t launch_head_mma(const float* h, const void* norm_w, const void* embed, float* logits, uint32_t* err,
                            int hidden, int vocab, int batch, float eps, const MmaWorkspace& ws, cudaStream_t st);

// Opt-in per-CTA timeline of spark_attn_decode's kernels (SPARK_TRACE_LAYER
// set in the environment): the stamp array of kernel `kind` (0 the
// projections and rope, 1 attention, 2 the gate and o_proj) of the call being
// enqueued -- two calls alternate between two halves of the workspace's trace
// region -- or null.
uint64_t* layer_trace(int kind);

// Number of SMs of the current device (cached per device).
int device_sm_count();

// A KV cache [rows][n_kv][256] (bf16 or fp32) as the attention kernels load
// it: one TMA box per K or V half of a 16-row tile of one KV head, landing in
// shared memory as 128-byte lines [line of the row][row][128 bytes] with the
// 128-byte swizzle.  The view is 4-D {elements of a line, rows, lines of a
// row, heads} with strides {row, 128 bytes, head}: one request replaces one
// per 128-byte line (a request costs the SM's TMA unit ~30 ns to issue, so a
// 16 KB tile took ~0.25 us to request as eight).
bool make_kv_tile_map(CUtensorMap* map, const void* base, bool bf16, int n_kv, int64_t rows);

// cuTensorMapEncodeTiled from the driver (null if the driver has none).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

}  // namespace spark
