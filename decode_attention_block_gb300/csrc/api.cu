// api.cu -- the library's C ABI (declared in include/spark_attn.h): argument
// validation, the per-class parameter selection and the launch sequence of
// one decode step.
//
// Host logic follows turbospark-runtime 0.3.0:
//  * src/families/spark/attn.rs, rope_params_for: full layers take
//    (full_rotary_dim, full_theta), sliding layers (head_dim, sliding_theta);
//  * src/families/spark/attn.rs, encode_attention_block: seq_len =
//    position + 1; full layers read [0, seq_len) with identity addressing;
//    sliding layers read [seq_len - window, seq_len) through the ring once
//    seq_len exceeds its capacity;
//  * RealForwardError::{Unsupported, Gpu} become the status codes.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "checks.h"
#include "launch.h"

namespace spark {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

namespace {
uint64_t* g_layer_trace = nullptr;  // trace region of the decode call being enqueued, or null
}

uint64_t* layer_trace(int kind) {
  return g_layer_trace ? g_layer_trace + (size_t)kind * kTraceCtas * kTraceEvs : nullptr;
}

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {

// One thread waits, with the same bounded wait every pipeline uses, for an
// mbarrier phase nothing completes; when the limit passes it raises the
// wait-timeout bit of the error word and the kernel returns.
__global__ void k_wait_timeout(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns)) atomicOr(err, kErrWaitTimeout);
  }
}

}  // namespace

}  // namespace spark

using namespace spark;
using namespace spark::checks;

namespace {

// Up to this batch the GEMV kernels read each weight once for all sequences
// (they keep every sequence's activations in registers); above it the
// projections run as GEMMs on the tensor cores.
constexpr int kGemvMaxBatch = 4;

MmaWorkspace mma_ws(void* ws, const WsLayout& L) {
  MmaWorkspace m;
  m.x = ws_at<__nv_bfloat16>(ws, L.mx);
  m.cs = ws_at<float2>(ws, L.mcs);
  m.part = ws_at<float>(ws, L.mpart);
  m.tickets = ws_at<uint32_t>(ws, L.mtick);
  m.trace = ws_at<uint64_t>(ws, L.trace);
  return m;
}

// Which kernels compute a projection: SPARK_PATH_MMA / SPARK_PATH_GEMV, or
// a negative status if the caller forced a path these arguments cannot take.
int pick_path(int32_t path, int wdtype, const spark_geom* g, int rotary_dim, int32_t batch) {
  if (path != SPARK_PATH_AUTO && path != SPARK_PATH_GEMV && path != SPARK_PATH_MMA)
    return SPARK_ERR_INVALID_ARG;
  if (path == SPARK_PATH_GEMV || (path == SPARK_PATH_AUTO && batch <= kGemvMaxBatch))
    return SPARK_PATH_GEMV;
  const bool ok = mma_projections_supported(wdtype, g->hidden, g->n_q, rotary_dim);
  if (path == SPARK_PATH_MMA) return ok ? SPARK_PATH_MMA : SPARK_ERR_UNSUPPORTED;
  return ok ? SPARK_PATH_MMA : SPARK_PATH_GEMV;
}

cudaError_t run_qkv(int path, const spark_geom* g, const float* h, const spark_layer_weights* w,
                    const spark_kv_layer* kv, int rotary_dim, double theta, const int32_t* positions,
                    int32_t batch, float* q_rot, float* g_logits, uint32_t* err, void* ws,
                    const WsLayout& L, cudaStream_t st) {
  if (path == SPARK_PATH_MMA)
    return launch_qkv_mma(kv->dtype, h, w->norm_w, w->qkv_w, w->g_w, q_rot, kv->k, kv->v, g_logits,
                          err, g->hidden, g->n_q, g->n_kv, batch, kv->capacity, kv->ring_capacity,
                          rotary_dim, theta, g->eps, positions, mma_ws(ws, L), st);
  return launch_qkv_rope(w->dtype, kv->dtype, h, w->norm_w, w->qkv_w, w->g_w, q_rot, kv->k, kv->v,
                         g_logits, err, g->hidden, g->n_q, g->n_kv, batch, kv->capacity,
                         kv->ring_capacity, rotary_dim, theta, g->eps, positions, st);
}

cudaError_t run_oproj(int path, const spark_geom* g, const float* a, const float* g_logits,
                      const float* h, const spark_layer_weights* w, int32_t batch, float* out,
                      uint32_t* err, void* ws, const WsLayout& L, cudaStream_t st, int free_sms = -1) {
  if (path == SPARK_PATH_MMA)
    return launch_oproj_mma(a, g_logits, h, w->o_w, out, err, g->hidden, g->n_q, batch, mma_ws(ws, L), st);
  return launch_oproj(w->dtype, a, g_logits, h, w->o_w, out, err, g->hidden, g->n_q, batch, st, free_sms);
}

}  // namespace

extern "C" {

void spark_geom_default(spark_geom* g) {
  if (!g) return;
  g->hidden = 2560;
  g->n_q = 16;
  g->n_kv = 4;
  g->head_dim = 256;
  g->full_rotary_dim = 64;
  g->window = 512;
  g->full_theta = 5.0e6f;
  g->sliding_theta = 1.0e4f;
  g->eps = 1.0e-6f;
  g->scale = 0.0625f;  // 256^-0.5
}

size_t spark_attn_workspace_bytes(const spark_geom* g, int32_t batch) {
  if (check_geom(g) != SPARK_OK || check_batch(batch) != SPARK_OK) return 0;
  return ws_layout(g->hidden, g->n_q, g->n_kv, batch).total;
}

int spark_attn_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return SPARK_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream));
}

int spark_attn_error_word(void* workspace, size_t workspace_bytes, uint32_t* word, void* stream) {
  if (!workspace || workspace_bytes < 256 || !word) return SPARK_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *word = host;
  return cuda_status(e);
}

int spark_dbg_qkv_rope(const spark_geom* g, const float* h, const spark_layer_weights* w,
                       const spark_kv_layer* kv, int32_t layer_class, const int32_t* positions,
                       int32_t batch, float* q_rot, float* g_logits, int32_t path, void* workspace,
                       size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_weights(w, true, false)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_kv(g, kv, layer_class, positions, batch)) != SPARK_OK) return s;
  if ((s = check_ws(g, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !q_rot || !g_logits || !aligned16(h) || !aligned16(q_rot) || !aligned16(g_logits))
    return SPARK_ERR_INVALID_ARG;
  int rotary_dim;
  double theta;
  rope_for(g, layer_class, &rotary_dim, &theta);
  const int chosen = pick_path(path, w->dtype, g, rotary_dim, batch);
  if (chosen < 0) return chosen;
  const WsLayout L = ws_layout(g->hidden, g->n_q, g->n_kv, batch);
  return cuda_status(run_qkv(chosen, g, h, w, kv, rotary_dim, theta, positions, batch, q_rot,
                             g_logits, ws_at<uint32_t>(workspace, L.err), workspace, L,
                             (cudaStream_t)stream));
}

int spark_dbg_attention(const spark_geom* g, const float* q_rot, const spark_kv_layer* kv,
                        int32_t layer_class, const int32_t* positions, int32_t batch, float* a,
                        int32_t n_ctas, void* workspace, size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_kv(g, kv, layer_class, positions, batch)) != SPARK_OK) return s;
  if ((s = check_ws(g, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!q_rot || !a || !aligned16(q_rot) || !aligned16(a)) return SPARK_ERR_INVALID_ARG;
  if (n_ctas < 0 || n_ctas > kMaxAttnCtas) return SPARK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(g->hidden, g->n_q, g->n_kv, batch);
  return cuda_status(launch_attention(
      kv->dtype, q_rot, kv->k, kv->v, g->n_kv, kv->capacity, kv->ring_capacity,
      layer_class == SPARK_FULL, g->window, g->scale, positions, batch, a,
      ws_at<float>(workspace, L.part), ws_at<uint32_t>(workspace, L.counters),
      ws_at<uint32_t>(workspace, L.err), n_ctas, nullptr, 0, (cudaStream_t)stream));
}

int spark_dbg_gate_oproj(const spark_geom* g, const float* a, const float* g_logits,
                         const float* h, const spark_layer_weights* w, int32_t batch, float* out,
                         int32_t path, void* workspace, size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_weights(w, false, true)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_ws(g, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!a || !g_logits || !h || !out || !aligned16(a) || !aligned16(g_logits) || !aligned16(h) ||
      !aligned16(out))
    return SPARK_ERR_INVALID_ARG;
  const int chosen = pick_path(path, w->dtype, g, 0, batch);
  if (chosen < 0) return chosen;
  const WsLayout L = ws_layout(g->hidden, g->n_q, g->n_kv, batch);
  return cuda_status(run_oproj(chosen, g, a, g_logits, h, w, batch, out,
                               ws_at<uint32_t>(workspace, L.err), workspace, L, (cudaStream_t)stream));
}

int spark_attn_decode(const spark_geom* g, const float* h, const spark_layer_weights* w,
                      const spark_kv_layer* kv, int32_t layer_class, const int32_t* positions,
                      int32_t batch, float* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_weights(w, true, true)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_kv(g, kv, layer_class, positions, batch)) != SPARK_OK) return s;
  if ((s = check_ws(g, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !out || !aligned16(h) || !aligned16(out)) return SPARK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(g->hidden, g->n_q, g->n_kv, batch);
  cudaStream_t st = (cudaStream_t)stream;
  float* g_logits = ws_at<float>(workspace, L.g);
  float* q_rot = ws_at<float>(workspace, L.q_rot);
  float* a = ws_at<float>(workspace, L.a);
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  int rotary_dim;
  double theta;
  rope_for(g, layer_class, &rotary_dim, &theta);
  static const bool tracing = getenv("SPARK_TRACE_LAYER") != nullptr;
  static unsigned calls = 0;
  if (tracing)
    g_layer_trace = ws_at<uint64_t>(workspace, L.trace) + (size_t)(calls++ & 1) * 3 * kTraceCtas * kTraceEvs;
  cudaError_t e = run_qkv(pick_path(SPARK_PATH_AUTO, w->dtype, g, rotary_dim, batch), g, h, w, kv,
                          rotary_dim, theta, positions, batch, q_rot, g_logits, err, workspace, L, st);
  int held = 0;  // SMs attention's CTAs hold while o_proj's first CTAs start
  if (e == cudaSuccess)
    e = launch_attention(kv->dtype, q_rot, kv->k, kv->v, g->n_kv, kv->capacity,
                         kv->ring_capacity, layer_class == SPARK_FULL, g->window, g->scale,
                         positions, batch, a, ws_at<float>(workspace, L.part),
                         ws_at<uint32_t>(workspace, L.counters), err, 0, nullptr, 0, st, ChunkSrc(),
                         kMaxAttnCtas, &held);
  if (e == cudaSuccess)
    e = run_oproj(pick_path(SPARK_PATH_AUTO, w->dtype, g, 0, batch), g, a, g_logits, h, w, batch, out,
                  err, workspace, L, st, held > 0 ? device_sm_count() - held : -1);
  g_layer_trace = nullptr;
  return cuda_status(e);
}

int spark_attn_prefill(const spark_geom* g, const float* h, const spark_layer_weights* w,
                       const spark_kv_layer* kv, int32_t layer_class, int32_t p0, int32_t m,
                       float* out, void* workspace, size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_weights(w, true, true)) != SPARK_OK) return s;
  if ((s = check_batch(m)) != SPARK_OK) return s;
  if (p0 < 0 || (int64_t)p0 + m - 1 >= (int64_t)INT32_MAX - 1) return SPARK_ERR_POSITION;
  const int32_t last = p0 + m - 1;  // the chunk's positions are p0 .. last
  if ((s = check_kv(g, kv, layer_class, &last, 1)) != SPARK_OK) return s;
  if ((s = check_ws(g, m, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !out || !aligned16(h) || !aligned16(out)) return SPARK_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(g->hidden, g->n_q, g->n_kv, m);
  cudaStream_t st = (cudaStream_t)stream;
  std::vector<int32_t> positions(m);
  for (int32_t t = 0; t < m; ++t) positions[t] = p0 + t;
  float* g_logits = ws_at<float>(workspace, L.g);
  float* q_rot = ws_at<float>(workspace, L.q_rot);
  float* a = ws_at<float>(workspace, L.a);
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  // the chunk's k and v rows go to a staging buffer first: on a ring a later
  // token's row replaces a row that earlier tokens of the chunk still read
  const size_t ce = kv->dtype == SPARK_BF16 ? 2 : 4;
  unsigned char* ks = ws_at<unsigned char>(workspace, L.stage);
  unsigned char* vs = ks + (size_t)m * g->n_kv * kHeadDim * ce;
  spark_kv_layer staged = *kv;
  staged.k = ks;
  staged.v = vs;
  staged.capacity = 1;       // row t of the staging buffer holds token t:
  staged.ring_capacity = 1;  // slot = position mod 1 = 0 of "sequence" t
  int rotary_dim;
  double theta;
  rope_for(g, layer_class, &rotary_dim, &theta);
  cudaError_t e = run_qkv(pick_path(SPARK_PATH_AUTO, w->dtype, g, rotary_dim, m), g, h, w, &staged,
                          rotary_dim, theta, positions.data(), m, q_rot, g_logits, err, workspace, L, st);
  ChunkSrc chunk;
  chunk.p0 = p0;
  chunk.k = ks;
  chunk.v = vs;
  if (e == cudaSuccess) {
    if (attention_chunk_grouped_applies(kv->dtype, m, g->n_kv))
      e = launch_attention_chunk_grouped(q_rot, kv->k, kv->v, g->n_kv, kv->capacity, kv->ring_capacity,
                                         layer_class == SPARK_FULL, g->window, g->scale, p0, m, ks, vs, a, err,
                                         st);
    else
      e = launch_attention(kv->dtype, q_rot, kv->k, kv->v, g->n_kv, kv->capacity, kv->ring_capacity,
                           layer_class == SPARK_FULL, g->window, g->scale, positions.data(), m, a,
                           ws_at<float>(workspace, L.part), ws_at<uint32_t>(workspace, L.counters), err,
                           0, nullptr, 0, st, chunk);
  }
  if (e == cudaSuccess)
    e = launch_commit_rows(kv->dtype, ks, vs, kv->k, kv->v, g->n_kv, p0, m, kv->ring_capacity, st);
  if (e == cudaSuccess)
    e = run_oproj(pick_path(SPARK_PATH_AUTO, w->dtype, g, 0, m), g, a, g_logits, h, w, m, out, err,
                  workspace, L, st);
  return cuda_status(e);
}

int spark_dbg_wait_timeout(void* workspace, size_t workspace_bytes, uint64_t limit_ns, void* stream) {
  if (!workspace || workspace_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return SPARK_ERR_WORKSPACE;
  if (limit_ns == 0 || limit_ns > kWaitLimitNs) return SPARK_ERR_INVALID_ARG;
  k_wait_timeout<<<1, 32, 0, (cudaStream_t)stream>>>(static_cast<uint32_t*>(workspace), limit_ns);
  return cuda_status(cudaGetLastError());
}

const char* spark_attn_status_string(int status) {
  switch (status) {
    case SPARK_OK: return "ok";
    case SPARK_ERR_INVALID_ARG: return "invalid argument";
    case SPARK_ERR_POSITION: return "position outside the layer's cache";
    case SPARK_ERR_BAD_RING: return "ring capacity would evict rows inside the window";
    case SPARK_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case SPARK_ERR_UNSUPPORTED: return "geometry not supported by the kernels";
    case SPARK_ERR_CUDA: return "CUDA runtime error";
    case SPARK_ERR_DEVICE: return "a kernel reported a failure in the workspace error word";
    default: return "unknown status";
  }
}

int32_t spark_attn_abi_version(void) { return SPARK_ATTN_ABI_VERSION; }

}  // extern "C"
