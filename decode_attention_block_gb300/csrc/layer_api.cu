// layer_api.cu -- the C ABI of the rest of the decoder layer and of the head
// (declared in include/spark_layer.h): argument validation, the choice
// between the GEMV and the tensor-core kernels, and the launches
// (turbospark-runtime 0.3.0, src/families/spark/mod.rs: produce_real_spark's
// layer loop -- the post-attention RMSNorm and mlp::encode_mlp_block -- and
// its head -- the final RMSNorm and the GEMV over the tied embedding).
#include "../../include/spark_layer.h"
#include "checks.h"
#include "launch.h"

using namespace spark;
using namespace spark::checks;

namespace {

constexpr int kGemvMaxBatch = 4;  // as for the attention block's projections
constexpr int32_t kMaxInter = 16384;
constexpr int32_t kMaxVocab = 1 << 22;

int check_inter(int32_t inter) {
  if (inter < 0) return SPARK_ERR_INVALID_ARG;
  if (inter < 8 || inter > kMaxInter || inter % 8 != 0) return SPARK_ERR_UNSUPPORTED;
  return SPARK_OK;
}

int check_mlp_ws(const spark_geom* g, int32_t inter, int32_t batch, void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPARK_ERR_WORKSPACE;
  if (bytes < mlp_ws_layout(g->hidden, inter, batch).total) return SPARK_ERR_WORKSPACE;
  return SPARK_OK;
}

// SPARK_PATH_GEMV / SPARK_PATH_MMA for these arguments, or a negative status
// if the caller forced a path they cannot take.
int pick(int32_t path, int32_t batch, bool mma_ok) {
  if (path != SPARK_PATH_AUTO && path != SPARK_PATH_GEMV && path != SPARK_PATH_MMA) return SPARK_ERR_INVALID_ARG;
  if (path == SPARK_PATH_GEMV || (path == SPARK_PATH_AUTO && batch <= kGemvMaxBatch)) return SPARK_PATH_GEMV;
  if (path == SPARK_PATH_MMA) return mma_ok ? SPARK_PATH_MMA : SPARK_ERR_UNSUPPORTED;
  return mma_ok ? SPARK_PATH_MMA : SPARK_PATH_GEMV;
}

}  // namespace

extern "C" {

size_t spark_mlp_workspace_bytes(const spark_geom* g, int32_t intermediate, int32_t batch) {
  if (check_geom(g) != SPARK_OK || check_batch(batch) != SPARK_OK) return 0;
  if (intermediate != 0 && check_inter(intermediate) != SPARK_OK) return 0;
  if (intermediate < 0) return 0;
  return mlp_ws_layout(g->hidden, intermediate, batch).total;
}

int spark_mlp_decode(const spark_geom* g, const float* h, const spark_mlp_weights* w, int32_t batch,
                     float* out, int32_t path, void* workspace, size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if (!w || check_dtype(w->dtype) != SPARK_OK) return SPARK_ERR_INVALID_ARG;
  if (!w->norm_w || !w->gate_w || !w->up_w || !w->down_w || !aligned16(w->norm_w) || !aligned16(w->gate_w) ||
      !aligned16(w->up_w) || !aligned16(w->down_w))
    return SPARK_ERR_INVALID_ARG;
  if ((s = check_inter(w->intermediate)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_mlp_ws(g, w->intermediate, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !out || !aligned16(h) || !aligned16(out)) return SPARK_ERR_INVALID_ARG;
  const int chosen = pick(path, batch, mma_mlp_supported(w->dtype, g->hidden, w->intermediate));
  if (chosen < 0) return chosen;
  const MlpWsLayout L = mlp_ws_layout(g->hidden, w->intermediate, batch);
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  cudaStream_t st = (cudaStream_t)stream;
  if (chosen == SPARK_PATH_MMA) {
    MmaWorkspace m;
    m.x = ws_at<__nv_bfloat16>(workspace, L.mx);
    m.cs = nullptr;
    m.part = ws_at<float>(workspace, L.mpart);
    m.tickets = ws_at<uint32_t>(workspace, L.mtick);
    m.trace = ws_at<uint64_t>(workspace, L.trace);
    return cuda_status(launch_mlp_mma(h, w->norm_w, w->gate_w, w->up_w, w->down_w, out, err, g->hidden,
                                      w->intermediate, batch, g->eps, m, ws_at<__nv_bfloat16>(workspace, L.md), st));
  }
  return cuda_status(launch_mlp_gemv(w->dtype, h, w->norm_w, w->gate_w, w->up_w, w->down_w,
                                     ws_at<float>(workspace, L.m), out, err, g->hidden, w->intermediate, batch,
                                     g->eps, st));
}

int spark_head_logits(const spark_geom* g, const float* h, const void* norm_w, const void* embed, int32_t vocab,
                      int32_t dtype, int32_t batch, float* logits, int32_t path, void* workspace,
                      size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if (check_dtype(dtype) != SPARK_OK) return SPARK_ERR_INVALID_ARG;
  if (!norm_w || !embed || !aligned16(norm_w) || !aligned16(embed)) return SPARK_ERR_INVALID_ARG;
  if (vocab < 1) return SPARK_ERR_INVALID_ARG;
  if (vocab < 8 || vocab > kMaxVocab || vocab % 8 != 0) return SPARK_ERR_UNSUPPORTED;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_mlp_ws(g, 0, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !logits || !aligned16(h) || !aligned16(logits)) return SPARK_ERR_INVALID_ARG;
  // the head's GEMM is the up GEMM's shape with vocab rows: the same checks
  const int chosen = pick(path, batch, mma_mlp_supported(dtype, g->hidden, vocab));
  if (chosen < 0) return chosen;
  const MlpWsLayout L = mlp_ws_layout(g->hidden, 0, batch);
  uint32_t* err = ws_at<uint32_t>(workspace, L.err);
  cudaStream_t st = (cudaStream_t)stream;
  if (chosen == SPARK_PATH_MMA) {
    MmaWorkspace m;
    m.x = ws_at<__nv_bfloat16>(workspace, L.mx);
    m.cs = nullptr;
    m.part = ws_at<float>(workspace, L.mpart);
    m.tickets = ws_at<uint32_t>(workspace, L.mtick);
    m.trace = ws_at<uint64_t>(workspace, L.trace);
    return cuda_status(launch_head_mma(h, norm_w, embed, logits, err, g->hidden, vocab, batch, g->eps, m, st));
  }
  return cuda_status(launch_head_gemv(dtype, h, norm_w, embed, logits, err, g->hidden, vocab, batch, g->eps, st));
}

}  // extern "C"
