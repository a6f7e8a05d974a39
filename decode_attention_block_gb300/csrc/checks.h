// checks.h -- host-side argument checks shared by the C entry points: every
// status they return is decided before anything is enqueued (the library's
// counterpart of the pages' RealForwardError::Unsupported,
// src/families/spark/mod.rs, produce_real_spark_inner).
#pragma once

#include <math.h>

#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"

namespace spark {
namespace checks {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int check_geom(const spark_geom* g) {
  if (!g) return SPARK_ERR_INVALID_ARG;
  if (g->head_dim != kHeadDim) return SPARK_ERR_UNSUPPORTED;
  if (g->n_kv < 1 || g->n_kv > 8 || g->n_q != kGroup * g->n_kv) return SPARK_ERR_UNSUPPORTED;
  if (g->hidden < 8 || g->hidden > 8192 || g->hidden % 8 != 0) return SPARK_ERR_UNSUPPORTED;
  if (g->full_rotary_dim < 2 || g->full_rotary_dim > kHeadDim || g->full_rotary_dim % 2 != 0)
    return SPARK_ERR_UNSUPPORTED;
  if (g->window < 1) return SPARK_ERR_INVALID_ARG;
  if (!(g->full_theta > 0.f) || !(g->sliding_theta > 0.f) || !isfinite(g->full_theta) ||
      !isfinite(g->sliding_theta))
    return SPARK_ERR_INVALID_ARG;
  if (!(g->eps >= 0.f) || !isfinite(g->eps) || !isfinite(g->scale)) return SPARK_ERR_INVALID_ARG;
  return SPARK_OK;
}

inline int check_dtype(int32_t dt) { return (dt == SPARK_F32 || dt == SPARK_BF16) ? SPARK_OK : SPARK_ERR_INVALID_ARG; }

inline int check_weights(const spark_layer_weights* w, bool need_qkv, bool need_o) {
  if (!w) return SPARK_ERR_INVALID_ARG;
  if (check_dtype(w->dtype) != SPARK_OK) return SPARK_ERR_INVALID_ARG;
  if (need_qkv && (!w->norm_w || !w->qkv_w || !w->g_w)) return SPARK_ERR_INVALID_ARG;
  if (need_qkv && (!aligned16(w->norm_w) || !aligned16(w->qkv_w) || !aligned16(w->g_w)))
    return SPARK_ERR_INVALID_ARG;
  if (need_o && (!w->o_w || !aligned16(w->o_w))) return SPARK_ERR_INVALID_ARG;
  return SPARK_OK;
}

inline int check_batch(int32_t batch) {
  return (batch >= 1 && batch <= SPARK_MAX_BATCH) ? SPARK_OK : SPARK_ERR_INVALID_ARG;
}

// The KV layer against the class and the positions: every row a call writes
// or reads must lie inside the buffer.
inline int check_kv(const spark_geom* g, const spark_kv_layer* kv, int32_t cls, const int32_t* positions,
             int32_t batch) {
  if (!kv || !positions) return SPARK_ERR_INVALID_ARG;
  if (cls != SPARK_FULL && cls != SPARK_SLIDING) return SPARK_ERR_INVALID_ARG;
  if (!kv->k || !kv->v || !aligned16(kv->k) || !aligned16(kv->v)) return SPARK_ERR_INVALID_ARG;
  if (check_dtype(kv->dtype) != SPARK_OK) return SPARK_ERR_INVALID_ARG;
  if (kv->capacity < 1 || kv->ring_capacity < 0) return SPARK_ERR_INVALID_ARG;
  if (kv->ring_capacity > 0) {
    if (cls == SPARK_FULL) return SPARK_ERR_BAD_RING;  // a full layer reads its whole history
    if (kv->ring_capacity > kv->capacity) return SPARK_ERR_INVALID_ARG;
    if (kv->ring_capacity < g->window) return SPARK_ERR_BAD_RING;  // would evict live rows
  }
  // TMA coordinates of cache rows are 32-bit
  if ((int64_t)batch * kv->capacity >= ((int64_t)1 << 31)) return SPARK_ERR_UNSUPPORTED;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t p = positions[b];
    if (p < 0 || p >= INT32_MAX - 1) return SPARK_ERR_POSITION;
    if (kv->ring_capacity == 0 && (int64_t)p >= kv->capacity) return SPARK_ERR_POSITION;
  }
  return SPARK_OK;
}

inline int check_ws(const spark_geom* g, int32_t batch, void* ws, size_t bytes) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SPARK_ERR_WORKSPACE;
  if (bytes < ws_layout(g->hidden, g->n_q, g->n_kv, batch).total) return SPARK_ERR_WORKSPACE;
  return SPARK_OK;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? SPARK_OK : SPARK_ERR_CUDA; }

template <typename T>
inline T* ws_at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<unsigned char*>(ws) + off);
}

inline void rope_for(const spark_geom* g, int32_t cls, int* rotary_dim, double* theta) {
  // attn.rs, rope_params_for
  if (cls == SPARK_FULL) {
    *rotary_dim = g->full_rotary_dim;
    *theta = (double)g->full_theta;
  } else {
    *rotary_dim = g->head_dim;
    *theta = (double)g->sliding_theta;
  }
}

// cos and sin of the rope angles position * theta^(-2i/r), i < r/2, for the
// first nb positions, computed in double on the host (at position 131072 an
// fp32 angle would be off by ~1e-2 rad) and handed to the kernels as fp32
// pairs: cs[b * stride + i] = (cos, sin).
// theta^(-2i/r) for i < r/2, in double, computed once per (r, theta)
inline const std::vector<double>& rope_inv_freq(int rotary_dim, double theta) {
  static std::mutex mu;
  static std::map<std::pair<int, double>, std::vector<double>> memo;
  std::lock_guard<std::mutex> lock(mu);
  std::vector<double>& f = memo[std::make_pair(rotary_dim, theta)];
  if (f.empty())
    for (int i = 0; i < rotary_dim / 2; ++i) f.push_back(pow(theta, -2.0 * i / (double)rotary_dim));
  return f;  // entries of a std::map stay where they are
}

inline void fill_rope_table(float2* cs, int stride, int nb, const int32_t* positions, int rotary_dim,
                            double theta) {
  const std::vector<double>& inv_freq = rope_inv_freq(rotary_dim, theta);
  for (int b = 0; b < nb; ++b)
    for (int i = 0; i < stride; ++i) {
      if (i < rotary_dim / 2) {
        const double ang = (double)positions[b] * inv_freq[i];
        cs[b * stride + i] = make_float2((float)cos(ang), (float)sin(ang));
      } else {
        cs[b * stride + i] = make_float2(1.f, 0.f);
      }
    }
}

}  // namespace checks
}  // namespace spark
