// launch.h -- host launchers of the block's kernels (internal to the library).
#pragma once

#include "common.cuh"

namespace spark {

// Input RMSNorm + q_k_v_proj + g_proj: qkvg[b] = [W_qkv; W_g] @ rms(h[b]) * w.
cudaError_t launch_qkv_gate(int wdtype, const float* h, const void* norm_w, const void* qkv_w,
                            const void* g_w, float* qkvg, int hidden, int n_q, int n_kv,
                            int batch, float eps, cudaStream_t st);

// Head gate + o_proj + raw residual: out[b] = h[b] + W_o @ (a[b] * sigmoid(g[b])).
cudaError_t launch_gate_oproj(int wdtype, const float* a, const float* qkvg, const float* h,
                              const void* o_w, float* out, int hidden, int n_q, int n_kv,
                              int batch, cudaStream_t st);

// Split + NeoX rope (q and k) + cache-row write of k and v.
cudaError_t launch_split_rope(int cdtype, const float* qkvg, float* q_rot, void* kc, void* vc,
                              int n_q, int n_kv, int64_t capacity, int ring_capacity,
                              int rotary_dim, double theta, const int32_t* positions, int batch,
                              uint32_t* err, cudaStream_t st);

// Split-K GQA decode attention with the log-sum-exp merge.
cudaError_t launch_attention(int cdtype, const float* q_rot, const void* kc, const void* vc,
                             int n_kv, int64_t capacity, int ring_capacity, bool full,
                             int window, float scale, const int32_t* positions, int batch,
                             float* a, float* part, uint32_t* counters, uint32_t* err,
                             int n_ctas, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace spark
