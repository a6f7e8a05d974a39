// proj.cu -- the block's two weight-streaming projections.
//
//  * qkv_gate: input RMSNorm fused with the q_k_v_proj GEMV and the g_proj
//    GEMV (turbospark-runtime 0.3.0, src/families/spark/attn.rs,
//    encode_attention_block: "the fused projection, as one GEMV" and "the
//    gate's projection" that reads the same normed x; src/families/spark/
//    mod.rs, "One decoder layer, transcribed": x = rms(h, w, 1e-6), plain w).
//  * gate_oproj: the headwise sigmoid gate fused with the o_proj GEMV and the
//    raw residual add (attn.rs: encode_sigmoid_head_gate_mul before o_proj;
//    mod.rs: encode_residual_add).
//
// Both are HBM-bound at small batch: each weight byte is read once and used
// for `batch` FMAs.  One warp owns kRowsPerWarp rows, streams them with
// 16-byte non-allocating loads and keeps the normalised activation vector of
// up to kBatchChunk sequences in shared memory; larger batches are processed
// in chunks of kBatchChunk.
#include "launch.h"

namespace spark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsPerWarp = 2;
constexpr int kBatchChunk = 4;

template <typename WT>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr int kElems = 4;
  __device__ __forceinline__ static void unpack(uint4 v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
};
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kElems = 8;
  __device__ __forceinline__ static void unpack(uint4 v, float* f) {
    float2 a = bf16x2_to_f32x2(v.x), b = bf16x2_to_f32x2(v.y);
    float2 c = bf16x2_to_f32x2(v.z), d = bf16x2_to_f32x2(v.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) t += red[i];
  return t;
}

// acc[r][b] += W[row0 + r, :] . xs[b, :] for r < nrows, b < nb; the warp's
// lanes stride over 16-byte chunks of the rows, four chunks in flight per row.
template <typename WT>
__device__ __forceinline__ void warp_rows_dot(const WT* __restrict__ W, int64_t ld, int row0,
                                              int nrows, const float* __restrict__ xs, int cols,
                                              int nb, float (&acc)[kRowsPerWarp][kBatchChunk]) {
  constexpr int E = Chunk<WT>::kElems;
  constexpr int U = 4;
  const int lane = threadIdx.x & 31;
  const int nchunk = cols / E;
  const WT* rp[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) rp[r] = W + (int64_t)(row0 + (r < nrows ? r : 0)) * ld;

  int c = lane;
  for (; c + 32 * (U - 1) < nchunk; c += 32 * U) {
    uint4 wv[U][kRowsPerWarp];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) wv[u][r] = ld_stream_u4(rp[r] + (c + 32 * u) * E);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float wf[kRowsPerWarp][E];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) Chunk<WT>::unpack(wv[u][r], wf[r]);
#pragma unroll
      for (int b = 0; b < kBatchChunk; ++b) {
        if (b < nb) {
          const float* xp = xs + b * cols + (c + 32 * u) * E;
#pragma unroll
          for (int e = 0; e < E; e += 4) {
            const float4 x4 = *reinterpret_cast<const float4*>(xp + e);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
              acc[r][b] = fmaf(wf[r][e + 0], x4.x, acc[r][b]);
              acc[r][b] = fmaf(wf[r][e + 1], x4.y, acc[r][b]);
              acc[r][b] = fmaf(wf[r][e + 2], x4.z, acc[r][b]);
              acc[r][b] = fmaf(wf[r][e + 3], x4.w, acc[r][b]);
            }
          }
        }
      }
    }
  }
  for (; c < nchunk; c += 32) {
    float wf[kRowsPerWarp][E];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) Chunk<WT>::unpack(ld_stream_u4(rp[r] + c * E), wf[r]);
#pragma unroll
    for (int b = 0; b < kBatchChunk; ++b) {
      if (b < nb) {
        const float* xp = xs + b * cols + c * E;
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 x4 = *reinterpret_cast<const float4*>(xp + e);
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            acc[r][b] = fmaf(wf[r][e + 0], x4.x, acc[r][b]);
            acc[r][b] = fmaf(wf[r][e + 1], x4.y, acc[r][b]);
            acc[r][b] = fmaf(wf[r][e + 2], x4.z, acc[r][b]);
            acc[r][b] = fmaf(wf[r][e + 3], x4.w, acc[r][b]);
          }
        }
      }
    }
  }
}

// Rows [0, rows_qkv) come from q_k_v_proj, rows [rows_qkv, rows_qkv + n_q)
// from g_proj; rows_qkv is a multiple of kRowsPerWarp, so a warp never
// straddles the two matrices.
template <typename WT>
__global__ void __launch_bounds__(kThreads)
    k_qkv_gate(const float* __restrict__ h, const WT* __restrict__ norm_w,
               const WT* __restrict__ qkv_w, const WT* __restrict__ g_w,
               float* __restrict__ qkvg, int hidden, int rows_qkv, int rows_g, int batch,
               float eps) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [kBatchChunk][hidden]
  __shared__ float red[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows_total = rows_qkv + rows_g;
  const int ld_out = rows_total;
  const int row0 = (blockIdx.x * kWarps + warp) * kRowsPerWarp;

  for (int b0 = 0; b0 < batch; b0 += kBatchChunk) {
    const int nb = min(kBatchChunk, batch - b0);
    __syncthreads();
    for (int bb = 0; bb < nb; ++bb) {
      const float* hb = h + (int64_t)(b0 + bb) * hidden;
      float ss = 0.f;
      for (int i = threadIdx.x; i < hidden; i += kThreads) {
        const float v = hb[i];
        ss = fmaf(v, v, ss);
      }
      ss = block_sum(ss, red);
      const float inv = 1.0f / sqrtf(ss / (float)hidden + eps);
      for (int i = threadIdx.x; i < hidden; i += kThreads)
        xs[bb * hidden + i] = hb[i] * inv * to_f32(norm_w[i]);
    }
    __syncthreads();
    if (row0 < rows_total) {
      float acc[kRowsPerWarp][kBatchChunk];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) acc[r][b] = 0.f;
      const bool is_g = row0 >= rows_qkv;
      const WT* W = is_g ? g_w : qkv_w;
      const int wrow0 = is_g ? row0 - rows_qkv : row0;
      const int nrows = min(kRowsPerWarp, (is_g ? rows_g : rows_qkv) - wrow0);
      warp_rows_dot<WT>(W, hidden, wrow0, nrows, xs, hidden, nb, acc);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) {
          const float v = warp_sum(acc[r][b]);
          if (lane == 0 && r < nrows && b < nb) qkvg[(int64_t)(b0 + b) * ld_out + row0 + r] = v;
        }
    }
  }
}

template <typename WT>
__global__ void __launch_bounds__(kThreads)
    k_gate_oproj(const float* __restrict__ a, const float* __restrict__ qkvg, int qkvg_ld,
                 int g_col, const float* h, const WT* __restrict__ o_w, float* out, int hidden,
                 int q_dim, int batch) {
  extern __shared__ float4 smem_f4[];
  float* xs = reinterpret_cast<float*>(smem_f4);  // [kBatchChunk][q_dim]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = (blockIdx.x * kWarps + warp) * kRowsPerWarp;

  for (int b0 = 0; b0 < batch; b0 += kBatchChunk) {
    const int nb = min(kBatchChunk, batch - b0);
    __syncthreads();
    for (int bb = 0; bb < nb; ++bb) {
      const float* ab = a + (int64_t)(b0 + bb) * q_dim;
      const float* gb = qkvg + (int64_t)(b0 + bb) * qkvg_ld + g_col;
      for (int i = threadIdx.x; i < q_dim; i += kThreads) {
        const float z = gb[i / kHeadDim];
        xs[bb * q_dim + i] = ab[i] * (1.0f / (1.0f + expf(-z)));
      }
    }
    __syncthreads();
    if (row0 < hidden) {
      float acc[kRowsPerWarp][kBatchChunk];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) acc[r][b] = 0.f;
      const int nrows = min(kRowsPerWarp, hidden - row0);
      warp_rows_dot<WT>(o_w, q_dim, row0, nrows, xs, q_dim, nb, acc);
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
        for (int b = 0; b < kBatchChunk; ++b) {
          const float v = warp_sum(acc[r][b]);
          if (lane == 0 && r < nrows && b < nb) {
            const int64_t i = (int64_t)(b0 + b) * hidden + row0 + r;
            out[i] = h[i] + v;  // each element read and written by the same thread: out may alias h
          }
        }
    }
  }
}

template <typename Kern>
cudaError_t set_smem(Kern k, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace

cudaError_t launch_qkv_gate(int wdtype, const float* h, const void* norm_w, const void* qkv_w,
                            const void* g_w, float* qkvg, int hidden, int n_q, int n_kv,
                            int batch, float eps, cudaStream_t st) {
  const int rows_qkv = n_q * kHeadDim + 2 * n_kv * kHeadDim;
  const int rows_total = rows_qkv + n_q;
  const int rows_per_block = kWarps * kRowsPerWarp;
  const dim3 grid((rows_total + rows_per_block - 1) / rows_per_block);
  const size_t smem = sizeof(float) * (size_t)kBatchChunk * hidden;
  cudaError_t e;
  if (wdtype == SPARK_BF16) {
    auto k = k_qkv_gate<__nv_bfloat16>;
    if ((e = set_smem(k, smem)) != cudaSuccess) return e;
    k<<<grid, kThreads, smem, st>>>(h, (const __nv_bfloat16*)norm_w,
                                    (const __nv_bfloat16*)qkv_w, (const __nv_bfloat16*)g_w,
                                    qkvg, hidden, rows_qkv, n_q, batch, eps);
  } else {
    auto k = k_qkv_gate<float>;
    if ((e = set_smem(k, smem)) != cudaSuccess) return e;
    k<<<grid, kThreads, smem, st>>>(h, (const float*)norm_w, (const float*)qkv_w,
                                    (const float*)g_w, qkvg, hidden, rows_qkv, n_q, batch, eps);
  }
  return cudaGetLastError();
}

cudaError_t launch_gate_oproj(int wdtype, const float* a, const float* qkvg, const float* h,
                              const void* o_w, float* out, int hidden, int n_q, int n_kv,
                              int batch, cudaStream_t st) {
  const int q_dim = n_q * kHeadDim;
  const int ld = qkvg_ld(n_q, n_kv);
  const int g_col = n_q * kHeadDim + 2 * n_kv * kHeadDim;
  const int rows_per_block = kWarps * kRowsPerWarp;
  const dim3 grid((hidden + rows_per_block - 1) / rows_per_block);
  const size_t smem = sizeof(float) * (size_t)kBatchChunk * q_dim;
  cudaError_t e;
  if (wdtype == SPARK_BF16) {
    auto k = k_gate_oproj<__nv_bfloat16>;
    if ((e = set_smem(k, smem)) != cudaSuccess) return e;
    k<<<grid, kThreads, smem, st>>>(a, qkvg, ld, g_col, h, (const __nv_bfloat16*)o_w, out,
                                    hidden, q_dim, batch);
  } else {
    auto k = k_gate_oproj<float>;
    if ((e = set_smem(k, smem)) != cudaSuccess) return e;
    k<<<grid, kThreads, smem, st>>>(a, qkvg, ld, g_col, h, (const float*)o_w, out, hidden,
                                    q_dim, batch);
  }
  return cudaGetLastError();
}

}  // namespace spark
