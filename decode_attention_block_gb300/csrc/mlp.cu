// mlp.cu -- the MLP half of a decoder layer and the model's head at small
// batch, as weight-streaming GEMV kernels (turbospark-runtime 0.3.0,
// src/families/spark/mod.rs: the module doc's transcription of one layer,
// x = rms(h, post_attention_layernorm, 1e-6) and
// h = h + down(gelu_erf(x @ gate_proj) * (x @ up_proj)); its last two lines,
// the final rms(h, model.norm, 1e-6) and logits = h @ embed_tokens with the
// head tied to the embedding; produce_real_spark's layer loop and head).
//
//  * up    RMSNorm + gate_proj + up_proj + the exact GELU product.  A unit
//          is the pair (gate row j, up row j), so the warp that finishes it
//          holds both dot products and writes m_j = gelu(g_j) * u_j.
//  * down  down_proj + the residual add: out = h + W_down m.
//  * head  final RMSNorm + the tied head: one row of the embedding per logit.
//
// Same streaming scheme as the attention block's projections (proj.cu): one
// CTA per SM owns a contiguous share of the units, the rows arrive by 1-D bulk
// copies into a pool of shared-memory stages requested before the kernel
// waits on its predecessor, and the RMSNorm's 1/rms scale is applied to the
// finished dot products.  The GELU is z/2 (1 + erf(z / sqrt 2)) with CUDA's
// erff.
#include <math.h>

#include "gemv_parts.cuh"
#include "launch.h"

namespace spark {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPer = 8192 / 4 / kThreads;  // float4 of a normed activation per thread
constexpr size_t kSmemBudget = 200 * 1024;
constexpr int kMaxChunk = 4;                   // sequences per launch (up, head)

enum GemvKind { kUp = 0, kHead = 1, kDown = 2 };

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

// xs_b = m_b permuted for row_dot (no scaling); every thread issues kU float4
// loads per sequence before it stores any (12 / NB: one round trip for a
// 10240-float vector of one sequence).  m comes from another kernel: loads
// bypass L1.
template <int E, int NB>
__device__ __forceinline__ void build_x_plain(const float* m, int n, int nb, float* xs, int xfloats, int t) {
  constexpr int kU = 12 / NB;
  for (int base = t; 4 * base < n; base += kU * kThreads) {
    float4 v[NB][kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int n4 = 4 * (base + u * kThreads);
#pragma unroll
      for (int b = 0; b < NB; ++b)
        v[b][u] = (n4 < n && b < nb) ? __ldcg(reinterpret_cast<const float4*>(m + (int64_t)b * n + n4))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int n4 = 4 * (base + u * kThreads);
      if (n4 < n) {
        const int pi = xperm_index<E>(n4);
#pragma unroll
        for (int b = 0; b < NB; ++b) *reinterpret_cast<float4*>(xs + b * xfloats + pi) = v[b][u];
      }
    }
  }
}

// One weight-streaming GEMV of kind KIND over `cols` input elements and
// `n_units` output units (pairs of rows for kUp), for nb <= NB sequences.
//   in     h [nb][cols] (kUp, kHead) or m [nb][cols] (kDown)
//   wa     gate_proj (kUp), embed_tokens (kHead), down_proj (kDown); wb up_proj
//   res    h [nb][n_units] (kDown: the residual)
//   out    m [nb][n_units] (kUp), logits [nb][n_units] (kHead), h' (kDown; may be res)
template <typename WT, int NB, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    k_mlp_gemv(const float* __restrict__ in, const WT* __restrict__ norm_w, const WT* __restrict__ wa,
               const WT* __restrict__ wb, const float* res, float* out, uint32_t* err, int cols,
               int n_units, int nb, int stages, float eps) {
  constexpr int E = Chunk<WT>::kElems;
  constexpr int kRows = KIND == kUp ? 2 : 1;  // weight rows per unit
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = cols / E;
  const int xfloats = ((nchunk + 31) / 32) * 32 * E;
  const size_t row_bytes = (size_t)cols * sizeof(WT);
  const size_t unit_bytes = kRows * row_bytes;
  float* xs = reinterpret_cast<float*>(smem);  // [NB][xfloats]
  unsigned char* pool = smem + sizeof(float) * NB * xfloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(pool + (size_t)stages * unit_bytes);
  __shared__ float red[kWarps][NB];
  __shared__ float inv_rms[NB];
  __shared__ int abort_flag;

  const int u0 = (int)((int64_t)n_units * blockIdx.x / gridDim.x);
  const int u1 = (int)((int64_t)n_units * (blockIdx.x + 1) / gridDim.x);
  const int cnt = u1 - u0;
  const int nw = stages < kWarps ? stages : kWarps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  auto issue = [&](int k) {
    const int s = k % stages;
    unsigned char* dst = pool + (size_t)s * unit_bytes;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)unit_bytes);
    bulk_load(dst, wa + (int64_t)(u0 + k) * cols, (uint32_t)row_bytes, &bars[s]);
    if (KIND == kUp) bulk_load(dst + row_bytes, wb + (int64_t)(u0 + k) * cols, (uint32_t)row_bytes, &bars[s]);
  };
  // the weight stream does not depend on the previous kernel
  if (lane == 0 && warp < nw)
    for (int k = warp; k < stages && k < cnt; k += nw) issue(k);
  __syncwarp();  // every lane waits only once its warp's requests are out
  pdl_wait();
  pdl_trigger();  // the next kernel starts only once the one before this has completed

  if (KIND == kDown) {
    build_x_plain<E, NB>(in, cols, nb, xs, xfloats, threadIdx.x);
    if (threadIdx.x < NB) inv_rms[threadIdx.x] = 1.0f;
  } else {
    float ss[NB];
    build_x_norm<E, WT, NB, kThreads, kMaxPer>(in, norm_w, cols, nb, xs, xfloats, ss, threadIdx.x);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float v = warp_sum(ss[b]);
      if (lane == 0) red[warp][b] = v;
    }
    __syncthreads();
    if (threadIdx.x < NB) {
      float t = 0.f;
      for (int w = 0; w < kWarps; ++w) t += red[w][threadIdx.x];
      inv_rms[threadIdx.x] = 1.0f / sqrtf(t / (float)cols + eps);
    }
  }
  __syncthreads();

  for (int k = warp; warp < nw && k < cnt; k += nw) {
    const int s = k % stages;
    const uint32_t parity = (uint32_t)((k / stages) & 1);
    float2 acc_a[NB], acc_b[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc_a[b] = acc_b[b] = make_float2(0.f, 0.f);
    const bool ok = wait_stage(&bars[s], parity, &abort_flag, err);
    if (ok) {
      const unsigned char* st = pool + (size_t)s * unit_bytes;
      if (KIND == kUp)
        row_dot2<WT, NB>(st, st + row_bytes, xs, xfloats, nchunk, acc_a, acc_b);
      else
        row_dot<WT, NB>(st, xs, xfloats, nchunk, acc_a);
    }
    __syncwarp();
    if (ok && lane == 0 && k + stages < cnt) issue(k + stages);
    if (!ok) continue;
    float va = 0.f, vb = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sa = warp_sum(acc_a[b].x + acc_a[b].y);
      const float sb = KIND == kUp ? warp_sum(acc_b[b].x + acc_b[b].y) : 0.f;
      if (lane == b) {
        va = sa * inv_rms[b];
        vb = sb * inv_rms[b];
      }
    }
    if (lane < nb) {
      const int64_t idx = (int64_t)lane * n_units + u0 + k;
      if (KIND == kUp)
        out[idx] = gelu_erf(va) * vb;
      else if (KIND == kHead)
        out[idx] = va;
      else
        out[idx] = res[idx] + va;  // read and written by the same thread: out may alias res
    }
  }
}

template <typename WT, int NB, int KIND>
cudaError_t gemv_launch(const float* in, const void* norm_w, const void* wa, const void* wb,
                        const float* res, float* out, uint32_t* err, int cols, int n_units, int nb,
                        float eps, cudaStream_t st) {
  const size_t unit_bytes = (KIND == kUp ? 2 : 1) * (size_t)cols * sizeof(WT);
  const size_t xb = gemv_xbytes<WT>(cols, NB);
  int grid = device_sm_count();
  if (grid > n_units) grid = n_units;
  const int stages = gemv_stages(kSmemBudget, kWarps, unit_bytes, xb, (n_units + grid - 1) / grid);
  if (stages == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = xb + (size_t)stages * (unit_bytes + 8);
  auto kern = k_mlp_gemv<WT, NB, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, in, (const WT*)norm_w, (const WT*)wa,
                    (const WT*)wb, res, out, err, cols, n_units, nb, stages, eps);
}

template <typename WT, int KIND>
cudaError_t gemv_chunk(int nb, const float* in, const void* norm_w, const void* wa, const void* wb,
                       const float* res, float* out, uint32_t* err, int cols, int n_units, float eps,
                       cudaStream_t st) {
  if (nb == 1) return gemv_launch<WT, 1, KIND>(in, norm_w, wa, wb, res, out, err, cols, n_units, nb, eps, st);
  if (nb == 2) return gemv_launch<WT, 2, KIND>(in, norm_w, wa, wb, res, out, err, cols, n_units, nb, eps, st);
  return gemv_launch<WT, 4, KIND>(in, norm_w, wa, wb, res, out, err, cols, n_units, nb, eps, st);
}

// Sequences per down_proj launch: 2 while the two activation vectors (each
// intermediate floats long) leave a pool of at least 4 rows -- at ~150 SMs
// that keeps well over the HBM's bandwidth-latency product in flight -- else 1.
template <typename WT>
int down_chunk(int inter) {
  const size_t unit = (size_t)inter * sizeof(WT);
  return gemv_stages(kSmemBudget, kWarps, unit, gemv_xbytes<WT>(inter, 2), 1 << 30) >= 4 ? 2 : 1;
}

template <typename WT>
cudaError_t mlp_gemv(const float* h, const void* norm_w, const void* gate_w, const void* up_w,
                     const void* down_w, float* m, float* out, uint32_t* err, int hidden, int inter,
                     int batch, float eps, cudaStream_t st) {
  for (int b0 = 0; b0 < batch; b0 += kMaxChunk) {
    const int nb = batch - b0 < kMaxChunk ? batch - b0 : kMaxChunk;
    cudaError_t e = gemv_chunk<WT, kUp>(nb, h + (int64_t)b0 * hidden, norm_w, gate_w, up_w, nullptr,
                                        m + (int64_t)b0 * inter, err, hidden, inter, eps, st);
    if (e != cudaSuccess) return e;
  }
  const int cd = down_chunk<WT>(inter);
  for (int b0 = 0; b0 < batch; b0 += cd) {
    const int nb = batch - b0 < cd ? batch - b0 : cd;
    cudaError_t e = gemv_chunk<WT, kDown>(nb, m + (int64_t)b0 * inter, nullptr, down_w, nullptr,
                                          h + (int64_t)b0 * hidden, out + (int64_t)b0 * hidden, err,
                                          inter, hidden, eps, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename WT>
cudaError_t head_gemv(const float* h, const void* norm_w, const void* embed, float* logits, uint32_t* err,
                      int hidden, int vocab, int batch, float eps, cudaStream_t st) {
  for (int b0 = 0; b0 < batch; b0 += kMaxChunk) {
    const int nb = batch - b0 < kMaxChunk ? batch - b0 : kMaxChunk;
    cudaError_t e = gemv_chunk<WT, kHead>(nb, h + (int64_t)b0 * hidden, norm_w, embed, nullptr, nullptr,
                                          logits + (int64_t)b0 * vocab, err, hidden, vocab, eps, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_mlp_gemv(int wdtype, const float* h, const void* norm_w, const void* gate_w,
                            const void* up_w, const void* down_w, float* m, float* out, uint32_t* err,
                            int hidden, int inter, int batch, float eps, cudaStream_t st) {
  return wdtype == SPARK_BF16
             ? mlp_gemv<__nv_bfloat16>(h, norm_w, gate_w, up_w, down_w, m, out, err, hidden, inter, batch, eps, st)
             : mlp_gemv<float>(h, norm_w, gate_w, up_w, down_w, m, out, err, hidden, inter, batch, eps, st);
}

cudaError_t launch_head_gemv(int wdtype, const float* h, const void* norm_w, const void* embed,
                             float* logits, uint32_t* err, int hidden, int vocab, int batch, float eps,
                             cudaStream_t st) {
  return wdtype == SPARK_BF16
             ? head_gemv<__nv_bfloat16>(h, norm_w, embed, logits, err, hidden, vocab, batch, eps, st)
             : head_gemv<float>(h, norm_w, embed, logits, err, hidden, vocab, batch, eps, st);
}

}  // namespace spark
