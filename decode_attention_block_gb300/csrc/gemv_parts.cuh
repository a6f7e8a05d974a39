// gemv_parts.cuh -- the pieces of the weight-streaming projections shared by
// the per-layer kernels (proj.cu) and the persistent decode kernel
// (stack.cu): activation layout, packed dot products of 16-byte weight
// chunks, the pairing of q_k_v_proj / g_proj rows for the rope epilogue
// (turbospark-runtime 0.3.0, src/families/spark/attn.rs, module doc items
// 1-2 and encode_attention_block).
#pragma once

#include <math.h>

#include "common.cuh"

namespace spark {

#if defined(__CUDACC__)

template <typename WT>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr int kElems = 4;
};
template <>
struct Chunk<__nv_bfloat16> {
  static constexpr int kElems = 8;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Activation vectors live in shared memory permuted so that lane l's values
// for its 16-byte weight chunk c = l + 32 i are read as consecutive float4s
// across lanes (no bank conflicts): element n of chunk c sits at float4
// ((i * E/4 + (n % E) / 4) * 32 + l), component n % 4.
template <int E>
__device__ __forceinline__ int xperm_index(int n) {
  const int c = n / E, l = c & 31, i = c >> 5, hq = (n % E) >> 2;
  return ((i * (E / 4) + hq) * 32 + l) * 4 + (n & 3);
}

// sum over the chunk of w[k] * x[k], accumulated pairwise into acc
template <typename WT>
__device__ __forceinline__ void dot_chunk(uint4 w, const float4* xp, float2& acc);

template <>
__device__ __forceinline__ void dot_chunk<__nv_bfloat16>(uint4 w, const float4* xp, float2& acc) {
  const float4 x0 = xp[0], x1 = xp[32];
  acc = ffma2(bf16x2_to_f32x2(w.x), make_float2(x0.x, x0.y), acc);
  acc = ffma2(bf16x2_to_f32x2(w.y), make_float2(x0.z, x0.w), acc);
  acc = ffma2(bf16x2_to_f32x2(w.z), make_float2(x1.x, x1.y), acc);
  acc = ffma2(bf16x2_to_f32x2(w.w), make_float2(x1.z, x1.w), acc);
}

template <>
__device__ __forceinline__ void dot_chunk<float>(uint4 w, const float4* xp, float2& acc) {
  const float4 x0 = xp[0];
  acc = ffma2(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), make_float2(x0.x, x0.y), acc);
  acc = ffma2(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), make_float2(x0.z, x0.w), acc);
}

// The same sum with the chunk's activations in registers (E/4 float4s).
template <typename WT>
__device__ __forceinline__ void dot_chunk_reg(uint4 w, const float4* x, float2& acc);

template <>
__device__ __forceinline__ void dot_chunk_reg<__nv_bfloat16>(uint4 w, const float4* x, float2& acc) {
  acc = ffma2(bf16x2_to_f32x2(w.x), make_float2(x[0].x, x[0].y), acc);
  acc = ffma2(bf16x2_to_f32x2(w.y), make_float2(x[0].z, x[0].w), acc);
  acc = ffma2(bf16x2_to_f32x2(w.z), make_float2(x[1].x, x[1].y), acc);
  acc = ffma2(bf16x2_to_f32x2(w.w), make_float2(x[1].z, x[1].w), acc);
}

template <>
__device__ __forceinline__ void dot_chunk_reg<float>(uint4 w, const float4* x, float2& acc) {
  acc = ffma2(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), make_float2(x[0].x, x[0].y), acc);
  acc = ffma2(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), make_float2(x[0].z, x[0].w), acc);
}

// Eight warp sums at once: on entry lane l holds its term v[i] of sum i; on
// exit v[0] on lane l is sum l / 4 (added in a fixed order).  The first three
// rounds halve the values a lane keeps, exchanging the other half with the
// lane 16, 8 and then 4 apart; two more rounds add over the remaining lanes:
// 9 shuffles for eight sums instead of 40.
__device__ __forceinline__ void warp_sums8(float (&v)[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16, n = 4; o >= 4; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const float send = up ? v[i] : v[i + n];
      const float keep = up ? v[i + n] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// Four consecutive weight elements as fp32 (read-only path).
__device__ __forceinline__ float4 load_w4(const float* w, int n) {
  return __ldg(reinterpret_cast<const float4*>(w + n));
}
__device__ __forceinline__ float4 load_w4(const __nv_bfloat16* w, int n) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(w + n));
  const float2 a = bf16x2_to_f32x2(u.x), b = bf16x2_to_f32x2(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

// The RMSNorm weight elements a thread of build_x_norm uses: they do not
// depend on the previous kernel, so a kernel may load them before its
// dependency wait.
template <typename WT, int NT, int MAXPER>
__device__ __forceinline__ void load_norm_w(const WT* w, int n, float4 (&wv)[MAXPER], int t) {
#pragma unroll
  for (int k = 0; k < MAXPER; ++k) {
    const int n4 = 4 * (t + k * NT);
    wv[k] = n4 < n ? load_w4(w, n4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// The activation prologue of the q_k_v_proj GEMV for up to NB sequences:
// xs_b = h_b * w (the RMSNorm's weight; the 1/rms scale is applied to the dot
// products), permuted for row_dot with E-element chunks, and ss[b] = sum h_b^2
// over this thread's elements.  NT threads take float4 groups t, t + NT, ...;
// each thread issues every load before it computes, so the prologue costs one
// memory round trip.  h comes from another CTA or kernel: loads bypass L1.
// wv holds the thread's norm weights (load_norm_w).
template <int E, int NB, int NT, int MAXPER>
__device__ __forceinline__ void build_x_norm_w(const float* h, const float4 (&wv)[MAXPER], int n, int nb,
                                               float* xs, int xfloats, float (&ss)[NB], int t) {
  float4 hv[NB][MAXPER];
#pragma unroll
  for (int k = 0; k < MAXPER; ++k) {
    const int n4 = 4 * (t + k * NT);
    if (n4 < n) {
#pragma unroll
      for (int b = 0; b < NB; ++b)
        hv[b][k] = b < nb ? __ldcg(reinterpret_cast<const float4*>(h + (int64_t)b * n + n4))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) ss[b] = 0.f;
#pragma unroll
  for (int k = 0; k < MAXPER; ++k) {
    const int n4 = 4 * (t + k * NT);
    if (n4 < n) {
      const int pi = xperm_index<E>(n4);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float4 v = hv[b][k];
        ss[b] = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss[b]))));
        *reinterpret_cast<float4*>(xs + b * xfloats + pi) =
            make_float4(v.x * wv[k].x, v.y * wv[k].y, v.z * wv[k].z, v.w * wv[k].w);
      }
    }
  }
}

template <int E, typename WT, int NB, int NT, int MAXPER>
__device__ __forceinline__ void build_x_norm(const float* h, const WT* w, int n, int nb, float* xs,
                                             int xfloats, float (&ss)[NB], int t) {
  float4 wv[MAXPER];
  load_norm_w<WT, NT, MAXPER>(w, n, wv, t);
  build_x_norm_w<E, NB, NT, MAXPER>(h, wv, n, nb, xs, xfloats, ss, t);
}

// The activation prologue of o_proj: xs_b = a_b * sigmoid(g_b[head]) (the
// headwise gate, one scalar per query head broadcast over head_dim), permuted
// as above; all loads issued before any use.  a and g come from other CTAs or
// kernels: loads bypass L1.
template <int E, int NB, int NT, int MAXPER>
__device__ __forceinline__ void build_x_gated(const float* a, const float* g, int q_dim, int n_q,
                                              int nb, float* xs, int xfloats, int t) {
  float4 av[NB][MAXPER];
  float gv[NB][MAXPER];
#pragma unroll
  for (int k = 0; k < MAXPER; ++k) {
    const int n4 = 4 * (t + k * NT);
    if (n4 < q_dim) {
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        av[b][k] = b < nb ? __ldcg(reinterpret_cast<const float4*>(a + (int64_t)b * q_dim + n4))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        gv[b][k] = b < nb ? __ldcg(g + (int64_t)b * n_q + n4 / kHeadDim) : 0.f;
      }
    }
  }
#pragma unroll
  for (int k = 0; k < MAXPER; ++k) {
    const int n4 = 4 * (t + k * NT);
    if (n4 < q_dim) {
      const int pi = xperm_index<E>(n4);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float s = 1.0f / (1.0f + expf(-gv[b][k]));
        const float4 v = av[b][k];
        *reinterpret_cast<float4*>(xs + b * xfloats + pi) = make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
      }
    }
  }
}

enum RowKind { kQ = 0, kK = 1, kV = 2, kG = 3 };

struct Unit {
  int row_a, row_b;  // rows of [q_k_v_proj; g_proj]
  int kind, head;    // head index within its kind
  int da, db;        // output dims of the two rows (within the head, or g index)
  int pair;          // rope pair index (-1: no rotation)
};

__device__ __forceinline__ Unit unit_of(int u, int n_q, int n_kv, int rotary_dim) {
  Unit x;
  const int n_heads = n_q + 2 * n_kv;
  if (u < n_heads * (kHeadDim / 2)) {
    const int hd = u / (kHeadDim / 2), t = u % (kHeadDim / 2);
    x.kind = hd < n_q ? kQ : (hd < n_q + n_kv ? kK : kV);
    x.head = x.kind == kQ ? hd : (x.kind == kK ? hd - n_q : hd - n_q - n_kv);
    const int half = rotary_dim / 2;
    if (x.kind != kV && t < half) {
      x.da = t;
      x.db = t + half;
      x.pair = t;
    } else {
      x.da = x.kind == kV ? 2 * t : rotary_dim + 2 * (t - half);
      x.db = x.da + 1;
      x.pair = -1;
    }
    x.row_a = hd * kHeadDim + x.da;
    x.row_b = hd * kHeadDim + x.db;
  } else {
    const int gi = u - n_heads * (kHeadDim / 2);
    x.kind = kG;
    x.head = 0;
    x.da = 2 * gi;
    x.db = 2 * gi + 1;
    x.pair = -1;
    x.row_a = n_heads * kHeadDim + x.da;
    x.row_b = x.row_a + 1;
  }
  return x;
}

// ---------------------------------------------------------------------------
// per-warp row streaming shared by both kernels
// ---------------------------------------------------------------------------

// Wait for this warp's stage, bounded; on time-out raise the block's abort
// flag and the error word.  Returns false if the stage must not be read.
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           uint32_t* err) {
  if (mbar_wait_bounded(bar, parity, abort_flag, kWaitLimitNs)) return true;
  if ((threadIdx.x & 31) == 0 && !*abort_flag) {
    *abort_flag = 1;
    if (err) atomicOr(err, kErrWaitTimeout);
  }
  return false;
}

// acc[b] (b < NB) += row . x_b for one weight row held in shared memory
template <typename WT, int NB>
__device__ __forceinline__ void row_dot(const unsigned char* row, const float* xs, int xfloats,
                                        int nchunk, float2 (&acc)[NB]) {
  constexpr int E = Chunk<WT>::kElems;
  const int lane = threadIdx.x & 31;
  for (int c = lane, i = 0; c < nchunk; c += 32, ++i) {
    const uint4 w = *reinterpret_cast<const uint4*>(row + (size_t)c * 16);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float4* xp = reinterpret_cast<const float4*>(xs + b * xfloats) + i * (E / 4) * 32 + lane;
      dot_chunk<WT>(w, xp, acc[b]);
    }
  }
}

// two rows sharing one pass over the activation
template <typename WT, int NB>
__device__ __forceinline__ void row_dot2(const unsigned char* ra, const unsigned char* rb,
                                         const float* xs, int xfloats, int nchunk,
                                         float2 (&acc_a)[NB], float2 (&acc_b)[NB]) {
  constexpr int E = Chunk<WT>::kElems;
  const int lane = threadIdx.x & 31;
#pragma unroll 2
  for (int c = lane, i = 0; c < nchunk; c += 32, ++i) {
    const uint4 wa = *reinterpret_cast<const uint4*>(ra + (size_t)c * 16);
    const uint4 wb = *reinterpret_cast<const uint4*>(rb + (size_t)c * 16);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float4* xp = reinterpret_cast<const float4*>(xs + b * xfloats) + i * (E / 4) * 32 + lane;
      dot_chunk<WT>(wa, xp, acc_a[b]);
      dot_chunk<WT>(wb, xp, acc_b[b]);
    }
  }
}

// ---------------------------------------------------------------------------
// host: launch shape of a weight-streaming kernel
// ---------------------------------------------------------------------------

// Stages of a CTA-wide pool of `budget` bytes of shared memory: one per unit
// of the CTA's share when they all fit next to the activations and the
// barriers, so no stage is reused.  Otherwise a multiple of the consuming
// warps: unit k lives in stage k % stages and belongs to warp k % nw, so the
// warp that frees a stage is the one that consumes its next unit and never
// waits on a barrier phase other than the next one (mbarrier parity tells
// only the last two phases apart).  With fewer stages than warps only that
// many warps consume; 0: not even one unit fits.
inline int gemv_stages(size_t budget, int warps, size_t unit_bytes, size_t x_bytes, int max_units) {
  if (x_bytes >= budget) return 0;
  const size_t room = budget - x_bytes;
  int s = (int)(room / (unit_bytes + 8));
  if (s >= max_units) return max_units;
  if (s >= warps) s -= s % warps;
  return s < 1 ? 0 : s;
}

// Shared-memory bytes of nb permuted activation vectors of `cols` elements.
template <typename WT>
inline size_t gemv_xbytes(int cols, int nb) {
  constexpr int E = Chunk<WT>::kElems;
  const int nchunk = cols / E;
  return sizeof(float) * (size_t)nb * ((nchunk + 31) / 32) * 32 * E;
}

#endif  // __CUDACC__

}  // namespace spark
