// rope.cu -- the split of the fused projection, the per-class NeoX rope and
// the cache-row write (turbospark-runtime 0.3.0, src/families/spark/attn.rs,
// encode_attention_block: encode_split_qkv puts q in scratch and k, v
// straight into their cache slots; encode_rope_neox_subdim then rotates q and
// the k slot; module doc item 2: the frequency divisor is the rotary dim).
//
// One CTA per (head, sequence) with one thread per output-dim pair.  The rope
// angle position * theta^(-2i/r) is formed in fp64 from fp64 frequencies the
// host computes once, reduced modulo 2*pi in fp64, and only then handed to
// fp32 sincosf: at position 131072 an fp32 angle would be off by ~1e-2 rad.
// k is rotated in fp32 and rounded once to the cache's element type.
#include "launch.h"

namespace spark {
namespace {

constexpr int kMaxRotaryHalf = kHeadDim / 2;

template <int MAXB>
struct RopeArgs {
  double inv_freq[kMaxRotaryHalf];  // theta^(-2i/r), i < r/2
  int32_t pos[MAXB];
};

__device__ __forceinline__ void store_elem(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// cos / sin of position * inv_freq, with the product reduced mod 2*pi in fp64
__device__ __forceinline__ void rope_cos_sin(int32_t pos, double inv_freq, float* c, float* s) {
  constexpr double kTwoPiHi = 6.283185307179586232;      // 2*pi rounded to double
  constexpr double kTwoPiLo = 2.4492935982947064e-16;    // 2*pi - kTwoPiHi
  constexpr double kInvTwoPi = 0.15915494309189533577;
  const double phi = (double)pos * inv_freq;
  const double n = rint(phi * kInvTwoPi);
  double r = fma(-n, kTwoPiHi, phi);
  r = fma(-n, kTwoPiLo, r);
  sincosf((float)r, s, c);
}

template <typename CT, int MAXB>
__global__ void __launch_bounds__(kHeadDim / 2)
    k_split_rope(const float* __restrict__ qkvg, int ld, float* __restrict__ q_rot,
                 CT* __restrict__ kc, CT* __restrict__ vc, int n_q, int n_kv, int64_t capacity,
                 int ring_capacity, int rotary_dim, uint32_t* err,
                 const __grid_constant__ RopeArgs<MAXB> args) {
  __shared__ float u[kHeadDim];
  const int hh = blockIdx.x;  // 0..n_q-1: q heads, then n_kv k heads, then n_kv v heads
  const int b = blockIdx.y;
  const int t = threadIdx.x;
  const int32_t p = args.pos[b];
  const float* src = qkvg + (int64_t)b * ld + (int64_t)hh * kHeadDim;
  const bool is_v = hh >= n_q + n_kv;
  u[t] = src[t];
  u[t + kHeadDim / 2] = src[t + kHeadDim / 2];
  __syncthreads();

  float out[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int d = t + k * (kHeadDim / 2);
    const int half = rotary_dim / 2;
    if (is_v || d >= rotary_dim) {
      out[k] = u[d];
    } else {
      const int i = d < half ? d : d - half;
      float c, s;
      rope_cos_sin(p, args.inv_freq[i], &c, &s);
      out[k] = d < half ? u[d] * c - u[d + half] * s : u[d] * c + u[i] * s;
    }
  }

  if (hh < n_q) {
    float* dst = q_rot + ((int64_t)b * n_q + hh) * kHeadDim;
    dst[t] = out[0];
    dst[t + kHeadDim / 2] = out[1];
    return;
  }
  const int j = is_v ? hh - n_q - n_kv : hh - n_q;
  const int64_t slot = write_slot_of(p, ring_capacity);
  if (p < 0 || slot >= capacity) {  // the host rejects such positions; never write out of bounds
    if (t == 0 && err) atomicOr(err, kErrIndex);
    return;
  }
  CT* dst = (is_v ? vc : kc) + (((int64_t)b * capacity + slot) * n_kv + j) * kHeadDim;
  store_elem(dst + t, out[0]);
  store_elem(dst + t + kHeadDim / 2, out[1]);
}

template <typename CT, int MAXB>
cudaError_t launch_t(const float* qkvg, float* q_rot, void* kc, void* vc, int n_q, int n_kv,
                     int64_t capacity, int ring_capacity, int rotary_dim, double theta,
                     const int32_t* positions, int batch, uint32_t* err, cudaStream_t st) {
  RopeArgs<MAXB> args;
  for (int i = 0; i < kMaxRotaryHalf; ++i)
    args.inv_freq[i] = i < rotary_dim / 2 ? pow(theta, -2.0 * i / (double)rotary_dim) : 0.0;
  for (int b = 0; b < MAXB; ++b) args.pos[b] = b < batch ? positions[b] : 0;
  const dim3 grid(n_q + 2 * n_kv, batch);
  k_split_rope<CT, MAXB><<<grid, kHeadDim / 2, 0, st>>>(qkvg, qkvg_ld(n_q, n_kv), q_rot, (CT*)kc,
                                                         (CT*)vc, n_q, n_kv, capacity,
                                                         ring_capacity, rotary_dim, err, args);
  return cudaGetLastError();
}

template <typename CT>
cudaError_t launch_ct(const float* qkvg, float* q_rot, void* kc, void* vc, int n_q, int n_kv,
                      int64_t capacity, int ring_capacity, int rotary_dim, double theta,
                      const int32_t* positions, int batch, uint32_t* err, cudaStream_t st) {
  if (batch <= 8)
    return launch_t<CT, 8>(qkvg, q_rot, kc, vc, n_q, n_kv, capacity, ring_capacity, rotary_dim,
                           theta, positions, batch, err, st);
  if (batch <= 64)
    return launch_t<CT, 64>(qkvg, q_rot, kc, vc, n_q, n_kv, capacity, ring_capacity, rotary_dim,
                            theta, positions, batch, err, st);
  return launch_t<CT, SPARK_MAX_BATCH>(qkvg, q_rot, kc, vc, n_q, n_kv, capacity, ring_capacity,
                                       rotary_dim, theta, positions, batch, err, st);
}

}  // namespace

cudaError_t launch_split_rope(int cdtype, const float* qkvg, float* q_rot, void* kc, void* vc,
                              int n_q, int n_kv, int64_t capacity, int ring_capacity,
                              int rotary_dim, double theta, const int32_t* positions, int batch,
                              uint32_t* err, cudaStream_t st) {
  if (cdtype == SPARK_BF16)
    return launch_ct<__nv_bfloat16>(qkvg, q_rot, kc, vc, n_q, n_kv, capacity, ring_capacity,
                                    rotary_dim, theta, positions, batch, err, st);
  return launch_ct<float>(qkvg, q_rot, kc, vc, n_q, n_kv, capacity, ring_capacity, rotary_dim,
                          theta, positions, batch, err, st);
}

}  // namespace spark
