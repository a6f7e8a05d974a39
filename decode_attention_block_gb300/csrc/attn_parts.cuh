// attn_parts.cuh -- the pieces of split-K GQA decode attention shared by the
// per-layer attention kernel (attn.cu) and the persistent decode kernel
// (stack.cu): the shared-memory tile layout, one warp's work on one 16-row
// tile (q.k, online softmax, p.v) and the merge of a group's partial states
// (turbospark-runtime 0.3.0, src/families/spark/attn.rs,
// encode_attention_block -> src/kv_write.rs, encode_attention_any: GQA decode
// attention over [kv_start, seq_len), scale 256^-0.5, no sinks).
#pragma once

#include <math.h>

#include "common.cuh"

namespace spark {

constexpr int kTile = 16;                 // KV rows per pipeline stage
constexpr int kConsumers = 4;             // consumer warps (== kGroup: one head each in the merge)
constexpr int kConsumerThreads = kConsumers * 32;
constexpr int kQStride = 4 * 64 + 4;      // floats per 64-dim q slice (4 heads) + bank shift
constexpr int kLine = 128;                // bytes per swizzled smem line
constexpr int kSubBytes = kTile * kLine;  // one TMA box: kTile rows x 128 bytes
constexpr int kBarConsumers = 1;          // named barrier id of the warps that hold attention states
constexpr int kBarMerge = 3;              // named barrier id of warps 0-3 while they merge a group

template <typename CT>
struct CacheT;
// Pipeline shape of the per-layer kernel.  The ring depth is a multiple of
// the consumer count (tile k lives in stage k % NS and belongs to warp k % 4,
// so each stage always serves one warp and no wait can alias an older
// mbarrier phase).  Long histories run two CTAs per SM with a 4-stage ring
// each (registers capped so both fit): with one consumer warp per SMSP the
// q.k / p.v FMA chains left the issue slots 60% idle, and a second CTA fills
// them (measured 75% -> 90% of HBM peak at 131072 rows; one CTA with eight
// consumer warps did not help, its single producer serialising on the ring).
// Short histories and batch-1 long ones take one CTA per SM, with a 12-stage
// bf16 ring: a short history's share (2-6 tiles) is requested before the
// dependency wait and no stage is refilled (4 stages instead of 8: the
// two-layer batch-1 step 48.8 vs 47.2 us, the 36-layer one 824.7 vs 806.5
// us), and a 16-CTA cluster's 32 tiles of an 8192-row layer keep more in
// flight (8 stages instead of 12: the 36-layer step 740.3 vs 733.5 us, once
// the cluster merge's receive area had shrunk to 5 KB).
template <>
struct CacheT<__nv_bfloat16> {
  static constexpr int kLineElems = 64;
  static constexpr int kDeep = 4;
  static constexpr int kDeepBlocks = 2;  // CTAs per SM
  static constexpr int kShallow = 12;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <>
struct CacheT<float> {
  static constexpr int kLineElems = 32;
  static constexpr int kDeep = 4;
  static constexpr int kDeepBlocks = 1;  // a 4-stage fp32 ring fills half the SM's shared memory
  static constexpr int kShallow = 4;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};

// bytes of one K (or V) half-stage: 16 rows x 256 elements as 128-byte boxes
template <typename CT>
__host__ __device__ constexpr int kv_half_bytes() {
  return (kHeadDim / CacheT<CT>::kLineElems) * kSubBytes;
}

#if defined(__CUDACC__)

// 8 consecutive dims [d0, d0 + 8) of tile row t of a K or V half-stage, as
// four fp32 pairs.  The TMA 128-byte swizzle stores 16-byte chunk q of row t
// at chunk q ^ (t & 7) of the row's line.
template <typename CT>
__device__ __forceinline__ void load8(const unsigned char* half, int t, int d0, float2 (&v)[4]);

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const unsigned char* half, int t, int d0,
                                                     float2 (&v)[4]) {
  const int sub = d0 >> 6, ch = (d0 & 63) >> 3;
  const uint4 w = *reinterpret_cast<const uint4*>(half + sub * kSubBytes + t * kLine +
                                                  ((ch ^ (t & 7)) << 4));
  v[0] = bf16x2_to_f32x2(w.x);
  v[1] = bf16x2_to_f32x2(w.y);
  v[2] = bf16x2_to_f32x2(w.z);
  v[3] = bf16x2_to_f32x2(w.w);
}

template <>
__device__ __forceinline__ void load8<float>(const unsigned char* half, int t, int d0,
                                             float2 (&v)[4]) {
  const int sub = d0 >> 5, ch = (d0 & 31) >> 2;
  const unsigned char* row = half + sub * kSubBytes + t * kLine;
  const float4 a = *reinterpret_cast<const float4*>(row + ((ch ^ (t & 7)) << 4));
  const float4 b = *reinterpret_cast<const float4*>(row + (((ch + 1) ^ (t & 7)) << 4));
  v[0] = make_float2(a.x, a.y);
  v[1] = make_float2(a.z, a.w);
  v[2] = make_float2(b.x, b.y);
  v[3] = make_float2(b.z, b.w);
}

// The token's own cache row of one KV head (K and V, written by the kernel
// before attention) as one warp holds it: lane l the 16-byte chunks
// [kU l, kU l + kU) of each.  A tile that holds this row is loaded before the
// dependency wait, so its copy of the row may be stale; the warp that folds
// the tile reads the row after the wait and writes it over tile row t.
template <typename CT>
struct NewRow {
  static constexpr int kU = sizeof(CT) / 2;  // chunks per lane: 1 (bf16), 2 (fp32)
  uint4 k[kU], v[kU];
  __device__ __forceinline__ void load(const CT* krow, const CT* vrow, int lane) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      k[u] = __ldcg(reinterpret_cast<const uint4*>(krow) + kU * lane + u);
      v[u] = __ldcg(reinterpret_cast<const uint4*>(vrow) + kU * lane + u);
    }
  }
  // chunk c of a row sits in 128-byte box c / 8 at chunk (c % 8) ^ (t % 8)
  // of the row's line (the TMA 128-byte swizzle)
  __device__ __forceinline__ void store(unsigned char* khalf, unsigned char* vhalf, int t, int lane) const {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = kU * lane + u;
      const int off = (c >> 3) * kSubBytes + t * kLine + (((c & 7) ^ (t & 7)) << 4);
      *reinterpret_cast<uint4*>(khalf + off) = k[u];
      *reinterpret_cast<uint4*>(vhalf + off) = v[u];
    }
  }
};

// One warp's running softmax state for the 4 query heads of a KV head: max
// and sum per head (base 2), and the unnormalised output, lane l holding dims
// [8 l, 8 l + 8) of each head.
struct AttnState {
  float m[4], l[4];
  float2 o[4][4];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[h][i] = make_float2(0.f, 0.f);
    }
  }
};

// q of the group's 4 heads into shared memory, in the slice layout attn_tile
// reads (consumer threads only).  Every thread issues all its loads before it
// stores anything, so the copy costs one L2 round trip, not eight.  q comes
// from another CTA or kernel: loads bypass L1.
template <int NT = kConsumerThreads>
__device__ __forceinline__ void attn_load_q(float* q_s, const float* qg, int tid) {
  constexpr int kF4 = kGroup * kHeadDim / 4;  // float4 of q
  constexpr int kPer = (kF4 + NT - 1) / NT;
  float4 v[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k)
    if (tid + k * NT < kF4) v[k] = __ldcg(reinterpret_cast<const float4*>(qg) + tid + k * NT);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    if (tid + k * NT < kF4) {
      const int e = 4 * (tid + k * NT);
      const int h = e >> 8, d = e & 255;
      *reinterpret_cast<float4*>(q_s + (d >> 6) * kQStride + h * 64 + (d & 63)) = v[k];
    }
  }
}

// One warp folds an n-row tile (rows 0..n-1 of the K and V half-stages) into
// its state.  q.k: lanes (sl, ri) cover dims [64 sl, 64 sl + 64) of rows ri
// and ri + 8 with packed fp32x2 FMAs, then sum over the four slices by
// shuffles; p.v: lane l owns dims [8 l, 8 l + 8).  p_w is the warp's 16-row
// probability scratch in shared memory.
template <typename CT>
__device__ __forceinline__ void attn_tile(const unsigned char* kst, const unsigned char* vst, int n,
                                          const float* q_s, float4* p_w, float scale_log2,
                                          AttnState& st) {
  const int lane = threadIdx.x & 31;
  const int sl = lane >> 3, ri = lane & 7;
  float2 acc[2][4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int h = 0; h < 4; ++h) acc[rr][h] = make_float2(0.f, 0.f);
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    const float* qp = q_s + sl * kQStride + cc * 8;
    float4 qa[4], qb[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      qa[h] = *reinterpret_cast<const float4*>(qp + h * 64);
      qb[h] = *reinterpret_cast<const float4*>(qp + h * 64 + 4);
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      float2 kk[4];
      load8<CT>(kst, ri + 8 * rr, sl * 64 + cc * 8, kk);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        acc[rr][h] = ffma2(kk[0], make_float2(qa[h].x, qa[h].y), acc[rr][h]);
        acc[rr][h] = ffma2(kk[1], make_float2(qa[h].z, qa[h].w), acc[rr][h]);
        acc[rr][h] = ffma2(kk[2], make_float2(qb[h].x, qb[h].y), acc[rr][h]);
        acc[rr][h] = ffma2(kk[3], make_float2(qb[h].z, qb[h].w), acc[rr][h]);
      }
    }
  }
  float sc[2][4];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float v = acc[rr][h].x + acc[rr][h].y;
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      sc[rr][h] = (ri + 8 * rr) < n ? v * scale_log2 : -INFINITY;
    }
  // online softmax (base 2)
  float pr[2][4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float mx = fmaxf(sc[0][h], sc[1][h]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    const float mn = fmaxf(st.m[h], mx);
    const float corr = exp2f(st.m[h] - mn);
    st.m[h] = mn;
    st.l[h] *= corr;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st.o[h][i].x *= corr;
      st.o[h][i].y *= corr;
    }
    pr[0][h] = exp2f(sc[0][h] - mn);
    pr[1][h] = exp2f(sc[1][h] - mn);
    if (sl == 0) st.l[h] += pr[0][h] + pr[1][h];
  }
  if (sl < 2) {
    const float4 pw = sl == 0 ? make_float4(pr[0][0], pr[0][1], pr[0][2], pr[0][3])
                              : make_float4(pr[1][0], pr[1][1], pr[1][2], pr[1][3]);
    p_w[ri + 8 * sl] = pw;
  }
  __syncwarp();
  auto pv_row = [&](int t) {
    const float4 pp = p_w[t];
    float2 vv[4];
    load8<CT>(vst, t, 8 * lane, vv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st.o[0][i] = ffma2(vv[i], make_float2(pp.x, pp.x), st.o[0][i]);
      st.o[1][i] = ffma2(vv[i], make_float2(pp.y, pp.y), st.o[1][i]);
      st.o[2][i] = ffma2(vv[i], make_float2(pp.z, pp.z), st.o[2][i]);
      st.o[3][i] = ffma2(vv[i], make_float2(pp.w, pp.w), st.o[3][i]);
    }
  };
  if (n == kTile) {
#pragma unroll 4
    for (int t = 0; t < kTile; ++t) pv_row(t);
  } else {
    for (int t = 0; t < n; ++t) pv_row(t);
  }
}

// The CTA that holds the last row of flat position x, for a grid of G CTAs
// sharing `total` rows equally (CTA c owns [total c / G, total (c+1) / G)).
__device__ __forceinline__ int cta_of(int64_t x, int64_t total, int G) {
  const int64_t cc = ((x + 1) * G - 1) / total;
  return (int)(cc < G - 1 ? cc : G - 1);
}

// Shared memory of the group merge: per warp holding a state, the max and
// the sum of each head and the unnormalised output of each head.
struct MergeSmem {
  float* ms;  // [NW][4]
  float* ls;  // [NW][4]
  float* os;  // [NW][4][256]
};

// Finish one group (sequence b, KV head j) of this CTA's share.  The NW warps
// holding states (NW * 32 threads, all of them call this) put their states in
// shared memory; warps 0-3 then merge them, warp w producing query head 4j + w
// (lane l its dims [8 l, 8 l + 8)).  If the group lies inside this CTA
// (cnt == 1) they write the normalised output, else this CTA's partial into
// slot c + g, take a ticket, and if it is the last of the group's cnt CTAs
// merge all the partials (slots c_first + g ...) into the output in one pass
// with a running max, loading KB partials per round trip.  flags[0] is the
// block's abort flag, flags[1] a scratch word.  a_head0 points at the output
// of the group's first query head.
// Put one warp's state (the CUDA-core tile layout) into the merge scratch.
__device__ __forceinline__ void attn_store_state(const AttnState& st, const MergeSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const float lw = warp_sum(st.l[h]);
    if (lane == 0) {
      sm.ms[warp * 4 + h] = st.m[h];
      sm.ls[warp * 4 + h] = lw;
    }
    float4* dst = reinterpret_cast<float4*>(sm.os + (warp * 4 + h) * kHeadDim + 8 * lane);
    dst[0] = make_float4(st.o[h][0].x, st.o[h][0].y, st.o[h][1].x, st.o[h][1].y);
    dst[1] = make_float4(st.o[h][2].x, st.o[h][2].y, st.o[h][3].x, st.o[h][3].y);
  }
}

template <int NW, int KB = 8>
__device__ __forceinline__ void attn_merge_group(const MergeSmem& sm, volatile int* flags, float* part,
                                                 uint32_t* counters, float* a_head0, int g, int c,
                                                 int c_first, int cnt, uint64_t* trace = nullptr);

template <int NW>
__device__ __forceinline__ void attn_finish_group(const AttnState& st, const MergeSmem& sm,
                                                  volatile int* flags, float* part,
                                                  uint32_t* counters, float* a_head0, int g, int c,
                                                  int c_first, int cnt) {
  attn_store_state(st, sm);
  attn_merge_group<NW>(sm, flags, part, counters, a_head0, g, c, c_first, cnt);
}

// The merge of attn_finish_group, once every warp's state is in `sm`.  KB:
// partials loaded per round trip (16 in the per-layer kernel: 76 partials of
// a 131072-row group in 5 rounds, 0.9 us less per launch; the persistent
// kernel keeps 8, its registers being short).
template <int NW, int KB>
__device__ __forceinline__ void attn_merge_group(const MergeSmem& sm, volatile int* flags, float* part,
                                                 uint32_t* counters, float* a_head0, int g, int c,
                                                 int c_first, int cnt, uint64_t* trace) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  named_bar_sync(kBarConsumers, NW * 32);
  if (warp >= kGroup) return;
  const int h = warp;
  float M = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, sm.ms[ww * 4 + h]);
  float L = 0.f, O[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) O[i] = 0.f;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) {
    const float mw = sm.ms[ww * 4 + h];
    const float scl = mw == -INFINITY ? 0.f : exp2f(mw - M);
    L = fmaf(sm.ls[ww * 4 + h], scl, L);
    const float4* src = reinterpret_cast<const float4*>(sm.os + (ww * 4 + h) * kHeadDim + 8 * lane);
    const float4 x0 = src[0], x1 = src[1];
    O[0] = fmaf(x0.x, scl, O[0]); O[1] = fmaf(x0.y, scl, O[1]);
    O[2] = fmaf(x0.z, scl, O[2]); O[3] = fmaf(x0.w, scl, O[3]);
    O[4] = fmaf(x1.x, scl, O[4]); O[5] = fmaf(x1.y, scl, O[5]);
    O[6] = fmaf(x1.z, scl, O[6]); O[7] = fmaf(x1.w, scl, O[7]);
  }
  float* a_dst = a_head0 + h * kHeadDim + 8 * lane;
  if (cnt == 1) {
    if (!flags[0]) {
      const float inv = 1.0f / L;
      reinterpret_cast<float4*>(a_dst)[0] = make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
      reinterpret_cast<float4*>(a_dst)[1] = make_float4(O[4] * inv, O[5] * inv, O[6] * inv, O[7] * inv);
    }
    return;
  }
  float* P = part + (int64_t)(c + g) * kPartFloats;
  if (!flags[0]) {
    float4* po = reinterpret_cast<float4*>(P + 8 + h * kHeadDim + 8 * lane);
    po[0] = make_float4(O[0], O[1], O[2], O[3]);
    po[1] = make_float4(O[4], O[5], O[6], O[7]);
    if (lane == 0) {
      P[h] = M;
      P[4 + h] = L;
    }
  }
  __threadfence();
  named_bar_sync(kBarMerge, kGroup * 32);
  if (tid == 0) {
    int last = 0;
    if (!flags[0]) last = atomicAdd(&counters[g], 1u) == (uint32_t)(cnt - 1);
    flags[1] = last;
  }
  named_bar_sync(kBarMerge, kGroup * 32);
  if (flags[1]) {
    __threadfence();
    if (threadIdx.x == 0) cta_stamp(trace, 6);
    const float* P0 = part + (int64_t)(c_first + g) * kPartFloats;
    float M2 = -INFINITY, L2 = 0.f, O2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) O2[i] = 0.f;
    constexpr int kBatch = KB;
    for (int q0 = 0; q0 < cnt; q0 += kBatch) {
      float mq[kBatch], lq[kBatch];
      float4 x0[kBatch], x1[kBatch];
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        if (q0 + t < cnt) {
          const float* Pq = P0 + (int64_t)(q0 + t) * kPartFloats;
          mq[t] = __ldcg(Pq + h);
          lq[t] = __ldcg(Pq + 4 + h);
          x0[t] = __ldcg(reinterpret_cast<const float4*>(Pq + 8 + h * kHeadDim + 8 * lane));
          x1[t] = __ldcg(reinterpret_cast<const float4*>(Pq + 8 + h * kHeadDim + 8 * lane + 4));
        } else {
          mq[t] = -INFINITY;
          lq[t] = 0.f;
          x0[t] = x1[t] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mb = M2;
#pragma unroll
      for (int t = 0; t < kBatch; ++t) mb = fmaxf(mb, mq[t]);
      const float rs = M2 == -INFINITY ? 0.f : exp2f(M2 - mb);  // rescale what came before
      L2 *= rs;
#pragma unroll
      for (int i = 0; i < 8; ++i) O2[i] *= rs;
      M2 = mb;
#pragma unroll
      for (int t = 0; t < kBatch; ++t) {
        const float scl = mq[t] == -INFINITY ? 0.f : exp2f(mq[t] - M2);
        L2 = fmaf(lq[t], scl, L2);
        O2[0] = fmaf(x0[t].x, scl, O2[0]); O2[1] = fmaf(x0[t].y, scl, O2[1]);
        O2[2] = fmaf(x0[t].z, scl, O2[2]); O2[3] = fmaf(x0[t].w, scl, O2[3]);
        O2[4] = fmaf(x1[t].x, scl, O2[4]); O2[5] = fmaf(x1[t].y, scl, O2[5]);
        O2[6] = fmaf(x1[t].z, scl, O2[6]); O2[7] = fmaf(x1[t].w, scl, O2[7]);
      }
    }
    const float inv = 1.0f / L2;
    reinterpret_cast<float4*>(a_dst)[0] = make_float4(O2[0] * inv, O2[1] * inv, O2[2] * inv, O2[3] * inv);
    reinterpret_cast<float4*>(a_dst)[1] = make_float4(O2[4] * inv, O2[5] * inv, O2[6] * inv, O2[7] * inv);
    if (tid == 0) counters[g] = 0;  // ready for the next call
    if (tid == 0) cta_stamp(trace, 7);
  }
}


// ---------------------------------------------------------------------------
// The same tile on the tensor cores (bf16 caches): warp-level
// mma.m16n8k16 (bf16 in, fp32 accumulate) for both contractions.
//   s = K q^T:  A = the 16-row K tile (rows x dims, from shared memory by
//               ldmatrix through the TMA swizzle), B = [q_hi | q_lo]^T, the
//               group's 4 query heads split into two bf16 halves (8 columns,
//               q = q_hi + q_lo keeps 16 significant bits), 16 steps of 16 dims;
//   o^T += V^T p^T: A = V^T (ldmatrix.trans of the V tile), B = [p_hi | p_lo]^T,
//               one MMA per 16 dims (16 of them), the accumulator o^T
//               (256 dims x 8 columns) held in registers across tiles.
// Lane (g = lane / 4, t = lane % 4) ends each tile holding the scores of
// rows g and g + 8 for heads 2 (t & 1) and 2 (t & 1) + 1 (the hi and lo
// columns added), and the running max / sum of those two heads.
// ---------------------------------------------------------------------------
struct MmaQ {
  uint32_t b[kHeadDim / 16][2];  // B fragments of [q_hi | q_lo]^T, one pair per 16-dim step
};

struct MmaState {
  float o[kHeadDim / 16][4];  // o^T fragments: dims (16 mt + g, + 8) x columns (2t, 2t + 1)
  float m[2], l[2];           // heads 2 (t & 1) + j, base 2
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int i = 0; i < kHeadDim / 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_elem, hi_elem);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// x, or its bf16 remainder x - bf16(x): the two halves of a hi / lo split
__device__ __forceinline__ float split_part(float x, bool lo) {
  return lo ? x - __bfloat162float(__float2bfloat16_rn(x)) : x;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// shared-memory address of the 16 bytes holding dims [d, d + 8) of tile row
// `row` in a bf16 half-stage (128-byte TMA swizzle, 64-dim boxes)
__device__ __forceinline__ uint32_t tile_chunk(uint32_t half, int row, int d) {
  return half + (uint32_t)((d >> 6) * kSubBytes + row * kLine + ((((d & 63) >> 3) ^ (row & 7)) << 4));
}

// B fragments of the group's queries from q_s (the layout attn_load_q
// writes: 4 heads x 256 fp32 in 64-dim slices): column n = g holds head
// g & 3, its hi half for g < 4 and its lo half after.
__device__ __forceinline__ void mma_q_from_smem(MmaQ& Q, const float* q_s) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const bool lo = g >= 4;
  const float* qh = q_s + (g & 3) * 64 + 2 * t;
#pragma unroll
  for (int ks = 0; ks < kHeadDim / 16; ++ks) {
    const float* p0 = qh + (ks >> 2) * kQStride + 16 * (ks & 3);
    const float2 x0 = *reinterpret_cast<const float2*>(p0);
    const float2 x1 = *reinterpret_cast<const float2*>(p0 + 8);
    Q.b[ks][0] = pack_bf16x2(split_part(x0.x, lo), split_part(x0.y, lo));
    Q.b[ks][1] = pack_bf16x2(split_part(x1.x, lo), split_part(x1.y, lo));
  }
}

// One warp folds rows [row_lo, n) of a tile into its state (bf16 K and V
// half-stages); rows outside take probability 0.  p_w: the warp's 16 x 4 fp32
// probability scratch.  kZeroTail: rows n..15 of the V half-stage are zeroed
// first (their probability is 0, and 0 * a non-finite stale value would not
// be); without it the caller has zeroed them, or they hold finite rows.
template <bool kZeroTail>
__device__ __forceinline__ void attn_tile_mma_rows(unsigned char* kst, unsigned char* vst, int row_lo, int n,
                                                   const MmaQ& Q, float* p_w, float scale_log2,
                                                   MmaState& st) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const uint32_t kbase = smem_u32(kst), vbase = smem_u32(vst);
  const int mi = lane >> 3, lr = lane & 7;
  // s = K [q_hi | q_lo]^T, even and odd 16-dim steps in two accumulator
  // chains (half the dependent MMA latency)
  float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int ks = 0; ks < kHeadDim / 16; ks += 2) {
    uint32_t a[4], a2[4];
    ldsm_x4(tile_chunk(kbase, lr + 8 * (mi & 1), 16 * ks + 8 * (mi >> 1)), a);
    ldsm_x4(tile_chunk(kbase, lr + 8 * (mi & 1), 16 * (ks + 1) + 8 * (mi >> 1)), a2);
    mma_16816(c, a, Q.b[ks][0], Q.b[ks][1]);
    mma_16816(c2, a2, Q.b[ks + 1][0], Q.b[ks + 1][1]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] += c2[i];
  if (kZeroTail && n < kTile) {
    for (int r = n; r < kTile; ++r)
      *reinterpret_cast<uint4*>(vst + (lane >> 3) * kSubBytes + r * kLine + (lane & 7) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills the stage
  }
  // hi + lo columns, scale, mask: sc[r][j] = row (g + 8 r), head 2 (t & 1) + j
  float sc[2][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] += __shfl_xor_sync(0xffffffffu, c[i], 2);
  const bool in0 = g >= row_lo && g < n, in1 = g + 8 >= row_lo && g + 8 < n;
  sc[0][0] = in0 ? c[0] * scale_log2 : -INFINITY;
  sc[0][1] = in0 ? c[1] * scale_log2 : -INFINITY;
  sc[1][0] = in1 ? c[2] * scale_log2 : -INFINITY;
  sc[1][1] = in1 ? c[3] * scale_log2 : -INFINITY;
  // online softmax over the tile's rows (the 8 lanes sharing t)
  float pr[2][2], corr[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(sc[0][j], sc[1][j]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mn = fmaxf(st.m[j], mx);
    corr[j] = exp2f(st.m[j] - mn);
    st.m[j] = mn;
    pr[0][j] = exp2f(sc[0][j] - mn);
    pr[1][j] = exp2f(sc[1][j] - mn);
    float rs = pr[0][j] + pr[1][j];
    rs += __shfl_xor_sync(0xffffffffu, rs, 4);
    rs += __shfl_xor_sync(0xffffffffu, rs, 8);
    rs += __shfl_xor_sync(0xffffffffu, rs, 16);
    st.l[j] = fmaf(st.l[j], corr[j], rs);
  }
  // p to the scratch ([row][head]), then the B fragments of [p_hi | p_lo]^T:
  // column g is head g & 3, rows 2t, 2t + 1, 2t + 8, 2t + 9
  __syncwarp();
  if (t < 2) {
    p_w[g * 4 + 2 * t] = pr[0][0];
    p_w[g * 4 + 2 * t + 1] = pr[0][1];
    p_w[(g + 8) * 4 + 2 * t] = pr[1][0];
    p_w[(g + 8) * 4 + 2 * t + 1] = pr[1][1];
  }
  __syncwarp();
  const int hp = g & 3;
  const bool lo = g >= 4;
  const uint32_t pb0 = pack_bf16x2(split_part(p_w[(2 * t) * 4 + hp], lo), split_part(p_w[(2 * t + 1) * 4 + hp], lo));
  const uint32_t pb1 =
      pack_bf16x2(split_part(p_w[(2 * t + 8) * 4 + hp], lo), split_part(p_w[(2 * t + 9) * 4 + hp], lo));
  // rescale o^T (columns 2t, 2t + 1 are heads 2 (t & 1), + 1 in both halves)
  if (!__all_sync(0xffffffffu, corr[0] == 1.f && corr[1] == 1.f)) {
#pragma unroll
    for (int mt = 0; mt < kHeadDim / 16; ++mt) {
      st.o[mt][0] *= corr[0];
      st.o[mt][1] *= corr[1];
      st.o[mt][2] *= corr[0];
      st.o[mt][3] *= corr[1];
    }
  }
  __syncwarp();  // zeroed V rows visible to every lane's ldmatrix
  // o^T += V^T [p_hi | p_lo]^T
#pragma unroll
  for (int mt = 0; mt < kHeadDim / 16; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(tile_chunk(vbase, lr + 8 * (mi >> 1), 16 * mt + 8 * (mi & 1)), a);
    mma_16816(st.o[mt], a, pb0, pb1);
  }
}

// The decode kernels' tile: rows [0, n), the stale tail zeroed here.
__device__ __forceinline__ void attn_tile_mma(unsigned char* kst, unsigned char* vst, int n,
                                              const MmaQ& Q, float* p_w, float scale_log2,
                                              MmaState& st) {
  attn_tile_mma_rows<true>(kst, vst, 0, n, Q, p_w, scale_log2, st);
}

// Put one warp's tensor-core state into the merge scratch in the layout
// attn_merge_group reads: the hi and lo columns added, heads 2 (t & 1) + j
// written by the lanes with t < 2.
__device__ __forceinline__ void attn_store_state_mma(MmaState& st, const MergeSmem& sm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < kHeadDim / 16; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mt][i] += __shfl_xor_sync(0xffffffffu, st.o[mt][i], 2);
  if (t < 2) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = 2 * t + j;
      float* os = sm.os + (warp * 4 + h) * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < kHeadDim / 16; ++mt) {
        os[16 * mt + g] = st.o[mt][j];
        os[16 * mt + g + 8] = st.o[mt][2 + j];
      }
      if (g == 0) {
        sm.ms[warp * 4 + h] = st.m[j];
        sm.ls[warp * 4 + h] = st.l[j];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// cluster mode: the CTAs of one cluster share one group and merge through DSMEM
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  return ra;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t ra) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_cluster_f4(uint32_t ra) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

// the cluster barrier split in two: arrive (release) early, wait (acquire)
// where the other CTAs' earlier writes are needed
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Remote stores into the shared memory of a CTA of the cluster (addr, bar:
// shared::cluster addresses) whose bytes complete that CTA's mbarrier
// transaction count; the data leaves from registers.
__device__ __forceinline__ void st_async_f32(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(addr), "f"(v),
               "r"(bar)
               : "memory");
}
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   addr),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
               : "memory");
}

// The CTA's state of its group from the NW warps' states in `sm`: warp h < 4
// merges head h into cst ([4] m, [4] l, [4][256] unnormalised o).
template <int NW>
__device__ __forceinline__ void attn_cta_state(const MergeSmem& sm, float* cst) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  named_bar_sync(kBarConsumers, NW * 32);
  if (warp >= kGroup) return;
  const int h = warp;
  float M = -INFINITY;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) M = fmaxf(M, sm.ms[ww * 4 + h]);
  float L = 0.f, O[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) O[i] = 0.f;
#pragma unroll
  for (int ww = 0; ww < NW; ++ww) {
    const float mw = sm.ms[ww * 4 + h];
    const float scl = mw == -INFINITY ? 0.f : exp2f(mw - M);
    L = fmaf(sm.ls[ww * 4 + h], scl, L);
    const float4* src = reinterpret_cast<const float4*>(sm.os + (ww * 4 + h) * kHeadDim + 8 * lane);
    const float4 x0 = src[0], x1 = src[1];
    O[0] = fmaf(x0.x, scl, O[0]); O[1] = fmaf(x0.y, scl, O[1]);
    O[2] = fmaf(x0.z, scl, O[2]); O[3] = fmaf(x0.w, scl, O[3]);
    O[4] = fmaf(x1.x, scl, O[4]); O[5] = fmaf(x1.y, scl, O[5]);
    O[6] = fmaf(x1.z, scl, O[6]); O[7] = fmaf(x1.w, scl, O[7]);
  }
  if (lane == 0) {
    cst[h] = M;
    cst[4 + h] = L;
  }
  float4* dst = reinterpret_cast<float4*>(cst + 8 + h * kHeadDim + 8 * lane);
  dst[0] = make_float4(O[0], O[1], O[2], O[3]);
  dst[1] = make_float4(O[4], O[5], O[6], O[7]);
}

#endif  // __CUDACC__

}  // namespace spark
