// attn.cu -- split-K GQA decode attention with a log-sum-exp merge
// (turbospark-runtime 0.3.0, src/families/spark/attn.rs,
// encode_attention_block -> src/kv_write.rs, encode_attention_any ->
// gpu::encode_attention_decode: attention over [kv_start, seq_len) with ring
// addressing when the ring is active, scale 256^-0.5, no sinks).
//
// Work decomposition.  The rows every sequence reads (its window, through the
// ring) form one flat list ordered by (sequence, KV head, row); the grid's
// CTAs each take an equal contiguous share of it, so a ragged batch and a
// single 131072-row sequence balance the same way.  A CTA's share meets one
// or more (sequence, KV head) groups; for each it keeps an online softmax for
// the group's 4 query heads (each KV row is read once and serves all 4) and
// emits either the finished output (the group lies inside its share) or a
// partial (m, l, o) into a slot of the workspace.  The last CTA to finish a
// group -- found with an atomic ticket, nobody waits -- merges the partials.
// Softmax is order-free, so a window that wraps the ring is read as two
// contiguous runs of cache rows.
//
// Inside a CTA.  One producer warp streams 16-row K and V tiles of one KV
// head (4 x 128-byte swizzled TMA boxes each for bf16) into an 8-stage
// shared-memory ring; four consumer warps each own every fourth tile.  A
// consumer computes q.k for its 16 rows x 4 heads with lanes split over four
// 64-dim slices and packed fp32x2 FMAs, reduces over the slices with
// shuffles, updates its own running max / sum, and accumulates p.v with each
// lane owning 8 of the 256 output dims.  At the end of a group the four warps'
// states are merged through shared memory.
#include <math.h>

#include "launch.h"

namespace spark {
namespace {

constexpr int kTile = 16;                     // KV rows per pipeline stage
constexpr int kConsumers = 4;                 // consumer warps (== kGroup: one head each in the merge)
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kConsumerThreads = kConsumers * 32;
constexpr int kQStride = 4 * 64 + 4;          // floats per 64-dim q slice (4 heads) + bank shift
constexpr int kLine = 128;                    // bytes per swizzled smem line
constexpr int kSubBytes = kTile * kLine;      // one TMA box: kTile rows x 128 bytes
constexpr int kMinRowsPerCta = 64;            // default grid: at least this many rows per CTA
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kBarConsumers = 1;              // named barrier id of the consumer warps

template <typename CT>
struct CacheT;
// Pipeline depth (a multiple of the consumer count: tile k lives in stage
// k % NS and belongs to warp k % 4, so each stage always serves one warp and
// no wait can alias an older mbarrier phase).  Long histories take a deep
// ring (the kernel runs alone for hundreds of microseconds); short ones a
// shallow ring, so the kernel's CTAs leave room on each SM for the next
// kernel's CTAs to start streaming o_proj's weights while attention runs.
template <>
struct CacheT<__nv_bfloat16> {
  static constexpr int kLineElems = 64;
  static constexpr int kDeep = 8;
  static constexpr int kShallow = 4;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <>
struct CacheT<float> {
  static constexpr int kLineElems = 32;
  static constexpr int kDeep = 4;
  static constexpr int kShallow = 4;
  static constexpr CUtensorMapDataType kTma = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
};
constexpr int64_t kDeepRows = 1 << 16;  // rows (x KV heads) per call from which the deep ring pays

template <typename CT, int NS>
struct Smem {
  static_assert(NS % kConsumers == 0, "each stage must belong to one consumer warp");
  static constexpr int kStages = NS;
  static constexpr int kSubs = kHeadDim / CacheT<CT>::kLineElems;
  static constexpr int kHalf = kSubs * kSubBytes;  // the K (or V) half of a stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kQ = kStages * kStage;
  static constexpr int kP = kQ + 4 * kQStride * 4;
  static constexpr int kM = kP + kConsumers * kTile * 16;
  static constexpr int kL = kM + kConsumers * 4 * 4;
  static constexpr int kO = kL + kConsumers * 4 * 4;
  static constexpr int kBars = kO + kConsumers * 4 * kHeadDim * 4;
  static constexpr int kFlags = kBars + 2 * kStages * 8;
  static constexpr int kBytes = kFlags + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 (128B swizzle)
};

template <int MAXB>
struct AttnArgs {
  int64_t prefix[MAXB + 1];  // rows read by sequences before b
  int32_t pos[MAXB];
};

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

// Enumerates, identically for the producer and the consumers, the groups a
// CTA's share meets and the tiles of each.
struct Share {
  int64_t f, f1;   // current flat position, end of share
  int b, j;        // current sequence, KV head
};

template <int MAXB>
__device__ __forceinline__ Share share_begin(const AttnArgs<MAXB>& args, int batch, int n_kv,
                                             int64_t f0, int64_t f1) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)n_kv * args.prefix[mid] <= f0) lo = mid; else hi = mid - 1;
  }
  Share s;
  s.f = f0;
  s.f1 = f1;
  s.b = lo;
  const int64_t rows = args.prefix[lo + 1] - args.prefix[lo];
  s.j = (int)((f0 - (int64_t)n_kv * args.prefix[lo]) / rows);
  return s;
}

template <typename CT, int NS, int MAXB>
__global__ void __launch_bounds__(kThreads, 1)
    k_attn_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const float* __restrict__ q_rot, float* __restrict__ a_out,
                  float* __restrict__ part, uint32_t* __restrict__ counters, uint32_t* err,
                  int batch, int n_kv, int64_t capacity, int ring_capacity, int full,
                  int window, float scale_log2, const unsigned char* l2_pf, int64_t l2_pf_bytes,
                  const __grid_constant__ AttnArgs<MAXB> args) {
  using S = Smem<CT, NS>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  float* q_s = reinterpret_cast<float*>(base + S::kQ);
  float4* p_s = reinterpret_cast<float4*>(base + S::kP);
  float* ms = reinterpret_cast<float*>(base + S::kM);
  float* ls = reinterpret_cast<float*>(base + S::kL);
  float* os = reinterpret_cast<float*>(base + S::kO);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + S::kBars);
  uint64_t* empty_bar = full_bar + NS;
  volatile int* flags = reinterpret_cast<volatile int*>(base + S::kFlags);  // [0] abort, [1] last

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    // A hint for the kernel after this one: its weights (o_proj) do not
    // depend on attention, so this CTA pulls its share of them into L2 while
    // HBM is otherwise idle.
    if (l2_pf != nullptr && l2_pf_bytes > 0) {
      const int64_t lo = (l2_pf_bytes * blockIdx.x / gridDim.x) & ~int64_t(15);
      const int64_t hi = (l2_pf_bytes * (blockIdx.x + 1) / gridDim.x) & ~int64_t(15);
      for (int64_t o = lo; o < hi; o += 65536) {
        const int64_t n = hi - o < 65536 ? hi - o : 65536;
        bulk_prefetch_l2(l2_pf + o, (uint32_t)n);
      }
    }
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // q_rot and the new cache rows come from the previous kernel

  const int64_t total = (int64_t)n_kv * args.prefix[batch];
  const int G = gridDim.x, c = blockIdx.x;
  const int64_t f0 = total * c / G, f1 = total * (c + 1) / G;
  if (f0 >= f1) return;
  const int32_t* pos = args.pos;

  // ------------------------------------------------------------ producer
  if (warp == kConsumers) {
    if (lane != 0) return;
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    uint32_t k = 0;
    bool ok = true;
    Share sh = share_begin(args, batch, n_kv, f0, f1);
    while (sh.f < sh.f1) {
      const int64_t rows = args.prefix[sh.b + 1] - args.prefix[sh.b];
      const int64_t gs = (int64_t)n_kv * args.prefix[sh.b] + sh.j * rows;
      const int64_t r0 = sh.f - gs, r1 = min(sh.f1, gs + rows) - gs;
      const Window w = window_of(pos[sh.b], full != 0, window, ring_capacity);
      for (int64_t r = r0; r < r1;) {
        int64_t e = min(r1, r + kTile);
        if (r < w.len_a && e > w.len_a) e = w.len_a;
        const int64_t slot = r < w.len_a ? w.first_slot + r : r - w.len_a;
        const int s = (int)(k % NS);
        const uint32_t u = k / NS;
        if (ok && u > 0 && !mbar_wait_bounded(&empty_bar[s], (u - 1) & 1, flags, kWaitLimitNs)) {
          ok = false;
          flags[0] = 1;
          atomicOr(err, kErrWaitTimeout);
        }
        if (ok) {
          mbar_arrive_expect_tx(&full_bar[s], S::kStage);
          unsigned char* kd = stages + s * S::kStage;
          unsigned char* vd = kd + S::kHalf;
          const int z = (int)((int64_t)sh.b * capacity + slot);
#pragma unroll
          for (int q = 0; q < S::kSubs; ++q) {
            tma_load_3d(kd + q * kSubBytes, &tm_k, &full_bar[s], q * CacheT<CT>::kLineElems, sh.j, z);
            tma_load_3d(vd + q * kSubBytes, &tm_v, &full_bar[s], q * CacheT<CT>::kLineElems, sh.j, z);
          }
        }
        ++k;
        r = e;
      }
      sh.f = gs + r1;
      if (++sh.j == n_kv) { sh.j = 0; ++sh.b; }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int sl = lane >> 3, ri = lane & 7;
  const int cta_last = G - 1;
  auto cta_of = [&](int64_t x) -> int {
    const int64_t cc = ((x + 1) * G - 1) / total;
    return (int)(cc < cta_last ? cc : cta_last);
  };
  uint32_t k = 0;
  Share sh = share_begin(args, batch, n_kv, f0, f1);
  while (sh.f < sh.f1) {
    const int b = sh.b, j = sh.j;
    const int64_t rows = args.prefix[b + 1] - args.prefix[b];
    const int64_t gs = (int64_t)n_kv * args.prefix[b] + j * rows;
    const int64_t r0 = sh.f - gs, r1 = min(sh.f1, gs + rows) - gs;
    const Window w = window_of(pos[b], full != 0, window, ring_capacity);

    named_bar_sync(kBarConsumers, kConsumerThreads);  // the previous group's merge is done
    {
      const float* qg = q_rot + ((int64_t)b * (kGroup * n_kv) + kGroup * j) * kHeadDim;
      for (int e = tid; e < kGroup * kHeadDim; e += kConsumerThreads) {
        const int h = e >> 8, d = e & 255;
        q_s[(d >> 6) * kQStride + h * 64 + (d & 63)] = qg[e];
      }
    }
    named_bar_sync(kBarConsumers, kConsumerThreads);

    float m[4], l[4];
    float2 o[4][4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[h][i] = make_float2(0.f, 0.f);
    }

    for (int64_t r = r0; r < r1;) {
      int64_t e = min(r1, r + kTile);
      if (r < w.len_a && e > w.len_a) e = w.len_a;
      const int n = (int)(e - r);
      if ((int)(k % kConsumers) == warp) {
        const int s = (int)(k % NS);
        const uint32_t u = k / NS;
        const bool ok = !flags[0] && mbar_wait_bounded(&full_bar[s], u & 1, flags, kWaitLimitNs);
        if (!ok) {
          if (lane == 0 && !flags[0]) {
            flags[0] = 1;
            atomicOr(err, kErrWaitTimeout);
          }
        } else {
          const unsigned char* kst = stages + s * S::kStage;
          const unsigned char* vst = kst + S::kHalf;
          // ---- scores: lanes (sl, ri) cover dims [64 sl, 64 sl + 64) of rows ri, ri + 8
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
          // ---- online softmax (base 2), per warp
          float pr[2][4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            float mx = fmaxf(sc[0][h], sc[1][h]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            const float mn = fmaxf(m[h], mx);
            const float corr = exp2f(m[h] - mn);
            m[h] = mn;
            l[h] *= corr;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[h][i].x *= corr;
              o[h][i].y *= corr;
            }
            pr[0][h] = exp2f(sc[0][h] - mn);
            pr[1][h] = exp2f(sc[1][h] - mn);
            if (sl == 0) l[h] += pr[0][h] + pr[1][h];
          }
          if (sl < 2) {
            const float4 pw = sl == 0 ? make_float4(pr[0][0], pr[0][1], pr[0][2], pr[0][3])
                                      : make_float4(pr[1][0], pr[1][1], pr[1][2], pr[1][3]);
            p_s[warp * kTile + ri + 8 * sl] = pw;
          }
          __syncwarp();
          // ---- p.v: lane owns dims [8 lane, 8 lane + 8)
          auto pv_row = [&](int t) {
            const float4 pp = p_s[warp * kTile + t];
            float2 vv[4];
            load8<CT>(vst, t, 8 * lane, vv);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[0][i] = ffma2(vv[i], make_float2(pp.x, pp.x), o[0][i]);
              o[1][i] = ffma2(vv[i], make_float2(pp.y, pp.y), o[1][i]);
              o[2][i] = ffma2(vv[i], make_float2(pp.z, pp.z), o[2][i]);
              o[3][i] = ffma2(vv[i], make_float2(pp.w, pp.w), o[3][i]);
            }
          };
          if (n == kTile) {
#pragma unroll 4
            for (int t = 0; t < kTile; ++t) pv_row(t);
          } else {
            for (int t = 0; t < n; ++t) pv_row(t);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      ++k;
      r = e;
    }

    // ---- merge the four warps' states of this group
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float lw = warp_sum(l[h]);
      if (lane == 0) {
        ms[warp * 4 + h] = m[h];
        ls[warp * 4 + h] = lw;
      }
      float4* dst = reinterpret_cast<float4*>(os + (warp * 4 + h) * kHeadDim + 8 * lane);
      dst[0] = make_float4(o[h][0].x, o[h][0].y, o[h][1].x, o[h][1].y);
      dst[1] = make_float4(o[h][2].x, o[h][2].y, o[h][3].x, o[h][3].y);
    }
    named_bar_sync(kBarConsumers, kConsumerThreads);
    const int h = warp;  // in the merge, warp w finishes query head 4j + w, lane its 8 dims
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) M = fmaxf(M, ms[ww * 4 + h]);
    float L = 0.f, O[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) O[i] = 0.f;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) {
      const float mw = ms[ww * 4 + h];
      const float scl = mw == -INFINITY ? 0.f : exp2f(mw - M);
      L = fmaf(ls[ww * 4 + h], scl, L);
      const float4* src = reinterpret_cast<const float4*>(os + (ww * 4 + h) * kHeadDim + 8 * lane);
      const float4 x0 = src[0], x1 = src[1];
      O[0] = fmaf(x0.x, scl, O[0]); O[1] = fmaf(x0.y, scl, O[1]);
      O[2] = fmaf(x0.z, scl, O[2]); O[3] = fmaf(x0.w, scl, O[3]);
      O[4] = fmaf(x1.x, scl, O[4]); O[5] = fmaf(x1.y, scl, O[5]);
      O[6] = fmaf(x1.z, scl, O[6]); O[7] = fmaf(x1.w, scl, O[7]);
    }
    const int g = b * n_kv + j;
    const int c_first = cta_of(gs), c_last = cta_of(gs + rows - 1);
    const int cnt = c_last - c_first + 1;
    float* a_dst = a_out + ((int64_t)b * (kGroup * n_kv) + kGroup * j + h) * kHeadDim + 8 * lane;
    if (cnt == 1) {
      if (!flags[0]) {
        const float inv = 1.0f / L;
        reinterpret_cast<float4*>(a_dst)[0] = make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
        reinterpret_cast<float4*>(a_dst)[1] = make_float4(O[4] * inv, O[5] * inv, O[6] * inv, O[7] * inv);
      }
    } else {
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
      named_bar_sync(kBarConsumers, kConsumerThreads);
      if (tid == 0) {
        int last = 0;
        if (!flags[0]) last = atomicAdd(&counters[g], 1u) == (uint32_t)(cnt - 1);
        flags[1] = last;
      }
      named_bar_sync(kBarConsumers, kConsumerThreads);
      if (flags[1]) {
        __threadfence();
        const float* P0 = part + (int64_t)(c_first + g) * kPartFloats;
        float M2 = -INFINITY;
        for (int q = 0; q < cnt; ++q) M2 = fmaxf(M2, __ldcg(P0 + (int64_t)q * kPartFloats + h));
        float L2 = 0.f, O2[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) O2[i] = 0.f;
        for (int q = 0; q < cnt; ++q) {
          const float* Pq = P0 + (int64_t)q * kPartFloats;
          const float scl = exp2f(__ldcg(Pq + h) - M2);
          L2 = fmaf(__ldcg(Pq + 4 + h), scl, L2);
          const float4 x0 = __ldcg(reinterpret_cast<const float4*>(Pq + 8 + h * kHeadDim + 8 * lane));
          const float4 x1 = __ldcg(reinterpret_cast<const float4*>(Pq + 8 + h * kHeadDim + 8 * lane + 4));
          O2[0] = fmaf(x0.x, scl, O2[0]); O2[1] = fmaf(x0.y, scl, O2[1]);
          O2[2] = fmaf(x0.z, scl, O2[2]); O2[3] = fmaf(x0.w, scl, O2[3]);
          O2[4] = fmaf(x1.x, scl, O2[4]); O2[5] = fmaf(x1.y, scl, O2[5]);
          O2[6] = fmaf(x1.z, scl, O2[6]); O2[7] = fmaf(x1.w, scl, O2[7]);
        }
        const float inv = 1.0f / L2;
        reinterpret_cast<float4*>(a_dst)[0] = make_float4(O2[0] * inv, O2[1] * inv, O2[2] * inv, O2[3] * inv);
        reinterpret_cast<float4*>(a_dst)[1] = make_float4(O2[4] * inv, O2[5] * inv, O2[6] * inv, O2[7] * inv);
        if (tid == 0) counters[g] = 0;  // ready for the next call
      }
    }
    sh.f = gs + r1;
    if (++sh.j == n_kv) { sh.j = 0; ++sh.b; }
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [rows = batch * capacity][n_kv][256] cache viewed as a 3-D tensor; boxes of
// kTile rows x one KV head x 128 bytes, 128-byte swizzle.
template <typename CT>
bool make_cache_map(CUtensorMap* map, const void* base, int n_kv, int64_t rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t es = sizeof(CT);
  const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_kv, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {kHeadDim * es, (cuuint64_t)n_kv * kHeadDim * es};
  const cuuint32_t box[3] = {(cuuint32_t)CacheT<CT>::kLineElems, 1, (cuuint32_t)kTile};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CacheT<CT>::kTma, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename CT, int NS, int MAXB>
cudaError_t launch_t(const float* q_rot, const void* kc, const void* vc, int n_kv,
                     int64_t capacity, int ring_capacity, bool full, int window, float scale,
                     const int32_t* positions, int batch, float* a, float* part,
                     uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                     size_t l2_pf_bytes, cudaStream_t st) {
  using S = Smem<CT, NS>;
  AttnArgs<MAXB> args;
  args.prefix[0] = 0;
  for (int b = 0; b < MAXB; ++b) {
    const int64_t rows = b < batch ? window_of(positions[b], full, window, ring_capacity).rows : 0;
    args.prefix[b + 1] = args.prefix[b] + rows;
    args.pos[b] = b < batch ? positions[b] : 0;
  }
  const int64_t total = (int64_t)n_kv * args.prefix[batch];
  int G = n_ctas;
  if (G <= 0) {
    const int64_t want = (total + kMinRowsPerCta - 1) / kMinRowsPerCta;
    G = (int)(want < device_sm_count() ? want : device_sm_count());
  }
  if (G < 1) G = 1;
  if (G > kMaxAttnCtas) G = kMaxAttnCtas;

  CUtensorMap mk, mv;
  if (!make_cache_map<CT>(&mk, kc, n_kv, (int64_t)batch * capacity) ||
      !make_cache_map<CT>(&mv, vc, n_kv, (int64_t)batch * capacity))
    return cudaErrorInvalidValue;
  auto kern = k_attn_decode<CT, NS, MAXB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
  if (e != cudaSuccess) return e;
  const float scale_log2 = scale * 1.4426950408889634f;
  return launch_pdl(kern, dim3(G), dim3(kThreads), S::kAlloc, st, mk, mv, q_rot, a, part, counters,
                    err, batch, n_kv, capacity, ring_capacity, full ? 1 : 0, window, scale_log2,
                    static_cast<const unsigned char*>(l2_pf), (int64_t)l2_pf_bytes, args);
}

template <typename CT, int NS>
cudaError_t launch_ns(const float* q_rot, const void* kc, const void* vc, int n_kv,
                      int64_t capacity, int ring_capacity, bool full, int window, float scale,
                      const int32_t* positions, int batch, float* a, float* part,
                      uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                      size_t l2_pf_bytes, cudaStream_t st) {
  if (batch <= 8)
    return launch_t<CT, NS, 8>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                               positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, st);
  if (batch <= 64)
    return launch_t<CT, NS, 64>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                                positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, st);
  return launch_t<CT, NS, SPARK_MAX_BATCH>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full,
                                           window, scale, positions, batch, a, part, counters, err,
                                           n_ctas, l2_pf, l2_pf_bytes, st);
}

template <typename CT>
cudaError_t launch_ct(const float* q_rot, const void* kc, const void* vc, int n_kv,
                      int64_t capacity, int ring_capacity, bool full, int window, float scale,
                      const int32_t* positions, int batch, float* a, float* part,
                      uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                      size_t l2_pf_bytes, cudaStream_t st) {
  int64_t rows = 0;
  for (int b = 0; b < batch; ++b) rows += window_of(positions[b], full, window, ring_capacity).rows;
  if ((int64_t)n_kv * rows >= kDeepRows)
    return launch_ns<CT, CacheT<CT>::kDeep>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window,
                                      scale, positions, batch, a, part, counters, err, n_ctas,
                                      l2_pf, l2_pf_bytes, st);
  return launch_ns<CT, CacheT<CT>::kShallow>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window,
                                       scale, positions, batch, a, part, counters, err, n_ctas,
                                       l2_pf, l2_pf_bytes, st);
}

}  // namespace

cudaError_t launch_attention(int cdtype, const float* q_rot, const void* kc, const void* vc,
                             int n_kv, int64_t capacity, int ring_capacity, bool full,
                             int window, float scale, const int32_t* positions, int batch,
                             float* a, float* part, uint32_t* counters, uint32_t* err,
                             int n_ctas, const void* l2_pf, size_t l2_pf_bytes, cudaStream_t st) {
  if (cdtype == SPARK_BF16)
    return launch_ct<__nv_bfloat16>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window,
                                    scale, positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, st);
  return launch_ct<float>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                          positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, st);
}

}  // namespace spark
