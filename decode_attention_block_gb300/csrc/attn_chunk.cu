// attn_chunk.cu -- attention for a chunk of consecutive tokens of one
// sequence (prefill, or verifying drafted tokens), grouped by query
// (turbospark-runtime 0.3.0, src/kv_write.rs, module doc: chunked prefill
// keeps the per-token attention; src/families/spark/attn.rs,
// encode_attention_block: each token attends over [kv_start, seq_len) of its
// own position, full or sliding window, GQA, scale 256^-0.5).
//
// The result is that of the per-token decode attention, token by token; only
// the schedule differs.  The per-token kernel reads every history row once
// per token: a 512-token chunk at position 700 re-reads ~1000 rows 512 times.
// Here one CTA takes NC consecutive tokens and one KV head: its producer warp
// streams the union of the tokens' windows once, tile by tile (TMA, 16 rows),
// and each consumer warp folds every tile into its own token's state (the
// tensor-core tile of the decode kernel, rows outside the token's window at
// probability 0).  No split over CTAs, so no merge: each warp writes its
// token's four heads at the end.  Rows the chunk itself produces come from
// the staging buffer (they reach the cache only after attention), older rows
// from the cache through the ring, exactly as in the per-token chunk mode.
#include <math.h>

#include "attn_parts.cuh"
#include "launch.h"

namespace spark {
namespace {

// Measured at 256-1024 tokens (p0 700, full + sliding): 4 tokens per CTA,
// two CTAs per SM, a 4-stage ring.  8 tokens per CTA (one CTA per SM, 4 or 8
// stages) was 2-4% slower, a 6-stage ring 15% slower (one CTA per SM).
constexpr int kChunkStages = 4;
constexpr int kChunkGroup = 4;  // consecutive tokens per CTA (one consumer warp each)
constexpr int kChunkMinBlocks = 2;

template <int NC>
struct ChunkSmem {
  static constexpr int kHalf = kv_half_bytes<__nv_bfloat16>();
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kQ = kChunkStages * kStage;     // [NC][4 x kQStride] fp32 queries
  static constexpr int kP = kQ + NC * 4 * kQStride * 4;  // [NC][16 x 4] fp32 probabilities
  static constexpr int kBars = kP + NC * kTile * 4 * 4;
  static constexpr int kFlags = kBars + 2 * kChunkStages * 8;
  static constexpr int kBytes = kFlags + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 (128B swizzle)
};

// The union of the windows of tokens t0 .. t1-1 (positions p0 + t): logical
// positions [lo, hi].  Rows r < c_rows come from the cache (slot first_slot
// + r for r < len_a, then r - len_a after the ring wraps), rows r >= c_rows
// from the staging buffer (row lo + r - p0).
struct Span {
  int64_t lo, rows, c_rows, first_slot, len_a;
};

__device__ __forceinline__ Span span_of(int64_t p0, int t0, int t1, bool full, int window, int ring) {
  const int64_t P0 = p0 + t0, P1 = p0 + t1 - 1;
  Span s;
  s.lo = full ? 0 : (P0 + 1 - window > 0 ? P0 + 1 - window : 0);
  s.rows = P1 - s.lo + 1;
  const int64_t c = p0 - s.lo;
  s.c_rows = c < 0 ? 0 : (c > s.rows ? s.rows : c);
  s.first_slot = ring > 0 ? s.lo % ring : s.lo;
  const int64_t to_end = ring > 0 ? ring - s.first_slot : s.c_rows;
  s.len_a = s.c_rows < to_end ? s.c_rows : to_end;
  return s;
}

// end of the tile that starts at row r: 16 rows, cut where the ring wraps and
// where the cache rows end
__device__ __forceinline__ int64_t tile_end(const Span& sp, int64_t r) {
  int64_t e = r + kTile < sp.rows ? r + kTile : sp.rows;
  if (r < sp.len_a && e > sp.len_a) e = sp.len_a;
  if (r < sp.c_rows && e > sp.c_rows) e = sp.c_rows;
  return e;
}

template <int NC, int MINB>
__global__ void __launch_bounds__((NC + 1) * 32, MINB)
    k_attn_chunk(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                 int64_t p0, int m, const float* __restrict__ q_rot, float* __restrict__ a_out,
                 uint32_t* err, int n_kv, int ring, int full, int window, float scale_log2) {
  using S = ChunkSmem<NC>;
  constexpr int kCT = NC * 32;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = base;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + S::kBars);
  uint64_t* empty_bar = full_bar + kChunkStages;
  volatile int* flags = reinterpret_cast<volatile int*>(base + S::kFlags);  // [0] abort

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the last groups (the latest tokens, the longest windows) first: with
  // more CTAs than fit at once, the short ones then fill the tail
  const int rb = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int j = rb % n_kv, grp = rb / n_kv;
  const int t0 = grp * NC, t1 = t0 + NC < m ? t0 + NC : m;
  const Span sp = span_of(p0, t0, t1, full != 0, window, ring);
  if (tid == 0) {
    for (int s = 0; s < kChunkStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], NC);  // every consumer warp reads every stage
    }
    flags[0] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NC) {
    // ---- producer: the span's tiles in order; cache rows (written by
    // kernels that completed before the previous one started) before the
    // wait on the previous kernel, staged rows after it
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      prefetch_tensormap(&tm_ks);
      prefetch_tensormap(&tm_vs);
      bool waited = false, ok = true;
      uint32_t k = 0;
      for (int64_t r = 0; r < sp.rows; ++k) {
        const int64_t e = tile_end(sp, r);
        const bool staged = r >= sp.c_rows;
        if (staged && !waited) {
          pdl_wait();
          pdl_trigger();
          fence_proxy_async_global();
          waited = true;
        }
        const int s = (int)(k % kChunkStages);
        const uint32_t u = k / kChunkStages;
        if (ok && u > 0 && !mbar_wait_bounded(&empty_bar[s], (u - 1) & 1, flags, kWaitLimitNs)) {
          ok = false;
          flags[0] = 1;
          atomicOr(err, kErrWaitTimeout);
        }
        if (ok) {
          mbar_arrive_expect_tx(&full_bar[s], S::kStage);
          unsigned char* kd = stages + s * S::kStage;
          unsigned char* vd = kd + S::kHalf;
          const int64_t slot = r < sp.len_a ? sp.first_slot + r : r - sp.len_a;
          const int z = staged ? (int)(sp.lo + r - p0) : (int)slot;
          const CUtensorMap* mk = staged ? &tm_ks : &tm_k;
          const CUtensorMap* mv = staged ? &tm_vs : &tm_v;
          tma_load_4d(kd, mk, &full_bar[s], 0, z, 0, j);
          tma_load_4d(vd, mv, &full_bar[s], 0, z, 0, j);
        }
        r = e;
      }
      if (!waited) {
        pdl_wait();
        pdl_trigger();
      }
    }
    __syncwarp();  // the other lanes wait only once lane 0 has issued its tiles
    if (lane != 0) {
      pdl_wait();
      pdl_trigger();
    }
    return;
  }

  // ---- consumers: warp w holds token t0 + w (if any)
  pdl_wait();
  pdl_trigger();
  const int tok = t0 + warp;
  const bool active = tok < t1;
  float* q_s = reinterpret_cast<float*>(base + S::kQ) + warp * 4 * kQStride;
  float* p_w = reinterpret_cast<float*>(base + S::kP) + warp * kTile * 4;
  MmaQ mq;
  MmaState st;
  st.reset();
  if (active) {
    attn_load_q<32>(q_s, q_rot + ((int64_t)tok * (kGroup * n_kv) + kGroup * j) * kHeadDim, lane);
    __syncwarp();
    mma_q_from_smem(mq, q_s);
  }
  // this token's rows of the span: [a0, a1)
  const int64_t P = p0 + tok;
  const int64_t ks = full ? 0 : (P + 1 - window > 0 ? P + 1 - window : 0);
  const int64_t a0 = ks - sp.lo, a1 = P - sp.lo + 1;
  uint32_t k = 0;
  bool ok = true;
  for (int64_t r = 0; r < sp.rows; ++k) {
    const int64_t e = tile_end(sp, r);
    const int n = (int)(e - r);
    const int s = (int)(k % kChunkStages);
    const uint32_t u = k / kChunkStages;
    ok = ok && __all_sync(0xffffffffu, !flags[0] && mbar_wait_bounded(&full_bar[s], u & 1, flags, kWaitLimitNs));
    if (!ok && lane == 0 && !flags[0]) {
      flags[0] = 1;
      atomicOr(err, kErrWaitTimeout);
    }
    unsigned char* kst = stages + s * S::kStage;
    if (n < kTile) {
      // a short tile: its stale tail rows are zeroed once, by warp 0, while
      // no warp reads the stage
      named_bar_sync(kBarConsumers, kCT);
      if (warp == 0 && ok) {
        for (int rr = n; rr < kTile; ++rr)
          *reinterpret_cast<uint4*>(kst + S::kHalf + (lane >> 3) * kSubBytes + rr * kLine + (lane & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills the stage
      }
      named_bar_sync(kBarConsumers, kCT);
    }
    const int64_t lo = a0 - r > 0 ? a0 - r : 0, hi = a1 - r < n ? a1 - r : n;
    if (ok && active && lo < hi)
      attn_tile_mma_rows<false>(kst, kst + S::kHalf, (int)lo, (int)hi, mq, p_w, scale_log2, st);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[s]);
    r = e;
  }
  if (!active || !ok) return;
  // a = o / l for the token's 4 heads: the hi and lo columns added, heads
  // 2 (t & 1) + jj held by the lanes with t < 2 (dims 16 mt + g, + 8)
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < kHeadDim / 16; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) st.o[mt][i] += __shfl_xor_sync(0xffffffffu, st.o[mt][i], 2);
  if (t < 2) {
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
      const int h = 2 * t + jj;
      const float inv = 1.0f / st.l[jj];
      float* dst = a_out + ((int64_t)tok * (kGroup * n_kv) + kGroup * j + h) * kHeadDim;
#pragma unroll
      for (int mt = 0; mt < kHeadDim / 16; ++mt) {
        dst[16 * mt + g] = st.o[mt][jj] * inv;
        dst[16 * mt + g + 8] = st.o[mt][2 + jj] * inv;
      }
    }
  }
}

template <int NC, int MINB>
cudaError_t launch_nc(const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mks,
                      const CUtensorMap& mvs, int64_t p0, int m, const float* q_rot, float* a, uint32_t* err,
                      int n_kv, int ring, bool full, int window, float scale_log2, cudaStream_t st) {
  using S = ChunkSmem<NC>;
  auto kern = k_attn_chunk<NC, MINB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
  if (e != cudaSuccess) return e;
  const int groups = (m + NC - 1) / NC;
  return launch_pdl(kern, dim3(groups * n_kv), dim3((NC + 1) * 32), S::kAlloc, st, mk, mv, mks, mvs, p0, m,
                    q_rot, a, err, n_kv, ring, full ? 1 : 0, window, scale_log2);
}

// the cache's [rows][n_kv][256] bf16 view for TMA, as the decode kernel's
bool chunk_cache_map(CUtensorMap* map, const void* base, int n_kv, int64_t rows) {
  return make_kv_tile_map(map, base, true, n_kv, rows);
}

}  // namespace

bool attention_chunk_grouped_applies(int cdtype, int m, int n_kv) {
  // enough (token group, KV head) CTAs to cover most of the GPU; shorter
  // chunks keep the per-token kernel, which splits long histories over every
  // SM (measured at position 700: 128 tokens 0.194 -> 0.169 ms per chunk
  // grouped, 64 tokens 0.139 -> 0.151 ms, so the switch sits between)
  return cdtype == SPARK_BF16 && ((m + kChunkGroup - 1) / kChunkGroup) * n_kv * 4 >= 3 * device_sm_count() &&
         tensor_map_encoder() != nullptr;
}

cudaError_t launch_attention_chunk_grouped(const float* q_rot, const void* kc, const void* vc, int n_kv,
                                           int64_t capacity, int ring_capacity, bool full, int window,
                                           float scale, int64_t p0, int m, const void* ks, const void* vs,
                                           float* a, uint32_t* err, cudaStream_t st) {
  CUtensorMap mk, mv, mks, mvs;
  if (!chunk_cache_map(&mk, kc, n_kv, capacity) || !chunk_cache_map(&mv, vc, n_kv, capacity) ||
      !chunk_cache_map(&mks, ks, n_kv, m) || !chunk_cache_map(&mvs, vs, n_kv, m))
    return cudaErrorInvalidValue;
  const float scale_log2 = scale * 1.4426950408889634f;
  return launch_nc<kChunkGroup, kChunkMinBlocks>(mk, mv, mks, mvs, p0, m, q_rot, a, err, n_kv, ring_capacity, full, window,
                                   scale_log2, st);
}

}  // namespace spark
