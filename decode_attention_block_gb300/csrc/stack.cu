// stack.cu -- one persistent kernel for a whole decode step over a stack of
// attention blocks (turbospark-runtime 0.3.0, src/families/spark/mod.rs,
// produce_real_spark_inner: the layer loop; each layer is
// src/families/spark/attn.rs, encode_attention_block, preceded by the input
// RMSNorm and followed by the raw residual add).
//
// Why one kernel.  At batch 1 a layer moves ~52 MB of weights; separate
// kernels each pay a launch, a pipeline ramp-up and a tail (measured ~4 us per
// kernel on GB300 at these sizes), more than half of the step.  Here one CTA
// per SM lives for the whole step.  Its producer warp streams, in order and
// as far ahead as the shared-memory ring allows, every byte the CTA will read:
// its share of layer l's q_k_v_proj rows, then (once layer l's new k and v are
// in the cache) its share of layer l's KV tiles, then its share of o_proj's
// rows, then layer l+1's q_k_v_proj rows...  The weights never wait for the
// computation; HBM keeps streaming across phase and layer boundaries.  Four
// compute warps consume the ring and meet the other CTAs at three grid
// barriers per layer: after the projections (q, k, v, g complete), after
// attention (every group merged) and after o_proj (h of the next layer
// complete).  The kernel is launched cooperatively, so all its CTAs are
// resident and the barriers cannot deadlock; every wait is bounded.
//
// The phases reuse the per-layer kernels' device code (gemv_parts.cuh,
// attn_parts.cuh):
//  P1  RMSNorm + q_k_v_proj + g_proj + rope + cache write, four rows per ring
//      stage (two rope pairs);
//  P2  split-K attention over the layer's rows, stream-K shares, last-CTA
//      merge through tickets;
//  P3  gate + o_proj + residual, two rows per ring stage.
#include <stdlib.h>

#include "attn_parts.cuh"
#include "checks.h"
#include "gemv_parts.cuh"
#include "launch.h"

namespace spark {
namespace {

constexpr int kComputeWarps = 7;                     // warps 0-6 compute (0-3 also attend), warp 7 produces
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kProducerWarp = kComputeWarps;
constexpr int kThreads = (kComputeWarps + 1) * 32;
constexpr int kBarCompute = 2;                       // named barrier id of all compute warps
constexpr int kMaxLayers = 40;                       // layers per launch (more: several launches)
constexpr int kMaxNB = 4;                            // sequences per launch
constexpr int kMinRowsPerCta = 64;
constexpr int kL2PrefetchTiles = 8;                  // KV tiles per CTA pulled into L2 ahead of P2
constexpr size_t kSmemMax = 227 * 1024;
constexpr int kMaxPer = (4096 / 4 + kComputeThreads - 1) / kComputeThreads;  // float4 of an activation vector per thread

struct LayerDesc {
  const __nv_bfloat16* norm_w;
  const __nv_bfloat16* qkv_w;
  const __nv_bfloat16* g_w;
  const __nv_bfloat16* o_w;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int64_t capacity;
  int32_t ring;
  int32_t full;
};

template <int NB>
struct StackArgs {
  CUtensorMap tm[kMaxLayers][2];     // K and V cache of each layer
  LayerDesc layer[kMaxLayers];
  float2 cs[2][NB][kHeadDim / 2];    // [full][b]: (cos, sin) of the rope angle of pair i
  int64_t prefix[2][NB + 1];         // [full]: attention rows of the sequences before b
  int32_t rotary[2];                 // [full]: rotary dim
  int32_t pos[NB];
};

struct Geo {
  int hidden, n_q, n_kv, window, nb, n_layers, stages, stage_bytes, xfloats;
  float scale_log2, eps;
};

struct Ws {
  const float* h_in;
  float* out;
  float* hbuf;     // [2][nb][hidden]
  float* q_rot;
  float* g;
  float* a;
  float* part;
  uint32_t* counters;
  uint32_t* gbar;  // [0] arrivals, [1] released epoch
  uint32_t* err;
  uint64_t* trace; // phase timestamps (CTA 0), or null
};

// trace slots per layer: compute 0..7, producer 8..11
enum TraceEv { kTrP1Start = 0, kTrP1End, kTrB1, kTrP2End, kTrB2, kTrP3Start, kTrP3End, kTrB3,
               kTrProdP1Issued = 8, kTrProdP2Start, kTrProdP3Start, kTrP2Q, kTrP2Tiles, kTrP2Merged };
constexpr int kTraceSlots = 16;

__device__ __forceinline__ void trace(const Ws& ws, int l, int ev) {
  if (ws.trace != nullptr && blockIdx.x == 0 && l * kTraceSlots + ev < kTraceWords / 2)
    ws.trace[l * kTraceSlots + ev] = global_timer_ns();
}
// per-CTA phase ends of the first layers: second half of the trace buffer
__device__ __forceinline__ void trace_cta(const Ws& ws, int l, int ev) {
  const int idx = kTraceWords / 2 + (l * 4 + ev) * 160 + (int)blockIdx.x;
  if (ws.trace != nullptr && blockIdx.x < 160 && idx < kTraceWords) ws.trace[idx] = global_timer_ns();
}

// ---------------------------------------------------------------------------
// the ring: stage i % NS holds item i; use[s] is the last use the producer
// has issued into stage s, so a consumer never waits on a barrier phase two
// uses ahead (mbarrier parity tells only the last two apart)
// ---------------------------------------------------------------------------
struct Ring {
  unsigned char* base;
  uint64_t* full;
  uint64_t* empty;
  volatile int* use;
  int ns, stage_bytes;
  __device__ __forceinline__ unsigned char* stage(uint32_t i) const {
    return base + (size_t)(i % ns) * stage_bytes;
  }
};

__device__ __forceinline__ bool spin_until(volatile int* word, int want, volatile int* abort) {
  if (*word >= want) return true;
  const uint64_t t0 = global_timer_ns();
  while (*word < want) {
    __nanosleep(32);  // leave the issue slots to the warps doing work
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// producer: claim stage of item i (wait until its previous use is consumed)
__device__ __forceinline__ bool ring_acquire(const Ring& r, uint32_t i, volatile int* abort) {
  const uint32_t u = i / r.ns;
  if (u == 0) return true;
  return mbar_wait_bounded(&r.empty[i % r.ns], (u - 1) & 1, abort, kWaitLimitNs);
}
// producer: the copies of item i are issued
__device__ __forceinline__ void ring_publish(const Ring& r, uint32_t i) {
  __threadfence_block();
  r.use[i % r.ns] = (int)(i / r.ns);
}
// consumer warp: wait for the data of item i
__device__ __forceinline__ bool ring_wait(const Ring& r, uint32_t i, volatile int* abort) {
  const int s = (int)(i % r.ns), u = (int)(i / r.ns);
  if (!spin_until(r.use + s, u, abort)) return false;
  __threadfence_block();
  return mbar_wait_bounded(&r.full[s], (uint32_t)u & 1, abort, kWaitLimitNs);
}
// consumer warp (lane 0): item i's stage may be refilled
__device__ __forceinline__ void ring_release(const Ring& r, uint32_t i) { mbar_arrive(&r.empty[i % r.ns]); }

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All CTAs' compute warps meet; epoch counts the barriers this CTA passed.
// Arrival is one fire-and-forget release add; the wait polls the counter
// until every CTA of this epoch has arrived (the counter only grows within a
// launch; the host zeroes it before each launch).
__device__ __forceinline__ void grid_barrier(uint32_t* gbar, uint32_t& epoch, volatile int* flags,
                                             uint32_t* err) {
  named_bar_sync(kBarCompute, kComputeThreads);
  ++epoch;
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(gbar) : "memory");
    const uint32_t target = epoch * gridDim.x;
    if (ld_acquire_gpu(gbar) < target) {
      const uint64_t t0 = global_timer_ns();
      while (ld_acquire_gpu(gbar) < target) {
        __nanosleep(32);
        if (flags[0]) break;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          flags[0] = 1;
          atomicOr(err, kErrWaitTimeout);
          break;
        }
      }
    }
  }
  named_bar_sync(kBarCompute, kComputeThreads);
}

// P1 item = a quad of rows: rope pairs 2q and 2q+1 of the unit order
struct Quad {
  Unit u0, u1;
  bool rotated;
};
__device__ __forceinline__ Quad quad_of(int q, int n_q, int n_kv, int rotary_dim) {
  Quad x;
  x.u0 = unit_of(2 * q, n_q, n_kv, rotary_dim);
  x.u1 = unit_of(2 * q + 1, n_q, n_kv, rotary_dim);
  x.rotated = x.u0.pair >= 0;
  return x;
}

// the CTA's attention share of layer l (cta c of G)
struct AttnShare {
  int64_t total, f0, f1;
  int G;
  bool active;
};

template <int NB>
__device__ __forceinline__ AttnShare attn_share(const StackArgs<NB>& args, int full, int nb, int n_kv) {
  AttnShare a;
  a.total = (int64_t)n_kv * args.prefix[full][nb];
  int64_t g = (a.total + kMinRowsPerCta - 1) / kMinRowsPerCta;

  if (g > (int64_t)gridDim.x) g = gridDim.x;
  if (g < 1) g = 1;
  a.G = (int)g;
  a.active = (int)blockIdx.x < a.G;
  a.f0 = a.total * blockIdx.x / a.G;
  a.f1 = a.total * (blockIdx.x + 1) / a.G;
  if (!a.active) a.f0 = a.f1 = 0;
  return a;
}

template <int NB>
__device__ __forceinline__ void share_start(const StackArgs<NB>& args, int full, int nb, int n_kv,
                                            int64_t f0, int& b, int& j) {
  int lo = 0, hi = nb - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)n_kv * args.prefix[full][mid] <= f0) lo = mid; else hi = mid - 1;
  }
  b = lo;
  const int64_t rows = args.prefix[full][lo + 1] - args.prefix[full][lo];
  j = (int)((f0 - (int64_t)n_kv * args.prefix[full][lo]) / rows);
}

template <int NB>
__global__ void __launch_bounds__(kThreads, 1)
    k_decode_stack(const __grid_constant__ StackArgs<NB> args, const Geo geo, const Ws ws) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = geo.hidden, n_q = geo.n_q, n_kv = geo.n_kv, nb = geo.nb;
  const int q_dim = n_q * kHeadDim;
  const size_t hrow = (size_t)H * sizeof(__nv_bfloat16);      // one q_k_v_proj row
  const size_t orow = (size_t)q_dim * sizeof(__nv_bfloat16);  // one o_proj row

  // ---- shared memory carve-up
  Ring ring;
  ring.base = base;
  ring.ns = geo.stages;
  ring.stage_bytes = geo.stage_bytes;
  unsigned char* p = base + (size_t)geo.stages * geo.stage_bytes;
  float* xs = reinterpret_cast<float*>(p);              // [NB][xfloats]
  p += sizeof(float) * NB * geo.xfloats;
  float* q_s = reinterpret_cast<float*>(p);
  p += sizeof(float) * 4 * kQStride;
  float4* p_s = reinterpret_cast<float4*>(p);
  p += sizeof(float4) * kComputeWarps * kTile;
  MergeSmem msm;
  msm.ms = reinterpret_cast<float*>(p);
  p += sizeof(float) * kComputeWarps * 4;
  msm.ls = reinterpret_cast<float*>(p);
  p += sizeof(float) * kComputeWarps * 4;
  msm.os = reinterpret_cast<float*>(p);
  p += sizeof(float) * kComputeWarps * 4 * kHeadDim;
  ring.full = reinterpret_cast<uint64_t*>(p);
  ring.empty = ring.full + geo.stages;
  p += sizeof(uint64_t) * 2 * geo.stages;
  ring.use = reinterpret_cast<volatile int*>(p);
  p += sizeof(int) * geo.stages;
  volatile int* flags = reinterpret_cast<volatile int*>(p);  // [0] abort, [1] last, [2] P1 done (layer + 1)
  p += sizeof(int) * 4;
  float* red = reinterpret_cast<float*>(p);                  // [kComputeWarps][NB]
  p += sizeof(float) * kComputeWarps * NB;
  float* inv_rms = reinterpret_cast<float*>(p);              // [NB]

  if (tid == 0) {
    for (int s = 0; s < geo.stages; ++s) {
      mbar_init(&ring.full[s], 1);
      mbar_init(&ring.empty[s], 1);
      ring.use[s] = -1;
    }
    flags[0] = flags[1] = flags[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int n_units = (n_q + 2 * n_kv) * (kHeadDim / 2) + n_q / 2;
  const int n_quads = n_units / 2;
  const int q0 = (int)((int64_t)n_quads * blockIdx.x / gridDim.x);
  const int q1 = (int)((int64_t)n_quads * (blockIdx.x + 1) / gridDim.x);
  const int n_pairs_o = H / 2;
  const int o0 = (int)((int64_t)n_pairs_o * blockIdx.x / gridDim.x);
  const int o1 = (int)((int64_t)n_pairs_o * (blockIdx.x + 1) / gridDim.x);

  // =================================================================== producer
  if (warp == kProducerWarp) {
    if (lane != 0) return;
    uint32_t i = 0;
    bool ok = true;
    auto fail = [&]() {
      if (ok) {
        ok = false;
        flags[0] = 1;
        atomicOr(ws.err, kErrWaitTimeout);
      }
    };
    for (int l = 0; l < geo.n_layers && ok; ++l) {
      const LayerDesc& L = args.layer[l];
      const int rot = args.rotary[L.full];
      const int rows_qkv = (n_q + 2 * n_kv) * kHeadDim;
      auto row_ptr = [&](int r) -> const __nv_bfloat16* {
        return r < rows_qkv ? L.qkv_w + (int64_t)r * H : L.g_w + (int64_t)(r - rows_qkv) * H;
      };
      // P1: q_k_v_proj / g_proj rows, four per stage
      for (int q = q0; q < q1 && ok; ++q, ++i) {
        if (!ring_acquire(ring, i, flags)) { fail(); break; }
        const Quad x = quad_of(q, n_q, n_kv, rot);
        uint64_t* bar = &ring.full[i % ring.ns];
        unsigned char* dst = ring.stage(i);
        mbar_arrive_expect_tx(bar, (uint32_t)(4 * hrow));
        if (x.rotated) {  // rows (a, a+1) and (b, b+1): [a0 a1 b0 b1]
          bulk_load(dst, row_ptr(x.u0.row_a), (uint32_t)(2 * hrow), bar);
          bulk_load(dst + 2 * hrow, row_ptr(x.u0.row_b), (uint32_t)(2 * hrow), bar);
        } else {          // four consecutive rows: [a0 b0 a1 b1]
          bulk_load(dst, row_ptr(x.u0.row_a), (uint32_t)(4 * hrow), bar);
        }
        ring_publish(ring, i);
      }
      if (!ok) break;
      trace(ws, l, kTrProdP1Issued);
      const AttnShare sh = attn_share(args, L.full, nb, n_kv);
      // While the projections run, pull the first KV tiles of this CTA's
      // attention share into L2.  Only one row per sequence changes in P1,
      // and L2 is coherent with those writes, so the early copies stay right.
      if (sh.active && sh.f0 < sh.f1) {
        int b, j, left = kL2PrefetchTiles;
        share_start(args, L.full, nb, n_kv, sh.f0, b, j);
        int64_t f = sh.f0;
        while (f < sh.f1 && left > 0) {
          const int64_t rows = args.prefix[L.full][b + 1] - args.prefix[L.full][b];
          const int64_t gs = (int64_t)n_kv * args.prefix[L.full][b] + j * rows;
          const int64_t r0 = f - gs, r1 = min(sh.f1, gs + rows) - gs;
          const Window w = window_of(args.pos[b], L.full != 0, geo.window, L.ring);
          for (int64_t r = r0; r < r1 && left > 0; --left) {
            int64_t e = min(r1, r + kTile);
            if (r < w.len_a && e > w.len_a) e = w.len_a;
            const int64_t slot = r < w.len_a ? w.first_slot + r : r - w.len_a;
            const int z = (int)((int64_t)b * L.capacity + slot);
            tma_prefetch_l2_4d(&args.tm[l][0], 0, z, 0, j);  // the caches' 4-D tile view (make_kv_tile_map)
            tma_prefetch_l2_4d(&args.tm[l][1], 0, z, 0, j);
            r = e;
          }
          f = gs + r1;
          if (++j == n_kv) { j = 0; ++b; }
        }
      }
      // P2: KV tiles, once every CTA has written layer l's new rows
      if (!spin_until(flags + 2, l + 1, flags)) { fail(); break; }
      trace(ws, l, kTrProdP2Start);
      __threadfence_block();
      fence_proxy_async_global();
      if (sh.active && sh.f0 < sh.f1) {
        int b, j;
        share_start(args, L.full, nb, n_kv, sh.f0, b, j);
        int64_t f = sh.f0;
        while (f < sh.f1 && ok) {
          const int64_t rows = args.prefix[L.full][b + 1] - args.prefix[L.full][b];
          const int64_t gs = (int64_t)n_kv * args.prefix[L.full][b] + j * rows;
          const int64_t r0 = f - gs, r1 = min(sh.f1, gs + rows) - gs;
          const Window w = window_of(args.pos[b], L.full != 0, geo.window, L.ring);
          for (int64_t r = r0; r < r1; ++i) {
            int64_t e = min(r1, r + kTile);
            if (r < w.len_a && e > w.len_a) e = w.len_a;
            const int64_t slot = r < w.len_a ? w.first_slot + r : r - w.len_a;
            if (!ring_acquire(ring, i, flags)) { fail(); break; }
            uint64_t* bar = &ring.full[i % ring.ns];
            unsigned char* kd = ring.stage(i);
            unsigned char* vd = kd + kv_half_bytes<__nv_bfloat16>();
            mbar_arrive_expect_tx(bar, 2 * kv_half_bytes<__nv_bfloat16>());
            const int z = (int)((int64_t)b * L.capacity + slot);
            tma_load_4d(kd, &args.tm[l][0], bar, 0, z, 0, j);
            tma_load_4d(vd, &args.tm[l][1], bar, 0, z, 0, j);
            ring_publish(ring, i);
            r = e;
          }
          f = gs + r1;
          if (++j == n_kv) { j = 0; ++b; }
        }
      }
      // P3: o_proj rows, two per stage
      trace(ws, l, kTrProdP3Start);
      for (int k = o0; k < o1 && ok; ++k, ++i) {
        if (!ring_acquire(ring, i, flags)) { fail(); break; }
        uint64_t* bar = &ring.full[i % ring.ns];
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * orow));
        bulk_load(ring.stage(i), L.o_w + (int64_t)(2 * k) * q_dim, (uint32_t)(2 * orow), bar);
        ring_publish(ring, i);
      }
      // Pull the next layer's share of q_k_v_proj rows into L2, so its P1
      // reads them from there.  Issued after this layer's o_proj rows: ahead
      // of them it delayed P3 (measured 1.135 -> 1.069 ms on 36 layers).
      if (l + 1 < geo.n_layers) {
        const LayerDesc& Ln = args.layer[l + 1];
        const int rotn = args.rotary[Ln.full];
        for (int q = q0; q < q1; ++q) {
          const Quad x = quad_of(q, n_q, n_kv, rotn);
          const int r = x.u0.row_a;
          const __nv_bfloat16* pa = r < rows_qkv ? Ln.qkv_w + (int64_t)r * H : Ln.g_w + (int64_t)(r - rows_qkv) * H;
          if (x.rotated) {
            const int rb = x.u0.row_b;
            bulk_prefetch_l2(pa, (uint32_t)(2 * hrow));
            bulk_prefetch_l2(Ln.qkv_w + (int64_t)rb * H, (uint32_t)(2 * hrow));
          } else {
            bulk_prefetch_l2(pa, (uint32_t)(4 * hrow));
          }
        }
      }
    }
    return;
  }

  // =================================================================== compute warps
  uint32_t i = 0, epoch = 0;
  for (int l = 0; l < geo.n_layers; ++l) {
    const LayerDesc& L = args.layer[l];
    const int rot = args.rotary[L.full];
    const float* src = l == 0 ? ws.h_in : ws.hbuf + (size_t)((l - 1) & 1) * nb * H;
    float* dst = l == geo.n_layers - 1 ? ws.out : ws.hbuf + (size_t)(l & 1) * nb * H;

    // ---- P1 prologue: x = h * w (unscaled) and 1/rms per sequence
    {
      float ss[NB];
      build_x_norm<8, __nv_bfloat16, NB, kComputeThreads, kMaxPer>(src, L.norm_w, H, nb, xs, geo.xfloats,
                                                                   ss, tid);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float v = warp_sum(ss[b]);
        if (lane == 0) red[warp * NB + b] = v;
      }
      named_bar_sync(kBarCompute, kComputeThreads);
      if (tid < NB) {
        float t = 0.f;
        for (int w = 0; w < kComputeWarps; ++w) t += red[w * NB + tid];
        inv_rms[tid] = 1.0f / sqrtf(t / (float)H + geo.eps);
      }
      named_bar_sync(kBarCompute, kComputeThreads);
    }

    // ---- P1: q_k_v_proj + g_proj + rope + cache write
    if (tid == 0) trace(ws, l, kTrP1Start);
    if (tid == 0) trace_cta(ws, l, 3);
    const int nchunk_h = H / 8;
    for (int q = q0; q < q1; ++q, ++i) {
      if ((int)(i % kComputeWarps) != warp) continue;
      const Quad x = quad_of(q, n_q, n_kv, rot);
      float2 acc[4][NB];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[rr][b] = make_float2(0.f, 0.f);
      const bool ok = !flags[0] && ring_wait(ring, i, flags);
      if (ok) {
        const unsigned char* sb = ring.stage(i);
        // rows of pair 0 and pair 1 in the stage (see the producer's layout)
        const unsigned char* a0 = sb;
        const unsigned char* b0 = sb + (x.rotated ? 2 : 1) * hrow;
        const unsigned char* a1 = sb + (x.rotated ? 1 : 2) * hrow;
        const unsigned char* b1 = sb + 3 * hrow;
        row_dot2<__nv_bfloat16, NB>(a0, b0, xs, geo.xfloats, nchunk_h, acc[0], acc[1]);
        row_dot2<__nv_bfloat16, NB>(a1, b1, xs, geo.xfloats, nchunk_h, acc[2], acc[3]);
      } else if (lane == 0 && !flags[0]) {
        flags[0] = 1;
        atomicOr(ws.err, kErrWaitTimeout);
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, i);
      if (!ok) continue;
#pragma unroll
      for (int pr = 0; pr < 2; ++pr) {
        const Unit& un = pr == 0 ? x.u0 : x.u1;
        float va = 0.f, vb = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const float sa = warp_sum(acc[2 * pr][b].x + acc[2 * pr][b].y);
          const float sbv = warp_sum(acc[2 * pr + 1][b].x + acc[2 * pr + 1][b].y);
          if (lane == b) {
            va = sa * inv_rms[b];
            vb = sbv * inv_rms[b];
          }
        }
        if (lane < nb) {
          const int b = lane;
          if (un.pair >= 0) {
            const float2 cs = args.cs[L.full][b][un.pair];
            const float ra = va * cs.x - vb * cs.y;
            const float rb = vb * cs.x + va * cs.y;
            va = ra;
            vb = rb;
          }
          if (un.kind == kQ) {
            float* qd = ws.q_rot + ((int64_t)b * n_q + un.head) * kHeadDim;
            qd[un.da] = va;
            qd[un.db] = vb;
          } else if (un.kind == kG) {
            ws.g[(int64_t)b * n_q + un.da] = va;
            ws.g[(int64_t)b * n_q + un.db] = vb;
          } else {
            const int64_t slot = write_slot_of(args.pos[b], L.ring);
            if (args.pos[b] < 0 || slot >= L.capacity) {
              atomicOr(ws.err, kErrIndex);
            } else {
              __nv_bfloat16* cd = (un.kind == kK ? L.k : L.v) +
                                  (((int64_t)b * L.capacity + slot) * n_kv + un.head) * kHeadDim;
              cd[un.da] = __float2bfloat16_rn(va);
              cd[un.db] = __float2bfloat16_rn(vb);
            }
          }
        }
      }
    }
    if (tid == 0) trace(ws, l, kTrP1End);
    if (tid == 0) trace_cta(ws, l, 0);
    grid_barrier(ws.gbar, epoch, flags, ws.err);   // q, k, v, g of layer l complete
    if (tid == 0) flags[2] = l + 1;                // the producer may load layer l's KV tiles
    if (tid == 0) trace(ws, l, kTrB1);

    // ---- P2: attention (all compute warps take tiles; warps 0-3 merge)
    const AttnShare sh = attn_share(args, L.full, nb, n_kv);
    if (sh.active && sh.f0 < sh.f1) {
      int b, j;
      share_start(args, L.full, nb, n_kv, sh.f0, b, j);
      int64_t f = sh.f0;
      while (f < sh.f1) {
        const int64_t rows = args.prefix[L.full][b + 1] - args.prefix[L.full][b];
        const int64_t gs = (int64_t)n_kv * args.prefix[L.full][b] + j * rows;
        const int64_t r0 = f - gs, r1 = min(sh.f1, gs + rows) - gs;
        const Window w = window_of(args.pos[b], L.full != 0, geo.window, L.ring);
        named_bar_sync(kBarConsumers, kComputeThreads);  // the previous group's merge is done
        attn_load_q<kComputeThreads>(q_s, ws.q_rot + ((int64_t)b * n_q + kGroup * j) * kHeadDim, tid);
        named_bar_sync(kBarConsumers, kComputeThreads);
        MmaQ mq;
        MmaState mst;
        mma_q_from_smem(mq, q_s);
        mst.reset();
        if (tid == 0 && f == sh.f0) trace(ws, l, kTrP2Q);
        for (int64_t r = r0; r < r1; ++i) {
          int64_t e = min(r1, r + kTile);
          if (r < w.len_a && e > w.len_a) e = w.len_a;
          if ((int)(i % kComputeWarps) == warp) {
            const bool ok = __all_sync(0xffffffffu, !flags[0] && ring_wait(ring, i, flags));
            if (ok) {
              unsigned char* kst = ring.stage(i);
              attn_tile_mma(kst, kst + kv_half_bytes<__nv_bfloat16>(), (int)(e - r), mq,
                            reinterpret_cast<float*>(p_s + warp * kTile), geo.scale_log2, mst);
            } else if (lane == 0 && !flags[0]) {
              flags[0] = 1;
              atomicOr(ws.err, kErrWaitTimeout);
            }
            __syncwarp();
            if (lane == 0) ring_release(ring, i);
          }
          r = e;
        }
        if (tid == 0 && f == sh.f0) trace(ws, l, kTrP2Tiles);
        {
          const int g = b * n_kv + j;
          const int c_first = cta_of(gs, sh.total, sh.G), c_last = cta_of(gs + rows - 1, sh.total, sh.G);
          attn_store_state_mma(mst, msm);
          attn_merge_group<kComputeWarps>(msm, flags, ws.part, ws.counters,
                                          ws.a + ((int64_t)b * n_q + kGroup * j) * kHeadDim, g,
                                          (int)blockIdx.x, c_first, c_last - c_first + 1);
          if (tid == 0 && f == sh.f0) trace(ws, l, kTrP2Merged);
        }
        f = gs + r1;
        if (++j == n_kv) { j = 0; ++b; }
      }
    }
    if (tid == 0) trace(ws, l, kTrP2End);
    if (tid == 0) trace_cta(ws, l, 1);
    grid_barrier(ws.gbar, epoch, flags, ws.err);   // every group of layer l merged
    if (tid == 0) trace(ws, l, kTrB2);

    // ---- P3 prologue: gated attention output a * sigmoid(g)
    build_x_gated<8, NB, kComputeThreads, kMaxPer>(ws.a, ws.g, q_dim, n_q, nb, xs, geo.xfloats, tid);
    named_bar_sync(kBarCompute, kComputeThreads);

    // ---- P3: o_proj + residual
    if (tid == 0) trace(ws, l, kTrP3Start);
    const int nchunk_o = q_dim / 8;
    for (int k = o0; k < o1; ++k, ++i) {
      if ((int)(i % kComputeWarps) != warp) continue;
      float2 acc[2][NB];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[rr][b] = make_float2(0.f, 0.f);
      const bool ok = !flags[0] && ring_wait(ring, i, flags);
      if (ok) {
        const unsigned char* sb = ring.stage(i);
        row_dot2<__nv_bfloat16, NB>(sb, sb + orow, xs, geo.xfloats, nchunk_o, acc[0], acc[1]);
      } else if (lane == 0 && !flags[0]) {
        flags[0] = 1;
        atomicOr(ws.err, kErrWaitTimeout);
      }
      __syncwarp();
      if (lane == 0) ring_release(ring, i);
      if (!ok) continue;
      float v0 = 0.f, v1 = 0.f;
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float s0 = warp_sum(acc[0][b].x + acc[0][b].y);
        const float s1 = warp_sum(acc[1][b].x + acc[1][b].y);
        if (lane == b) {
          v0 = s0;
          v1 = s1;
        }
      }
      if (lane < nb) {
        const int64_t idx = (int64_t)lane * H + 2 * k;
        const float h0 = __ldcg(src + idx), h1 = __ldcg(src + idx + 1);
        dst[idx] = h0 + v0;       // read and written by the same thread: out may alias h
        dst[idx + 1] = h1 + v1;
      }
    }
    if (tid == 0) trace(ws, l, kTrP3End);
    if (tid == 0) trace_cta(ws, l, 2);
    if (l + 1 < geo.n_layers) grid_barrier(ws.gbar, epoch, flags, ws.err);  // h of layer l+1 complete
    if (tid == 0) trace(ws, l, kTrB3);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
bool make_bf16_cache_map(CUtensorMap* map, const void* base, int n_kv, int64_t rows) {
  return make_kv_tile_map(map, base, true, n_kv, rows);
}

int xfloats_of(int cols) { return ((cols / 8 + 31) / 32) * 32 * 8; }

// smem besides the ring for NB sequences
size_t fixed_smem(int nb_tmpl, int xfloats) {
  return sizeof(float) * nb_tmpl * xfloats + sizeof(float) * 4 * kQStride +
         sizeof(float4) * kComputeWarps * kTile + sizeof(float) * kComputeWarps * (8 + 4 * kHeadDim) +
         sizeof(int) * 4 + sizeof(float) * kComputeWarps * nb_tmpl + sizeof(float) * nb_tmpl + 64;
}

template <int NB>
int launch_stack(const spark_geom* g, const float* h, int n_layers, const spark_layer_weights* w,
                 const spark_kv_layer* kv, const int32_t* cls, const int32_t* positions, int batch,
                 float* out, void* workspace, cudaStream_t st) {
  using namespace checks;
  StackArgs<NB>* args = new StackArgs<NB>();
  for (int l = 0; l < n_layers; ++l) {
    LayerDesc& d = args->layer[l];
    d.norm_w = (const __nv_bfloat16*)w[l].norm_w;
    d.qkv_w = (const __nv_bfloat16*)w[l].qkv_w;
    d.g_w = (const __nv_bfloat16*)w[l].g_w;
    d.o_w = (const __nv_bfloat16*)w[l].o_w;
    d.k = (__nv_bfloat16*)kv[l].k;
    d.v = (__nv_bfloat16*)kv[l].v;
    d.capacity = kv[l].capacity;
    d.ring = kv[l].ring_capacity;
    d.full = cls[l] == SPARK_FULL ? 1 : 0;
    if (!make_bf16_cache_map(&args->tm[l][0], kv[l].k, g->n_kv, (int64_t)batch * kv[l].capacity) ||
        !make_bf16_cache_map(&args->tm[l][1], kv[l].v, g->n_kv, (int64_t)batch * kv[l].capacity)) {
      delete args;
      return SPARK_ERR_CUDA;
    }
  }
  for (int f = 0; f < 2; ++f) {
    int r;
    double theta;
    rope_for(g, f ? SPARK_FULL : SPARK_SLIDING, &r, &theta);
    args->rotary[f] = r;
    fill_rope_table(&args->cs[f][0][0], kHeadDim / 2, batch, positions, r, theta);
    args->prefix[f][0] = 0;
    for (int b = 0; b < NB; ++b)
      args->prefix[f][b + 1] =
          args->prefix[f][b] +
          (b < batch ? window_of(positions[b], f == 1, g->window, 0).rows : 0);  // rows do not depend on the ring
  }
  for (int b = 0; b < NB; ++b) args->pos[b] = b < batch ? positions[b] : 0;

  const WsLayout Lw = ws_layout(g->hidden, g->n_q, g->n_kv, batch);
  Ws ws;
  ws.h_in = h;
  ws.out = out;
  ws.hbuf = ws_at<float>(workspace, Lw.hbuf);
  ws.q_rot = ws_at<float>(workspace, Lw.q_rot);
  ws.g = ws_at<float>(workspace, Lw.g);
  ws.a = ws_at<float>(workspace, Lw.a);
  ws.part = ws_at<float>(workspace, Lw.part);
  ws.counters = ws_at<uint32_t>(workspace, Lw.counters);
  ws.gbar = ws_at<uint32_t>(workspace, Lw.gbar);
  ws.err = ws_at<uint32_t>(workspace, Lw.err);
  static const bool tracing = getenv("SPARK_TRACE_STACK") != nullptr;
  ws.trace = tracing ? ws_at<uint64_t>(workspace, Lw.trace) : nullptr;

  Geo geo;
  geo.hidden = g->hidden;
  geo.n_q = g->n_q;
  geo.n_kv = g->n_kv;
  geo.window = g->window;
  geo.nb = batch;
  geo.n_layers = n_layers;
  geo.scale_log2 = g->scale * 1.4426950408889634f;
  geo.eps = g->eps;
  const int q_dim = g->n_q * kHeadDim;
  geo.xfloats = xfloats_of(g->hidden > q_dim ? g->hidden : q_dim);
  size_t sb = 4 * (size_t)g->hidden * 2;
  if (2 * (size_t)q_dim * 2 > sb) sb = 2 * (size_t)q_dim * 2;
  if ((size_t)2 * kv_half_bytes<__nv_bfloat16>() > sb) sb = 2 * kv_half_bytes<__nv_bfloat16>();
  sb = (sb + 1023) / 1024 * 1024;
  geo.stage_bytes = (int)sb;
  const size_t fixed = fixed_smem(NB, geo.xfloats);
  const size_t per_stage = sb + 2 * sizeof(uint64_t) + sizeof(int);
  const int stages = (int)((kSmemMax - 1024 - fixed) / per_stage);
  if (stages < 4) {
    delete args;
    return SPARK_ERR_UNSUPPORTED;
  }
  geo.stages = stages;
  const size_t smem = 1024 + fixed + (size_t)stages * per_stage;

  auto kern = k_decode_stack<NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) e = cudaMemsetAsync(ws.gbar, 0, 2 * sizeof(uint32_t), st);
  if (e == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(device_sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, *args, geo, ws);
  }
  delete args;
  return cuda_status(e);
}

}  // namespace
}  // namespace spark

using namespace spark;
using namespace spark::checks;

extern "C" int spark_attn_decode_stack(const spark_geom* g, const float* h, int32_t n_layers,
                                       const spark_layer_weights* w, const spark_kv_layer* kv,
                                       const int32_t* layer_class, const int32_t* positions,
                                       int32_t batch, float* out, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if (n_layers < 1 || !w || !kv || !layer_class) return SPARK_ERR_INVALID_ARG;
  if ((s = check_ws(g, batch, workspace, workspace_bytes)) != SPARK_OK) return s;
  if (!h || !out || !aligned16(h) || !aligned16(out)) return SPARK_ERR_INVALID_ARG;
  bool fused = batch <= kMaxNB && g->n_kv <= 4 && g->full_rotary_dim % 4 == 0 && g->hidden <= 4096;
  for (int l = 0; l < n_layers; ++l) {
    if ((s = check_weights(&w[l], true, true)) != SPARK_OK) return s;
    if ((s = check_kv(g, &kv[l], layer_class[l], positions, batch)) != SPARK_OK) return s;
    if (w[l].dtype != SPARK_BF16 || kv[l].dtype != SPARK_BF16) fused = false;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (!fused) {  // layer by layer through the per-layer kernels
    const float* cur = h;
    for (int l = 0; l < n_layers; ++l) {
      if ((s = spark_attn_decode(g, cur, &w[l], &kv[l], layer_class[l], positions, batch, out, workspace,
                                 workspace_bytes, stream)) != SPARK_OK)
        return s;
      cur = out;
    }
    return SPARK_OK;
  }
  for (int l0 = 0; l0 < n_layers; l0 += kMaxLayers) {
    const int n = n_layers - l0 < kMaxLayers ? n_layers - l0 : kMaxLayers;
    const float* src = l0 == 0 ? h : out;
    const spark_kv_layer* kvs = kv + l0;
    if (batch == 1)
      s = launch_stack<1>(g, src, n, w + l0, kvs, layer_class + l0, positions, batch, out, workspace, st);
    else if (batch == 2)
      s = launch_stack<2>(g, src, n, w + l0, kvs, layer_class + l0, positions, batch, out, workspace, st);
    else
      s = launch_stack<4>(g, src, n, w + l0, kvs, layer_class + l0, positions, batch, out, workspace, st);
    if (s != SPARK_OK) return s;
  }
  return SPARK_OK;
}
