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
#include <stdlib.h>

#include <algorithm>

#include <type_traits>

#include "attn_parts.cuh"
#include "launch.h"
#include "partition.h"

namespace spark {
namespace {

constexpr int kMinRowsPerCta = 64;            // default grid: at least this many rows per CTA
constexpr int64_t kDeepRows = 1 << 16;        // rows (x KV heads) per call from which the deep ring pays
// Cluster mode (short histories): up to 8 CTAs per group, about 64 rows
// each, for groups of at most 1536 rows.  Measured against 96 rows per CTA:
// default step 53.0 -> 52.7 us, 36-layer stack 0.944 -> 0.925 ms (its
// 512-row sliding layers now take 8 CTAs instead of 6).  Launches whose
// groups all fit as 16-CTA clusters (batch 1) take up to 16 CTAs of 32 rows
// (plan_attention).
constexpr int kMaxCluster = 8;
// Long histories at small batch (more than kClusterMaxRows rows, few
// groups): one cluster of kLongCluster CTAs per group (a non-portable
// cluster size) when the clusters all fit at once.  The 8192-row full layers
// of the 36-layer batch-1 step: 16 CTAs per KV head merging through DSMEM
// instead of 38 with a ticket merge, 828.3 -> 821.7 us per step (the 64
// CTAs stream the rows more slowly, 2.8 TB/s, but the merge tail shrinks).
constexpr int kLongCluster = 16;
constexpr int kStateBytes = (8 + kGroup * kHeadDim) * 4;  // a CTA's state: m[4], l[4], o[4][256]
// Cluster mode merges a group's state spread over the ranks (partition.h:
// merge_unit0, merge_owner, merge_slot_floats).
static_assert(kMergeUnits * 8 == kGroup * kHeadDim, "a merge unit is 8 floats of the group's output");
static_assert(kMergeMaxCluster >= kLongCluster && kMergeMaxCluster >= kMaxCluster, "the receive area covers every cluster");
template <int MINB>
constexpr int kRecvBytes = MINB == 1 ? merge_recv_bytes_max() : 0;  // cluster mode only with one CTA per SM
// When the next kernel may launch: 0 = right after the dependency wait, 1 =
// once this CTA's tiles are all in and its states merged or published.  Since
// every decode tile is requested before the wait (the token's own row comes
// from L2 after it), an early o_proj weight stream no longer delays the tiles
// at small batch: the two-layer batch-1 step 50.0 -> 49.1 us, the 36-layer one
// 865 -> 859 us.  Batches of more than kEarlyTriggerBatch keep the late
// trigger (64 sequences: 737.5 vs 740.7 us; at 64 short contexts 149.3 vs
// 152.7 us).  With o_proj's column path, the late trigger at batch 1 cost
// the 36-layer step 762 -> 794 us.
constexpr int kEarlyTriggerBatch = 4;
constexpr int kClusterRowsPerCta = 64;
constexpr int64_t kClusterMaxRows = 1536;

// RECV: bytes of the receive area of the cluster merge (0 in the
// two-CTAs-per-SM kernel, which never runs in cluster mode)
template <typename CT, int NS, int NC, int RECV>
struct Smem {
  static_assert(NS % NC == 0, "each stage must belong to one consumer warp");
  static constexpr int kStages = NS;
  static constexpr int kHalf = kv_half_bytes<CT>();  // the K (or V) half of a stage
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kQ = kStages * kStage;
  static constexpr int kP = kQ + 4 * kQStride * 4;
  static constexpr int kM = kP + NC * kTile * 16;
  static constexpr int kL = kM + NC * 4 * 4;
  static constexpr int kO = kL + NC * 4 * 4;
  static constexpr int kBars = kO + NC * 4 * kHeadDim * 4;
  static constexpr int kCst = kBars + 2 * kStages * 8;       // cluster mode: the CTA's state
  static constexpr int kFlags = kCst + kStateBytes;
  static constexpr int kRecv = kFlags + 16;                   // cluster mode: the other ranks' slices
  static constexpr int kMergeBar = kRecv + RECV;
  static constexpr int kBytes = kMergeBar + 16;
  static_assert(kCst % 16 == 0 && kRecv % 16 == 0, "bulk copies of the states need 16-byte alignment");
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 (128B swizzle)
};

// The long-history kernel runs two CTAs per SM: both must fit the SM's
// 228 KB of shared memory (1 KB of it reserved per CTA).
static_assert(CacheT<__nv_bfloat16>::kDeepBlocks *
                      (Smem<__nv_bfloat16, CacheT<__nv_bfloat16>::kDeep, kConsumers,
                            kRecvBytes<CacheT<__nv_bfloat16>::kDeepBlocks>>::kAlloc + 1024) <=
                  228 * 1024,
              "the two-CTAs-per-SM attention kernel no longer fits two CTAs on an SM");

template <int MAXB>
struct AttnArgs {
  int64_t prefix[MAXB + 1];  // rows read by sequences before b
  int32_t pos[MAXB];
};

// Enumerates, identically for the producer and the consumers, the groups a
// CTA's share meets and the tiles of each.
struct Share {
  int64_t f, f1;   // current flat position, end of share
  int b, j;        // current sequence, KV head
};

// The rows one group reads, by logical position kv_start + r, r < rows.
// Rows r < c_rows come from the cache: slot first_slot + r for r < len_a,
// then r - len_a (a ring wraps to row 0).  Rows r >= c_rows come from the
// staging buffer of a chunk of tokens (row kv_start + r - p0): the rows the
// chunk itself produces, which reach the cache only after attention.
struct Rows {
  int64_t kv_start, rows, c_rows, first_slot, len_a;
};

__host__ __device__ inline Rows rows_of(int64_t pos, bool full, int window, int ring, int64_t chunk_p0) {
  const Window w = window_of(pos, full, window, ring);
  Rows r{w.kv_start, w.rows, w.rows, w.first_slot, w.len_a};
  if (chunk_p0 >= 0) {
    // the cache holds the positions before the chunk: slot(x) = x mod ring
    // (x itself before the ring first fills), for every such x
    const int64_t c = chunk_p0 - w.kv_start;
    r.c_rows = c < 0 ? 0 : (c > w.rows ? w.rows : c);
    r.first_slot = ring > 0 ? w.kv_start % ring : w.kv_start;
    const int64_t to_end = ring > 0 ? ring - r.first_slot : r.c_rows;
    r.len_a = r.c_rows < to_end ? r.c_rows : to_end;
  }
  return r;
}

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

template <typename CT, int NS, int NC, int MINB, int MAXB>
__global__ void __launch_bounds__((NC + 1) * 32, MINB)
    k_attn_decode(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs,
                  const void* kcache, const void* vcache, int64_t chunk_p0, int cl, const float* __restrict__ q_rot, float* __restrict__ a_out,
                  float* __restrict__ part, uint32_t* __restrict__ counters, uint32_t* err,
                  int batch, int n_kv, int64_t capacity, int ring_capacity, int full,
                  int window, float scale_log2, const unsigned char* l2_pf, int64_t l2_pf_bytes,
                  int trig, uint64_t* trace, const __grid_constant__ AttnArgs<MAXB> args) {
  using S = Smem<CT, NS, NC, kRecvBytes<MINB>>;
  constexpr int kCT = NC * 32;  // consumer threads
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
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(base + S::kMergeBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    if (cl > 0) {
      // every rank receives the other ranks' m, l and its units: one phase
      const int r = (int)(blockIdx.x % cl);
      const int units = merge_unit0(r + 1, cl) - merge_unit0(r, cl);
      mbar_init(merge_bar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(merge_bar, (uint32_t)((cl - 1) * 32 * (1 + units)));
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    cta_stamp(trace, 0);
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
  // cluster mode: every rank's merge barrier is ready once every rank has
  // passed here (the matching wait comes before a rank sends its state)
  if (cl > 0) cluster_arrive();

  // Programmatic dependent launch.  q_rot and the token's own cache row
  // (the last row of each (sequence, KV head) group) come from the kernel
  // before this one, so they are read after pdl_wait().  Every other row
  // was written by kernels that completed before that one started: each
  // kernel of the block lets its successor launch only after its own
  // pdl_wait() has returned.  The setup below reads only this kernel's
  // arguments, and the producer issues the tiles of older rows, before the
  // wait.
  const int64_t total = (int64_t)n_kv * args.prefix[batch];
  const int G = gridDim.x, c = blockIdx.x;
  int64_t f0, f1;
  Share sh0{};  // cluster mode: where this CTA's share starts
  int64_t pos0 = 0;  // cluster mode: the group's position
  if (cl > 0) {
    // cluster mode: the cl CTAs of a cluster split one group's rows evenly
    // (a CTA may get none) and merge through DSMEM.  The group follows from
    // the CTA's index, and its arguments are read together: the producer's
    // first tile waits on these reads, and a search over the sequences
    // (dependent reads of the argument block) held it back by ~1 us.
    const int g = c / cl, r = c % cl, b = g / n_kv, j = g % n_kv;
    const int64_t p_lo = args.prefix[b], p_hi = args.prefix[b + 1];
    pos0 = args.pos[b];
    const int64_t rows_g = p_hi - p_lo;
    const int64_t gs = (int64_t)n_kv * p_lo + j * rows_g;
    f0 = gs + rows_g * r / cl;
    f1 = gs + rows_g * (r + 1) / cl;
    sh0.f = f0;
    sh0.f1 = f1;
    sh0.b = b;
    sh0.j = j;
  } else {
    f0 = total * c / G;
    f1 = total * (c + 1) / G;
    if (f0 >= f1) return;
  }
  const int32_t* pos = args.pos;
  float* cst = reinterpret_cast<float*>(base + S::kCst);  // [4] m, [4] l, [4][256] o

  // ------------------------------------------------------------ producer
  if (warp == NC) {
   if (lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if (chunk_p0 >= 0) {
      prefetch_tensormap(&tm_ks);
      prefetch_tensormap(&tm_vs);
    }
    uint32_t k = 0;
    bool ok = true, waited = false;
    Share sh = cl > 0 ? sh0 : share_begin(args, batch, n_kv, f0, f1);
    while (sh.f < sh.f1) {
      const int64_t rows = args.prefix[sh.b + 1] - args.prefix[sh.b];
      const int64_t gs = (int64_t)n_kv * args.prefix[sh.b] + sh.j * rows;
      const int64_t r0 = sh.f - gs, r1 = min(sh.f1, gs + rows) - gs;
      const Rows w = rows_of(cl > 0 ? pos0 : pos[sh.b], full != 0, window, ring_capacity, chunk_p0);
      for (int64_t r = r0; r < r1;) {
        int64_t e = min(r1, r + kTile);
        if (r < w.len_a && e > w.len_a) e = w.len_a;
        if (r < w.c_rows && e > w.c_rows) e = w.c_rows;
        const bool staged = r >= w.c_rows;
        const int64_t slot = r < w.len_a ? w.first_slot + r : r - w.len_a;
        // tiles holding rows the previous kernel wrote: any row of the
        // chunk's staging buffer.  (In decode the token's own row is written
        // over its tile by the consumer after the wait.)
        if (chunk_p0 >= 0 && staged && !waited) {
          pdl_wait();
          if (trig == 0) pdl_trigger();
          fence_proxy_async_global();
          waited = true;
        }
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
          const CUtensorMap* mk = staged ? &tm_ks : &tm_k;
          const CUtensorMap* mv = staged ? &tm_vs : &tm_v;
          const int z = staged ? (int)(w.kv_start + r - chunk_p0)
                               : (int)((int64_t)(chunk_p0 >= 0 ? 0 : sh.b) * capacity + slot);
          tma_load_4d(kd, mk, &full_bar[s], 0, z, 0, sh.j);
          tma_load_4d(vd, mv, &full_bar[s], 0, z, 0, sh.j);
        }
        ++k;
        if (cl > 0 && k == (uint32_t)NS) cta_stamp(trace, 6);  // timeline: a ring's worth of tiles requested
        r = e;
      }
      sh.f = gs + r1;
      if (++sh.j == n_kv) { sh.j = 0; ++sh.b; }
    }
    if (!waited) {
      pdl_wait();
      if (trig == 0) pdl_trigger();
    }
   }
    // The other lanes wait only once lane 0 has issued its tiles: had they
    // waited in a divergent branch of their own, that branch could run first
    // and hold lane 0's requests until the previous kernel completed.
    __syncwarp();
    if (lane != 0) {
      pdl_wait();
      if (trig == 0) pdl_trigger();
    }
    __syncwarp();
    if (cl == 0) return;
  } else {
  // ------------------------------------------------------------ consumers
  // bf16 caches take the tensor-core tile, fp32 caches the CUDA-core one
  constexpr bool kMma = std::is_same<CT, __nv_bfloat16>::value;
  const MergeSmem msm{ms, ls, os};
  uint32_t k = 0;
  Share sh = cl > 0 ? sh0 : share_begin(args, batch, n_kv, f0, f1);
  bool waited = false;
  AttnState st;
  MmaQ mq;
  MmaState mst;
  if (f0 >= f1) {  // cluster mode, no rows: an empty state
    pdl_wait();
    if (trig == 0) pdl_trigger();
    if (tid < kGroup) {
      cst[tid] = -INFINITY;
      cst[4 + tid] = 0.f;
    }
    for (int i = tid; i < kGroup * kHeadDim; i += kCT) cst[8 + i] = 0.f;
  }
  while (sh.f < sh.f1) {
    const int b = sh.b, j = sh.j;
    const int64_t rows = args.prefix[b + 1] - args.prefix[b];
    const int64_t gs = (int64_t)n_kv * args.prefix[b] + j * rows;
    const int64_t r0 = sh.f - gs, r1 = min(sh.f1, gs + rows) - gs;
    const Rows w = rows_of(pos[b], full != 0, window, ring_capacity, chunk_p0);

    named_bar_sync(kBarConsumers, kCT);  // the previous group's merge is done
    if (!waited) {
      pdl_wait();
      if (trig == 0) pdl_trigger();
      waited = true;
      if (tid == 0) cta_stamp(trace, 1);
    }
    // decode: the token's own row, if this share holds the group's last row
    const bool own_row = chunk_p0 < 0 && r1 == rows;
    NewRow<CT> nr;
    if (own_row) {
      const int64_t off = (((int64_t)b * capacity + write_slot_of(pos[b], ring_capacity)) * n_kv + j) * kHeadDim;
      nr.load(reinterpret_cast<const CT*>(kcache) + off, reinterpret_cast<const CT*>(vcache) + off, lane);
    }
    const float* qg = q_rot + ((int64_t)b * (kGroup * n_kv) + kGroup * j) * kHeadDim;
    attn_load_q<kCT>(q_s, qg, tid);
    named_bar_sync(kBarConsumers, kCT);
    if (tid == 0 && r0 == sh.f - gs && sh.f == f0) cta_stamp(trace, 2);
    if constexpr (kMma) {
      mma_q_from_smem(mq, q_s);
      mst.reset();
    } else {
      st.reset();
    }

    for (int64_t r = r0; r < r1;) {
      int64_t e = min(r1, r + kTile);
      if (r < w.len_a && e > w.len_a) e = w.len_a;
      if (r < w.c_rows && e > w.c_rows) e = w.c_rows;
      const int n = (int)(e - r);
      if ((int)(k % NC) == warp) {
        const int s = (int)(k % NS);
        const uint32_t u = k / NS;
        const bool ok = __all_sync(0xffffffffu, !flags[0] && mbar_wait_bounded(&full_bar[s], u & 1, flags, kWaitLimitNs));
        if (!ok) {
          if (lane == 0 && !flags[0]) {
            flags[0] = 1;
            atomicOr(err, kErrWaitTimeout);
          }
        } else {
          // timeline (cluster mode): consumer warp 0's first tile in
          const bool stamp = cl > 0 && warp == 0 && lane == 0 && u == 0;
          if (stamp) cta_stamp(trace, 7);
          unsigned char* kst = stages + s * S::kStage;
          const bool patch = own_row && e == rows;
          if (patch) {
            nr.store(kst, kst + S::kHalf, n - 1, lane);
            __syncwarp();
          }
          if constexpr (kMma)
            attn_tile_mma(kst, kst + S::kHalf, n, mq, reinterpret_cast<float*>(p_s + warp * kTile), scale_log2, mst);
          else
            attn_tile<CT>(kst, kst + S::kHalf, n, q_s, p_s + warp * kTile, scale_log2, st);
        }
        if (own_row && e == rows) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // before TMA refills the stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      ++k;
      r = e;
    }

    if (tid == 0) cta_stamp(trace, 3);
    const int g = b * n_kv + j;
    const int c_first = cta_of(gs, total, G), c_last = cta_of(gs + rows - 1, total, G);
    float* a_head0 = a_out + ((int64_t)b * (kGroup * n_kv) + kGroup * j) * kHeadDim;
    if constexpr (kMma)
      attn_store_state_mma(mst, msm);
    else
      attn_store_state(st, msm);
    if (cl > 0)
      attn_cta_state<NC>(msm, cst);
    else
      attn_merge_group<NC, 16>(msm, flags, part, counters, a_head0, g, c, c_first, c_last - c_first + 1, trace);
    sh.f = gs + r1;
    if (++sh.j == n_kv) { sh.j = 0; ++sh.b; }
  }
  if (tid == 0) cta_stamp(trace, 4);
  // trig 1: the next kernel may launch once this CTA's tiles are all in and
  // its group states merged or published
  if (trig == 1) pdl_trigger();
  }  // consumers

  if (cl > 0) {
    // The group's state is merged spread over the ranks.  Each rank sends,
    // with remote stores that complete on the receiver's merge barrier, its
    // m and l to every other rank and each unit of its o to the unit's owner;
    // each rank then merges its own units over the ranks, in rank order, and
    // writes them.  (Every state to rank 0, which merged them all: its 28 KB
    // (8 ranks) to 60 KB (16) of incoming stores landed 1.0-1.7 us after the
    // last was sent, and its merge took 1.6-2.0 us more.)
    __syncthreads();  // this CTA's state is complete
    cluster_wait();   // every rank's merge barrier is initialised
    const int r = c % cl;
    const int sf = merge_slot_floats(cl);
    if (tid < kMergeUnits) {  // consumer thread u sends unit u (and m, l to rank u)
      const int u = tid;
      const int q = merge_owner(u, cl);
      if (q != r) {
        const uint32_t bar = cluster_addr(merge_bar, (uint32_t)q);
        const uint32_t dst = cluster_addr(base + S::kRecv + (r * sf + 8 + 8 * (u - merge_unit0(q, cl))) * 4, (uint32_t)q);
        const float4* src = reinterpret_cast<const float4*>(cst + 8 + 8 * u);
        st_async_f32x4(dst, src[0], bar);
        st_async_f32x4(dst + 16, src[1], bar);
      }
      if (u < cl && u != r) {
        const uint32_t bar = cluster_addr(merge_bar, (uint32_t)u);
        const uint32_t dst = cluster_addr(base + S::kRecv + r * sf * 4, (uint32_t)u);
        const float4* src = reinterpret_cast<const float4*>(cst);
        st_async_f32x4(dst, src[0], bar);
        st_async_f32x4(dst + 16, src[1], bar);
      }
    }
    const int u0 = merge_unit0(r, cl), nu = merge_unit0(r + 1, cl) - u0;
    if (tid < kCT) {
      // bounded; on time-out the merge still waits (bounded again) so that
      // no store lands in the shared memory of an exited CTA
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(merge_bar, 0, flags, kWaitLimitNs));
      if (!ok) {
        if (lane == 0 && !flags[0]) {
          flags[0] = 1;
          atomicOr(err, kErrWaitTimeout);
        }
        int never = 0;
        mbar_wait_bounded(merge_bar, 0, &never, kWaitLimitNs);
      }
      // One lane per (unit, rank): the ranks of a unit sit in an aligned
      // group of ql lanes that takes the max and the sums by shuffles (a
      // loop over the ranks on one thread per unit took 1.1 us at 8 ranks
      // and 1.7-2.5 us at 16).  Fixed order: the results do not vary.
      const int ql = cl <= 2 ? 2 : cl <= 4 ? 4 : cl <= 8 ? 8 : 16;
      const float* rv = reinterpret_cast<const float*>(base + S::kRecv);
      const int g = c / cl, b = g / n_kv, j = g % n_kv;
      float* a_grp = a_out + ((int64_t)b * (kGroup * n_kv) + kGroup * j) * kHeadDim;
      for (int i0 = 0; i0 < nu * ql; i0 += kCT) {  // the same trip count in every lane
        const int i = i0 + tid, t = i / ql, q = i % ql;
        const int u = u0 + t, h = u / 32;
        const bool live = t < nu && q < cl;
        float m = -INFINITY, l = 0.f;
        float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
        if (live) {
          const float* sq = q == r ? cst : rv + q * sf;
          const float4* oq = reinterpret_cast<const float4*>(q == r ? cst + 8 + 8 * u : sq + 8 + 8 * t);
          m = sq[h];
          l = sq[4 + h];
          x0 = oq[0];
          x1 = oq[1];
        }
        float M = m;
        for (int o = ql >> 1; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float sc = m == -INFINITY ? 0.f : exp2f(m - M);
        float v[9] = {l * sc, x0.x * sc, x0.y * sc, x0.z * sc, x0.w * sc, x1.x * sc, x1.y * sc, x1.z * sc, x1.w * sc};
        for (int o = ql >> 1; o > 0; o >>= 1)
#pragma unroll
          for (int k = 0; k < 9; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
        if (q == 0 && t < nu && !flags[0]) {
          const float inv = 1.0f / v[0];
          float4* dst = reinterpret_cast<float4*>(a_grp + 8 * u);
          dst[0] = make_float4(v[1] * inv, v[2] * inv, v[3] * inv, v[4] * inv);
          dst[1] = make_float4(v[5] * inv, v[6] * inv, v[7] * inv, v[8] * inv);
        }
      }
    }
    if (tid == 0) cta_stamp(trace, 5);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <typename CT>
bool make_cache_map(CUtensorMap* map, const void* base, int n_kv, int64_t rows) {
  return make_kv_tile_map(map, base, std::is_same<CT, __nv_bfloat16>::value, n_kv, rows);
}

// The grid of a launch: `total` rows x KV heads, the longest group
// `max_rows` and the shortest `min_rows`, `groups` = batch x KV heads,
// `n_ctas` > 0 an explicit grid (stream-K split, no cluster), `max_ctas` the
// partial slots available, `long_clusters` the clusters of kLongCluster CTAs
// of this kernel that fit on the GPU at once.
struct AttnPlan {
  int ctas;     // CTAs of the launch
  int cluster;  // CTAs per cluster (cluster mode), 0 otherwise
};
template <int MINB>
AttnPlan plan_attention(int64_t total, int64_t max_rows, int64_t min_rows, int groups, int n_ctas, int max_ctas,
                        int long_clusters) {
  // Short histories in small launches: one cluster of cl CTAs per group,
  // merging through DSMEM (no partials in the workspace, no ticket).
  int cl = (int)((max_rows + kClusterRowsPerCta - 1) / kClusterRowsPerCta);
  if (cl > kMaxCluster) cl = kMaxCluster;
  // Groups few enough that they all fit as kLongCluster-CTA clusters at
  // once (batch 1): half the rows per CTA, up to kLongCluster CTAs.  With
  // the merge spread over the ranks, 16 CTAs of 32 rows beat 8 of 64 for
  // the 513-row sliding layers: the 36-layer batch-1 step 776 -> 762 us.
  if (MINB == 1 && cl >= 2 && groups <= long_clusters) {
    const int half = kClusterRowsPerCta / 2;
    const int cl_half = (int)((max_rows + half - 1) / half);
    cl = cl_half < kLongCluster ? cl_half : kLongCluster;
  }
  if (n_ctas > 0 || cl < 2 || max_rows > kClusterMaxRows ||
      (int64_t)groups * cl > device_sm_count() || (int64_t)groups * cl > max_ctas || MINB > 1)
    cl = 0;  // cluster mode only in the kernel of one CTA per SM (it holds the ranks' state slots)
  // longer histories at small batch: clusters of kLongCluster, if they all fit
  if (cl == 0 && n_ctas <= 0 && MINB == 1 && max_rows > kClusterMaxRows && groups <= long_clusters &&
      (int64_t)groups * kLongCluster <= max_ctas)
    cl = kLongCluster;
  int G = cl > 0 ? groups * cl : n_ctas;
  if (cl == 0 && G <= 0) {
    const int64_t want = (total + kMinRowsPerCta - 1) / kMinRowsPerCta;
    const int cap = MINB * device_sm_count();
    G = (int)(want < cap ? want : cap);
    // Groups of equal length that nearly fill the GPU (the sliding layer of
    // a large batch), or so short that the default grid has fewer CTAs than
    // groups: one CTA per group, no partials and no merge tail (64 sequences
    // of 512 rows: 34.8 -> 30.7 us per launch, the default 64-sequence step
    // 725.6 -> 720.3 us)
    if (max_rows == min_rows && groups <= cap && (4 * groups >= 3 * cap || want <= groups) && groups <= max_ctas)
      G = groups;
  }
  if (G < 1) G = 1;
  if (G > kMaxAttnCtas) G = kMaxAttnCtas;
  if (G > max_ctas) G = max_ctas;
  return {G, cl};
}

template <typename CT, int NS, int NC, int MINB, int MAXB>
cudaError_t launch_t(const float* q_rot, const void* kc, const void* vc, int n_kv,
                     int64_t capacity, int ring_capacity, bool full, int window, float scale,
                     const int32_t* positions, int batch, float* a, float* part,
                     uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                     size_t l2_pf_bytes, const ChunkSrc& chunk, int max_ctas, cudaStream_t st, int* held) {
  using S = Smem<CT, NS, NC, kRecvBytes<MINB>>;
  AttnArgs<MAXB> args;
  args.prefix[0] = 0;
  for (int b = 0; b < MAXB; ++b) {
    const int64_t rows = b < batch ? rows_of(positions[b], full, window, ring_capacity, chunk.p0).rows : 0;
    args.prefix[b + 1] = args.prefix[b] + rows;
    args.pos[b] = b < batch ? positions[b] : 0;
  }
  const int64_t total = (int64_t)n_kv * args.prefix[batch];
  int64_t max_rows = 0, min_rows = INT64_MAX;
  for (int b = 0; b < batch; ++b) {
    max_rows = std::max(max_rows, args.prefix[b + 1] - args.prefix[b]);
    min_rows = std::min(min_rows, args.prefix[b + 1] - args.prefix[b]);
  }
  auto kern = k_attn_decode<CT, NS, NC, MINB, MAXB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
  if (e != cudaSuccess) return e;
  // clusters of kLongCluster CTAs that fit at once, per device (0: none)
  static int long_clusters[64];
  static bool long_known[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (MINB == 1 && dev >= 0 && dev < 64 && !long_known[dev]) {
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(kLongCluster * 8);
      qc.blockDim = dim3((NC + 1) * 32);
      qc.dynamicSmemBytes = S::kAlloc;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = kLongCluster;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.attrs = qa;
      qc.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &qc) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a refused query or attribute leaves no sticky error
    long_clusters[dev] = n;
    long_known[dev] = true;
  }
  const int long_cl = MINB == 1 && dev >= 0 && dev < 64 ? long_clusters[dev] : 0;
  const AttnPlan plan = plan_attention<MINB>(total, max_rows, min_rows, batch * n_kv, n_ctas, max_ctas, long_cl);
  const int G = plan.ctas, cl = plan.cluster;
  // one CTA per SM: G SMs; two per SM: where they land is the scheduler's
  // choice, so every SM counts as held
  if (held) *held = MINB == 1 && G < device_sm_count() ? G : device_sm_count();

  // a chunk's tokens share one sequence's cache; decode rows are per sequence
  const int64_t cache_rows = chunk.p0 >= 0 ? capacity : (int64_t)batch * capacity;
  CUtensorMap mk, mv, mks, mvs;
  if (!make_cache_map<CT>(&mk, kc, n_kv, cache_rows) || !make_cache_map<CT>(&mv, vc, n_kv, cache_rows))
    return cudaErrorInvalidValue;
  if (chunk.p0 >= 0) {
    if (!make_cache_map<CT>(&mks, chunk.k, n_kv, batch) || !make_cache_map<CT>(&mvs, chunk.v, n_kv, batch))
      return cudaErrorInvalidValue;
  } else {
    mks = mk;
    mvs = mv;
  }
  const float scale_log2 = scale * 1.4426950408889634f;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3((NC + 1) * 32);
  cfg.dynamicSmemBytes = S::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cl > 0 ? (unsigned)cl : 1u;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cl > 0 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, mk, mv, mks, mvs, kc, vc, (int64_t)chunk.p0, cl, q_rot, a, part, counters,
                            err, batch, n_kv, capacity, ring_capacity, full ? 1 : 0, window, scale_log2,
                            static_cast<const unsigned char*>(l2_pf), (int64_t)l2_pf_bytes,
                            chunk.p0 < 0 && batch <= kEarlyTriggerBatch ? 0 : 1,
                            chunk.p0 < 0 ? layer_trace(1) : (uint64_t*)nullptr, args);
}

template <typename CT, int NS, int NC, int MINB>
cudaError_t launch_ns(const float* q_rot, const void* kc, const void* vc, int n_kv,
                      int64_t capacity, int ring_capacity, bool full, int window, float scale,
                      const int32_t* positions, int batch, float* a, float* part,
                      uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                      size_t l2_pf_bytes, const ChunkSrc& chunk, int max_ctas, cudaStream_t st, int* held) {
  if (batch <= 8)
    return launch_t<CT, NS, NC, MINB, 8>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                               positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, chunk, max_ctas, st, held);
  if (batch <= 64)
    return launch_t<CT, NS, NC, MINB, 64>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                                positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, chunk, max_ctas, st, held);
  return launch_t<CT, NS, NC, MINB, SPARK_MAX_BATCH>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full,
                                           window, scale, positions, batch, a, part, counters, err,
                                           n_ctas, l2_pf, l2_pf_bytes, chunk, max_ctas, st, held);
}

template <typename CT>
cudaError_t launch_ct(const float* q_rot, const void* kc, const void* vc, int n_kv,
                      int64_t capacity, int ring_capacity, bool full, int window, float scale,
                      const int32_t* positions, int batch, float* a, float* part,
                      uint32_t* counters, uint32_t* err, int n_ctas, const void* l2_pf,
                      size_t l2_pf_bytes, const ChunkSrc& chunk, int max_ctas, cudaStream_t st, int* held) {
  int64_t rows = 0;
  for (int b = 0; b < batch; ++b) rows += window_of(positions[b], full, window, ring_capacity).rows;
  if ((int64_t)n_kv * rows >= kDeepRows)
    return launch_ns<CT, CacheT<CT>::kDeep, kConsumers, CacheT<CT>::kDeepBlocks>(
        q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale, positions, batch, a, part,
        counters, err, n_ctas, l2_pf, l2_pf_bytes, chunk, max_ctas, st, held);
  return launch_ns<CT, CacheT<CT>::kShallow, kConsumers, 1>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window,
                                       scale, positions, batch, a, part, counters, err, n_ctas,
                                       l2_pf, l2_pf_bytes, chunk, max_ctas, st, held);
}

}  // namespace

bool make_kv_tile_map(CUtensorMap* map, const void* base, bool bf16, int n_kv, int64_t rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t es = bf16 ? 2 : 4;
  const cuuint64_t line = kLine / es;  // elements of a 128-byte line
  const cuuint64_t dims[4] = {line, (cuuint64_t)rows, kHeadDim / line, (cuuint64_t)n_kv};
  const cuuint64_t strides[3] = {(cuuint64_t)n_kv * kHeadDim * es, (cuuint64_t)kLine, kHeadDim * es};
  const cuuint32_t box[4] = {(cuuint32_t)line, (cuuint32_t)kTile, (cuuint32_t)(kHeadDim / line), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_attention(int cdtype, const float* q_rot, const void* kc, const void* vc,
                             int n_kv, int64_t capacity, int ring_capacity, bool full,
                             int window, float scale, const int32_t* positions, int batch,
                             float* a, float* part, uint32_t* counters, uint32_t* err,
                             int n_ctas, const void* l2_pf, size_t l2_pf_bytes, cudaStream_t st,
                             const ChunkSrc& chunk, int max_ctas, int* sms_held) {
  if (cdtype == SPARK_BF16)
    return launch_ct<__nv_bfloat16>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window,
                                    scale, positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, chunk,
                                    max_ctas, st, sms_held);
  return launch_ct<float>(q_rot, kc, vc, n_kv, capacity, ring_capacity, full, window, scale,
                          positions, batch, a, part, counters, err, n_ctas, l2_pf, l2_pf_bytes, chunk, max_ctas, st,
                          sms_held);
}

namespace {

// Copy the staged k / v rows of a chunk of tokens into their cache slots,
// once attention has read them: token t of the chunk goes to the slot of
// position p0 + t.  On a ring only the last `ring` tokens are copied (an
// earlier token's slot is taken by a later token of the same chunk).  One
// CTA per copied token.
template <typename CT>
__global__ void __launch_bounds__(256)
    k_commit_rows(const CT* __restrict__ ks, const CT* __restrict__ vs, CT* kc, CT* vc, int row_elems,
                  int64_t p0, int first, int ring) {
  pdl_wait();  // attention has finished reading the slots these rows replace
  pdl_trigger();
  const int t = first + blockIdx.x;
  const int64_t pos = p0 + t;
  const int64_t slot = ring > 0 ? pos % ring : pos;
  const int vec = (int)(row_elems * sizeof(CT) / 16);
  const uint4* sk = reinterpret_cast<const uint4*>(ks + (int64_t)t * row_elems);
  const uint4* sv = reinterpret_cast<const uint4*>(vs + (int64_t)t * row_elems);
  uint4* dk = reinterpret_cast<uint4*>(kc + slot * row_elems);
  uint4* dv = reinterpret_cast<uint4*>(vc + slot * row_elems);
  for (int i = threadIdx.x; i < vec; i += blockDim.x) {
    dk[i] = __ldcg(sk + i);
    dv[i] = __ldcg(sv + i);
  }
}

}  // namespace

cudaError_t launch_commit_rows(int cdtype, const void* ks, const void* vs, void* kc, void* vc,
                               int n_kv, int64_t p0, int m, int ring_capacity, cudaStream_t st) {
  const int first = ring_capacity > 0 && m > ring_capacity ? m - ring_capacity : 0;
  const int row_elems = n_kv * kHeadDim;
  if (cdtype == SPARK_BF16)
    return launch_pdl(k_commit_rows<__nv_bfloat16>, dim3(m - first), dim3(256), 0, st,
                      static_cast<const __nv_bfloat16*>(ks), static_cast<const __nv_bfloat16*>(vs),
                      static_cast<__nv_bfloat16*>(kc), static_cast<__nv_bfloat16*>(vc), row_elems, p0,
                      first, ring_capacity);
  return launch_pdl(k_commit_rows<float>, dim3(m - first), dim3(256), 0, st, static_cast<const float*>(ks),
                    static_cast<const float*>(vs), static_cast<float*>(kc), static_cast<float*>(vc),
                    row_elems, p0, first, ring_capacity);
}

}  // namespace spark
