// mma.cu -- the block's two projections for a batch of sequences, on the
// tensor cores (tcgen05 MMA with its accumulator in tensor memory, operands
// staged in shared memory by TMA):
//
//  * qkv: input RMSNorm, q_k_v_proj and g_proj of every sequence, with the
//    split into q / k / v, the per-class NeoX rope and the cache-row write
//    fused into the epilogue (turbospark-runtime 0.3.0,
//    src/families/spark/attn.rs, encode_attention_block: the fused
//    projection, the gate's projection of the same normed x, encode_split_qkv
//    with k and v landing in their slots, encode_rope_neox_subdim on q and k);
//  * o: the headwise sigmoid gate, o_proj and the raw residual add (attn.rs,
//    encode_sigmoid_head_gate_mul before the o_proj GEMV; mod.rs, the layer
//    loop's residual add);
//  * the rest of the decoder layer and the head (mod.rs, the module doc's
//    transcription of one layer and its last two lines): up -- the
//    post-attention RMSNorm, gate_proj and up_proj with the exact GELU product
//    in the epilogue, which writes the product straight into the (hi, lo)
//    rows down_proj reads; down -- down_proj and the residual add (the o
//    epilogue); head -- the final RMSNorm and the tied embedding (the o
//    epilogue without a residual).
//
// With B sequences a projection is the GEMM out[r][b] = sum_c W[r][c] x_b[c].
// The weight rows are the MMA's M side (128 rows a tile, bf16 straight from
// HBM), the sequences its N side, so the weights -- the bytes that bound the
// step -- are read once for the whole batch.  The MMA takes both operands in
// one 16-bit type, so each fp32 activation is split into two bf16 numbers,
// x = hi + lo with lo = bf16(x - hi): the B side holds [hi_0..hi_{B-1},
// lo_0..lo_{B-1}] (N = 2 * B rounded up to 8) and the epilogue adds the two
// halves of each sequence.  hi + lo keeps 16 significant bits of x, so the
// result is as close to the fp32 GEMV's as rounding order allows, while the
// HBM traffic is that of the bf16 weights alone.
//
// Two kernel launches per projection, for any batch (chunks of up to 128
// sequences, one MMA's 256 hi/lo columns each, covered by one grid):
//   k_prep_norm / k_prep_gate  build the activations' (hi, lo) rows and, for
//                              qkv, each sequence's rope (cos, sin) table;
//   k_proj_mma                 the GEMM.  A CTA is (weight tile, chunk,
//                              K-split); the chunks of a tile run side by side
//                              so its rows come from L2 after the first.
//                              Tiles of 128 weight rows are cut along K into
//                              `splits` pieces (1..8) so that the SMs stream
//                              weights.  The pieces of a tile are added in
//                              split order: by the CTAs of a thread-block
//                              cluster through DSMEM, each adding and
//                              finishing a share of the sequences; or, for
//                              small batches, through fp32 partials in the
//                              workspace, the last CTA of the tile (an atomic
//                              ticket) adding them and running the epilogue.
//                              Long grids of unsplit tiles run two CTAs per
//                              SM (up to two waves) or two weight tiles per
//                              CTA (the head).
//
// Warp roles in k_proj_mma (192 threads): warp 0 issues the TMA loads (one
// elected lane), warp 1 owns the tensor-memory columns and issues the MMAs
// (one elected lane), warps 2-5 read the accumulator back (warp w reads TMEM
// lanes 32 * (w % 4) .. +31, the quarter a warp may access) and run the
// epilogue.  With SPARK_TRACE_MMA set in the environment each CTA stamps its
// phases (%globaltimer) into the workspace's trace region.  Every wait is
// bounded (kWaitLimitNs): on time-out the kernel
// raises the error word, stops issuing, lets its copies in flight land and
// frees its tensor memory before it returns.
#include <math.h>
#include <stdlib.h>

#include <map>
#include <mutex>
#include <tuple>

#include "checks.h"
#include "launch.h"

namespace spark {
namespace {

// Weight stages the producer requests before the dependency wait; the
// activations of the first stages follow the wait, then the rest of their
// weights.  With every stage's weights requested first, the activations
// queued behind them (batch 64: 1% slower per step than 2 or 4).
constexpr int kMmaPreW = 4;
constexpr int kMmaThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kKBlock = 64;                                   // K elements per stage = one 128 B row
constexpr uint32_t kRowBytes = kKBlock * 2;                   // bf16
constexpr uint32_t kABytes = kMmaTileRows * kRowBytes;        // 16 KB: a tile's rows for one stage
constexpr int kBoxRows = 64;                                  // weight rows per TMA box
constexpr int kMaxStages = 16;
constexpr int kClusterMinBpad = 32;                           // cluster reduction from this many sequences
constexpr int kBarEpi = 1;                                    // named barrier of the epilogue warps
constexpr size_t kMaxDynSmem = 232448;                        // 227 KB per block on sm_100 parts
constexpr size_t kStageBudget = kMaxDynSmem - 2048;           // static smem + alignment slack
constexpr int kPrepThreads = 256;
constexpr int kMaxPairs = kHeadDim / 2;
constexpr size_t kSmemPerSm = 233472;                         // 228 KB of shared memory per SM
constexpr uint32_t kTmemCols = 512;                           // tensor-memory columns per SM

// ---------------------------------------------------------------------------
// tcgen05 helpers (inline PTX)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(cols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16, bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Two 8-column reads of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld_8x2(uint32_t ta, uint32_t tb, float (&a)[8], float (&b)[8]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(ta), "r"(tb)
      : "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a[i] = __uint_as_float(r[i]);
    b[i] = __uint_as_float(r[8 + i]);
  }
}

// Shared-memory matrix descriptor of a K-major operand written by TMA with
// the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// Bits: start address >> 4 [0,14), leading byte offset >> 4 [16,30) (unused
// by swizzled K-major layouts), stride byte offset >> 4 [32,46), descriptor
// version 1 [46,48), swizzle mode [61,64) (2 = 128-byte).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator [4,6) = 1, A and B
// bf16 [7,10) = [10,13) = 1, both K-major (bits 15, 16 = 0), N >> 3 at
// [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bit) {
  if (err) atomicOr(err, bit);
}

// every thread of every CTA of the cluster: arrive (release), then wait (acquire)
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// float4 at the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ float4 ld_cluster_f4(const void* local, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(local)), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(ra)
               : "memory");
  return v;
}

// four consecutive cache elements in one store (8 bytes bf16, 16 bytes fp32)
__device__ __forceinline__ void store_cache4(float* dst, const float (&v)[4]) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store_cache4(__nv_bfloat16* dst, const float (&v)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
  *reinterpret_cast<uint2*>(dst) = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// x -> (hi, lo) in bf16 with x ~= hi + lo
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ void store_split4(__nv_bfloat16* xh, __nv_bfloat16* xl, int i, float4 v) {
  __nv_bfloat16 h[4], l[4];
  split_bf16(v.x, h[0], l[0]);
  split_bf16(v.y, h[1], l[1]);
  split_bf16(v.z, h[2], l[2]);
  split_bf16(v.w, h[3], l[3]);
  *reinterpret_cast<uint2*>(xh + i) = *reinterpret_cast<const uint2*>(h);
  *reinterpret_cast<uint2*>(xl + i) = *reinterpret_cast<const uint2*>(l);
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < kPrepThreads / 32; ++i) t += red[i];
  return t;
}

// ---------------------------------------------------------------------------
// activation prologues
// ---------------------------------------------------------------------------
struct PrepArgs {
  double inv_freq[kMaxPairs];  // theta^(-2i/r) for i < r/2, in double (host)
  int32_t pos[SPARK_MAX_BATCH];
};

// Row pointers of padded sequence bb (of a launch's chunks of bpad) in the
// activation rows [chunk][2][bpad][k]: hi, then lo.
__device__ __forceinline__ void chunk_rows(__nv_bfloat16* x, int bb, int bpad, int k, __nv_bfloat16*& xh,
                                           __nv_bfloat16*& xl) {
  const int c = bb / bpad, b = bb - c * bpad;
  xh = x + ((size_t)c * 2 * bpad + b) * k;
  xl = x + ((size_t)c * 2 * bpad + bpad + b) * k;
}

// One CTA per (padded) sequence b: x = RMSNorm(h_b) * w ("plain w", eps
// inside the root) split into its hi and lo rows (chunk_rows); padded
// sequences get zero rows.  Also the rope table of sequence b:
// cs[b][i] = (cos, sin) of pos_b * theta^(-2i/r), the angle formed and
// reduced modulo 2 pi in double (at position 131072 an fp32 angle would be
// off by ~1e-2 rad), then evaluated in fp32.
// float4 groups of an activation row per prologue thread (rows of up to 8192)
constexpr int kPrepPer = 8192 / 4 / kPrepThreads;

__global__ void __launch_bounds__(kPrepThreads)
k_prep_norm(const float* __restrict__ h, const __nv_bfloat16* __restrict__ norm_w,
            __nv_bfloat16* __restrict__ x, float2* __restrict__ cs, int hidden, int nb, int bpad,
            float eps, int rotary_dim, const __grid_constant__ PrepArgs args) {
  __shared__ float red[kPrepThreads / 32];
  const int b = blockIdx.x;
  __nv_bfloat16 *xh, *xl;
  chunk_rows(x, b, bpad, hidden, xh, xl);
  // the norm weights do not depend on the previous kernel
  uint2 wr[kPrepPer];
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k) {
    const int i = 4 * (threadIdx.x + k * kPrepThreads);
    if (i < hidden) wr[k] = __ldg(reinterpret_cast<const uint2*>(norm_w + i));
  }
  pdl_wait();
  pdl_trigger();
  if (b >= nb) {
    for (int i = 4 * threadIdx.x; i < hidden; i += 4 * kPrepThreads) {
      *reinterpret_cast<uint2*>(xh + i) = make_uint2(0u, 0u);
      *reinterpret_cast<uint2*>(xl + i) = make_uint2(0u, 0u);
    }
    return;
  }
  // every load of h before any arithmetic: one round trip
  const float* hb = h + (size_t)b * hidden;
  float4 v[kPrepPer];
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k) {
    const int i = 4 * (threadIdx.x + k * kPrepThreads);
    v[k] = i < hidden ? __ldcg(reinterpret_cast<const float4*>(hb + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (threadIdx.x < rotary_dim / 2) {
    // the angle's whole turns: rint(ang / 2 pi), with the quotient formed as
    // a product (a correctly rounded division is a long fp64 sequence here);
    // the nearest integer is all that is needed, the reduction itself is the
    // fp64 fma below
    const int i = threadIdx.x;
    const double ang = (double)args.pos[b] * args.inv_freq[i];
    const double two_pi = 6.283185307179586476925;
    const double k = rint(ang * (1.0 / two_pi));
    const float r = (float)fma(-k, two_pi, ang);
    float sn, cn;
    sincosf(r, &sn, &cn);
    cs[(size_t)b * kMaxPairs + i] = make_float2(cn, sn);
  }
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k)
    ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
  const float inv = 1.0f / sqrtf(block_sum(ss, red) / (float)hidden + eps);
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k) {
    const int i = 4 * (threadIdx.x + k * kPrepThreads);
    if (i < hidden) {
      const float2 w01 = bf16x2_to_f32x2(wr[k].x), w23 = bf16x2_to_f32x2(wr[k].y);
      store_split4(xh, xl, i,
                   make_float4(v[k].x * w01.x * inv, v[k].y * w01.y * inv, v[k].z * w23.x * inv,
                               v[k].w * w23.y * inv));
    }
  }
}

// One CTA per (padded) sequence: the gated attention output a_b * sigmoid(g_b)
// (one gate per query head, broadcast over head_dim) split into hi / lo rows.
// Every load is issued before any arithmetic (one round trip).
__global__ void __launch_bounds__(kPrepThreads)
k_prep_gate(const float* __restrict__ a, const float* __restrict__ g, __nv_bfloat16* __restrict__ x,
            int q_dim, int n_q, int nb, int bpad) {
  const int b = blockIdx.x;
  __nv_bfloat16 *xh, *xl;
  chunk_rows(x, b, bpad, q_dim, xh, xl);
  pdl_wait();
  pdl_trigger();
  if (b >= nb) {
    for (int i = 4 * threadIdx.x; i < q_dim; i += 4 * kPrepThreads) {
      *reinterpret_cast<uint2*>(xh + i) = make_uint2(0u, 0u);
      *reinterpret_cast<uint2*>(xl + i) = make_uint2(0u, 0u);
    }
    return;
  }
  const float* ab = a + (size_t)b * q_dim;
  float4 v[kPrepPer];
  float gv[kPrepPer];
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k) {
    const int i = 4 * (threadIdx.x + k * kPrepThreads);
    if (i < q_dim) {
      v[k] = __ldcg(reinterpret_cast<const float4*>(ab + i));
      gv[k] = __ldcg(g + (size_t)b * n_q + i / kHeadDim);
    }
  }
#pragma unroll
  for (int k = 0; k < kPrepPer; ++k) {
    const int i = 4 * (threadIdx.x + k * kPrepThreads);
    if (i < q_dim) {
      const float sg = 1.0f / (1.0f + expf(-gv[k]));
      store_split4(xh, xl, i, make_float4(v[k].x * sg, v[k].y * sg, v[k].z * sg, v[k].w * sg));
    }
  }
}

// ---------------------------------------------------------------------------
// the GEMM
// ---------------------------------------------------------------------------
enum { kEpiQkv = 0, kEpiO = 1, kEpiUp = 2 };

struct MmaParams {
  int n_main_tiles;   // tiles over the main weight (the g tile follows them)
  int splits;         // K pieces per tile
  int kblocks;        // K / 64
  int bpad;           // sequences of a chunk rounded up to 8 (N = 2 * bpad)
  int nb;             // sequences of the launch (all chunks)
  int chunks;         // chunks of bpad sequences in the launch (1 up to 128 sequences)
  int mt;             // 128-row weight tiles per CTA (2: o epilogue, unsplit, two accumulators)
  int seq0;           // first sequence of this CTA's chunk (set in the kernel)
  int stages;         // pipeline depth
  int tmem_cols;      // allocated accumulator columns (power of two >= 2 * bpad)
  int split_halves;   // qkv: a tile pairs head dims d and d + 128 (rotary_dim 256)
  int cluster;        // 1: the splits of a tile form a cluster and reduce through DSMEM
  int g_rows;         // rows of the g tile (qkv), 0 for o
  uint32_t stage_bytes;
  // qkv epilogue
  float* q_rot;
  void* kc;
  void* vc;
  float* g_out;
  const float2* cs;
  int n_q, n_kv, rotary_dim;
  int64_t capacity;
  // o epilogue (also down_proj and the head: h null means no residual)
  const float* h;
  float* out;
  int hidden;  // output rows (hidden, or vocab for the head)
  // up epilogue
  __nv_bfloat16* xd;  // [chunk][2][bpad][inter] (hi, lo) rows of the GELU product (this chunk's in the kernel)
  int inter;
  // split-K and errors
  float* part;
  uint32_t* tickets;
  uint32_t* err;
  uint64_t* trace;  // [grid][kTraceEvents] %globaltimer stamps, or null (opt-in)
};

// Stamps of the opt-in timeline (SPARK_TRACE_MMA): per CTA, in this order.
enum { kTrStart, kTrXIssued, kTrFirstFull, kTrLastFull, kTrDone, kTrTicket, kTrReduced, kTrEnd,
       kTrStaged, kTrStored, kTraceEvents };

__device__ __forceinline__ void stamp(const MmaParams& p, int ev) {
  if (p.trace) p.trace[(size_t)blockIdx.x * kTraceEvents + ev] = global_timer_ns();
}

struct MmaSeq {
  int32_t slot[SPARK_MAX_BATCH];  // cache row each sequence writes (qkv)
};

constexpr int kMaxSplits = 8;
constexpr int kUnroll = 4;  // float4 elements per thread whose loads are all in flight together

// Y[b][m] = sum of part[s][b][m] over the splits, added in split order.  A
// thread owns float4 column m4 of rows b = b_first + 4k; every split of
// kUnroll elements is loaded before anything is added, so the loads overlap
// instead of paying the L2 latency one by one.
__device__ __forceinline__ void reduce_parts(float* Y, const float* base, int splits, int bpad, int et) {
  const int m4 = et & 31, b_first = et >> 5;
  const int nel = bpad >> 2;
  for (int k0 = 0; k0 < nel; k0 += kUnroll) {
    float4 v[kMaxSplits][kUnroll];
#pragma unroll
    for (int s = 0; s < kMaxSplits; ++s)
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (s < splits && k0 + u < nel)
          v[s][u] = __ldcg(reinterpret_cast<const float4*>(
                               base + ((size_t)s * bpad + b_first + 4 * (k0 + u)) * kMmaTileRows) + m4);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (k0 + u < nel) {
        float4 acc = v[0][u];
#pragma unroll
        for (int s = 1; s < kMaxSplits; ++s) {
          if (s < splits) {
            acc.x += v[s][u].x;
            acc.y += v[s][u].y;
            acc.z += v[s][u].z;
            acc.w += v[s][u].w;
          }
        }
        *reinterpret_cast<float4*>(Y + (size_t)(b_first + 4 * (k0 + u)) * kMmaTileRows + 4 * m4) = acc;
      }
    }
  }
  named_bar_sync(kBarEpi, kEpiThreads);
}

// out[b][R] = h[b][R] + the sum of the splits (in split order), float4 per
// thread, for sequences [bb0, bb1); without h (the head) out[b][R] = the sum.  Y non-null: the sum is already in Y
// ([bpad][128], the cluster reduction); else the splits' partials are read
// from `base`.
__device__ __forceinline__ void epilogue_o(const MmaParams& p, int tile, const float* base, const float* Y,
                                           int bb0, int bb1, int et) {
  const int m4 = et & 31, b_first = bb0 + (et >> 5);
  const int R = kMmaTileRows * tile + 4 * m4;
  if (R >= p.hidden) return;  // hidden % 64 == 0: a float4 is wholly inside or outside
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  if (Y) {
    for (int b = b_first; b < bb1; b += 4) {
      const float4 hv = p.h ? __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)b * p.hidden + R)) : zero;
      const float4 y = *reinterpret_cast<const float4*>(Y + (size_t)b * kMmaTileRows + 4 * m4);
      *reinterpret_cast<float4*>(p.out + (size_t)b * p.hidden + R) =
          make_float4(hv.x + y.x, hv.y + y.y, hv.z + y.z, hv.w + y.w);
    }
    return;
  }
  const int nel = bb1 > b_first ? (bb1 - b_first + 3) / 4 : 0;
  for (int k0 = 0; k0 < nel; k0 += kUnroll) {
    float4 v[kMaxSplits][kUnroll], hv[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int b = b_first + 4 * (k0 + u);
      if (k0 + u < nel) {
        hv[u] = p.h ? __ldcg(reinterpret_cast<const float4*>(p.h + (size_t)b * p.hidden + R)) : zero;
#pragma unroll
        for (int s = 0; s < kMaxSplits; ++s)
          if (s < p.splits)
            v[s][u] = __ldcg(reinterpret_cast<const float4*>(base + ((size_t)s * p.bpad + b) * kMmaTileRows) + m4);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (k0 + u < nel) {
        const int b = b_first + 4 * (k0 + u);
        float4 acc = v[0][u];
#pragma unroll
        for (int s = 1; s < kMaxSplits; ++s) {
          if (s < p.splits) {
            acc.x += v[s][u].x;
            acc.y += v[s][u].y;
            acc.z += v[s][u].z;
            acc.w += v[s][u].w;
          }
        }
        *reinterpret_cast<float4*>(p.out + (size_t)b * p.hidden + R) =
            make_float4(hv[u].x + acc.x, hv[u].y + acc.y, hv[u].z + acc.z, hv[u].w + acc.w);
      }
    }
  }
}

__device__ __forceinline__ float gelu_erf(float z) { return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f)); }

// The up tile's rows 0..63 are gate_proj rows j0..j0+63 and rows 64..127 the
// up_proj rows of the same j: m[b][j] = gelu(gate) * up, written as the
// (hi, lo) rows b and bpad + b of down_proj's input, float4 per thread, for
// sequences [bb0, bb1) (padded sequences included: their Y is zero).
__device__ __forceinline__ void epilogue_up(const MmaParams& p, int tile, const float* Y, int bb0, int bb1,
                                            int et) {
  const int c4 = et & 15;
  const int j = kBoxRows * tile + 4 * c4;
  if (j >= p.inter) return;  // inter % 8 == 0: a float4 is wholly inside or outside
  for (int b = bb0 + (et >> 4); b < bb1; b += kEpiThreads / 16) {
    const float4 g = *reinterpret_cast<const float4*>(Y + (size_t)b * kMmaTileRows + 4 * c4);
    const float4 u = *reinterpret_cast<const float4*>(Y + (size_t)b * kMmaTileRows + kBoxRows + 4 * c4);
    const float4 m = make_float4(gelu_erf(g.x) * u.x, gelu_erf(g.y) * u.y, gelu_erf(g.z) * u.z, gelu_erf(g.w) * u.w);
    store_split4(p.xd + (size_t)b * p.inter, p.xd + (size_t)(p.bpad + b) * p.inter, j, m);
  }
}

// q / k / v / g of one tile from Y ([bpad][128] fp32, the reduced GEMM):
// rope on the q and k dims below the rotary dim (the pair partner is another
// row of the same tile), q to q_rot, k and v to their cache rows, g to g_out.
// The rope (cos, sin) of the tile's 64 pairs for every sequence are first
// copied to CS ([bpad][64] float2) with all loads in flight together.
template <typename CT>
__device__ __forceinline__ void epilogue_qkv(const MmaParams& p, const MmaSeq& seq, int tile, bool g_tile,
                                             const float* Y, float2* CS, int m, int et, int bb0, int bb1) {
  if (g_tile) {
    if (m < p.g_rows)
      for (int b = bb0; b < bb1; ++b) p.g_out[(size_t)b * p.n_q + m] = Y[b * kMmaTileRows + m];
    return;
  }
  const int unit = tile >> 1, sel = tile & 1;
  const bool halves = p.split_halves != 0;
  const bool has_rot = unit < p.n_q + p.n_kv && (halves || sel == 0);
  const int p0 = halves ? kBoxRows * sel : 0;  // first rope pair of the tile
  if (has_rot) {
    const int c4 = et & 31, b_first = bb0 + (et >> 5);  // float4 = two pairs
    const int nel = bb1 > b_first ? (bb1 - b_first + 3) / 4 : 0;
    for (int k0 = 0; k0 < nel; k0 += 2 * kUnroll) {
      float4 v[2 * kUnroll];
#pragma unroll
      for (int u = 0; u < 2 * kUnroll; ++u)
        if (k0 + u < nel)
          v[u] = __ldcg(reinterpret_cast<const float4*>(p.cs + (size_t)(b_first + 4 * (k0 + u)) * kMaxPairs + p0) + c4);
#pragma unroll
      for (int u = 0; u < 2 * kUnroll; ++u)
        if (k0 + u < nel) reinterpret_cast<float4*>(CS + (size_t)(b_first + 4 * (k0 + u)) * kBoxRows)[c4] = v[u];
    }
  }
  named_bar_sync(kBarEpi, kEpiThreads);
  if (et == 0) stamp(p, kTrStaged);
  // A thread owns rows m4 .. m4 + 3 of the tile (one 64-row box never splits
  // them) for sequences b_first, b_first + 4, ...: it reads its four values
  // and their rope partners from Y and writes them with one vector store.
  const int m4 = 4 * (et & 31), b_first = bb0 + (et >> 5);
  int dd[4], pp[4], mm[4];
  float sg[4];
  bool rr[4];
  int kind = 0, head = 0, R0 = 0;
  const int hr = p.rotary_dim >> 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m_ = m4 + i;
    const int d = halves ? (m_ < kBoxRows ? kBoxRows * sel + m_ : 2 * kBoxRows + kBoxRows * sel + (m_ - kBoxRows))
                         : kMmaTileRows * sel + m_;
    if (i == 0) {
      R0 = kHeadDim * unit + d;
      if (unit < p.n_q) {
        kind = 0;
        head = unit;
      } else if (unit < p.n_q + p.n_kv) {
        kind = 1;
        head = unit - p.n_q;
      } else {
        kind = 2;
        head = unit - p.n_q - p.n_kv;
      }
    }
    dd[i] = d;
    rr[i] = kind != 2 && d < p.rotary_dim;
    mm[i] = m_;
    pp[i] = 0;
    sg[i] = 0.f;
    if (rr[i]) {
      if (d < hr) {
        pp[i] = d;
        sg[i] = -1.f;
        mm[i] = halves ? m_ + kBoxRows : m_ + hr;
      } else {
        pp[i] = d - hr;
        sg[i] = 1.f;
        mm[i] = halves ? m_ - kBoxRows : m_ - hr;
      }
      pp[i] -= p0;  // pair within the staged table
    }
  }
  const int q_dim = p.n_q * kHeadDim;
  CT* cache = static_cast<CT*>(kind == 1 ? p.kc : p.vc);
  // the four rows usually rotate alike with consecutive partners and pairs:
  // then they are read as float4 (scalar reads at stride 4 conflict 4-way)
  bool vec = true;
#pragma unroll
  for (int i = 1; i < 4; ++i)
    vec = vec && rr[i] == rr[0] && sg[i] == sg[0] && mm[i] == mm[0] + i && pp[i] == pp[0] + i;
  vec = vec && (mm[0] & 3) == 0 && (pp[0] & 1) == 0;
  for (int b = b_first; b < bb1; b += 4) {
    float val[4];
    if (vec) {
      const float4 y = *reinterpret_cast<const float4*>(Y + b * kMmaTileRows + m4);
      if (rr[0]) {
        const float4 yp = *reinterpret_cast<const float4*>(Y + b * kMmaTileRows + mm[0]);
        const float4 c01 = *reinterpret_cast<const float4*>(CS + b * kBoxRows + pp[0]);
        const float4 c23 = *reinterpret_cast<const float4*>(CS + b * kBoxRows + pp[0] + 2);
        val[0] = fmaf(sg[0] * yp.x, c01.y, y.x * c01.x);
        val[1] = fmaf(sg[0] * yp.y, c01.w, y.y * c01.z);
        val[2] = fmaf(sg[0] * yp.z, c23.y, y.z * c23.x);
        val[3] = fmaf(sg[0] * yp.w, c23.w, y.w * c23.z);
      } else {
        val[0] = y.x;
        val[1] = y.y;
        val[2] = y.z;
        val[3] = y.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v = Y[b * kMmaTileRows + m4 + i];
        if (rr[i]) {
          const float2 c = CS[b * kBoxRows + pp[i]];
          val[i] = fmaf(sg[i] * Y[b * kMmaTileRows + mm[i]], c.y, v * c.x);
        } else {
          val[i] = v;
        }
      }
    }
    if (kind == 0) {
      *reinterpret_cast<float4*>(p.q_rot + (size_t)b * q_dim + R0) = make_float4(val[0], val[1], val[2], val[3]);
    } else {
      CT* dst = cache + (((size_t)b * p.capacity + seq.slot[p.seq0 + b]) * p.n_kv + head) * kHeadDim + dd[0];
      store_cache4(dst, val);
    }
  }
  if (et == 0) stamp(p, kTrStored);
}

// The epilogue of one tile for sequences [bb0, bb1), run by the 128 epilogue
// threads: from Y ([bpad][128] fp32, the finished sum), or -- parts non-null
// -- from the splits' partial results in the workspace.
template <int E, typename CT>
__device__ __forceinline__ void epilogue(const MmaParams& p, const MmaSeq& seq, int tile, bool g_tile, float* Y,
                                         const float* parts, int bb0, int bb1, int m, int et) {
  if (E == kEpiO) {
    epilogue_o(p, tile, parts, parts ? nullptr : Y, bb0, bb1, et);
  } else {
    if (parts) {
      reduce_parts(Y, parts, p.splits, p.bpad, et);
      if (et == 0) stamp(p, kTrReduced);
    }
    if (E == kEpiQkv)
      epilogue_qkv<CT>(p, seq, tile, g_tile, Y, reinterpret_cast<float2*>(Y + p.bpad * kMmaTileRows), m, et, bb0,
                       bb1);
    else
      epilogue_up(p, tile, Y, bb0, bb1, et);
  }
  if (p.trace) {
    named_bar_sync(kBarEpi, kEpiThreads);
    if (et == 0) stamp(p, kTrEnd);
  }
}

template <int E, typename CT>
__global__ void __launch_bounds__(kMmaThreads, 1)
k_proj_mma(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_g,
           const __grid_constant__ CUtensorMap tm_x, const MmaParams pk,
           const __grid_constant__ MmaSeq seq) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t done_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag, last_flag, no_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA = (tile, chunk, split), split fastest (a cluster's CTAs are
  // consecutive), then chunk: the chunks of one weight tile run side by side
  // and all but the first find its rows in L2
  const int cta = blockIdx.x / pk.splits;
  const int split = blockIdx.x - cta * pk.splits;
  const int chunk = cta % pk.chunks, tile = cta / pk.chunks;
  MmaParams p = pk;  // this chunk's view: its sequences and their outputs
  p.seq0 = chunk * pk.bpad;
  p.nb = pk.nb - p.seq0 < pk.bpad ? pk.nb - p.seq0 : pk.bpad;
  if (chunk > 0) {
    const size_t s0 = (size_t)p.seq0;
    if (p.q_rot) p.q_rot += s0 * p.n_q * kHeadDim;
    if (p.g_out) p.g_out += s0 * p.n_q;
    if (p.cs) p.cs += s0 * kMaxPairs;
    if (p.kc) p.kc = static_cast<CT*>(p.kc) + s0 * p.capacity * p.n_kv * kHeadDim;
    if (p.vc) p.vc = static_cast<CT*>(p.vc) + s0 * p.capacity * p.n_kv * kHeadDim;
    if (p.h) p.h += s0 * p.hidden;
    if (p.out) p.out += s0 * p.hidden;
    if (p.xd) p.xd += (size_t)chunk * 2 * p.bpad * p.inter;
  }
  const int x_row = chunk * 2 * pk.bpad;  // this chunk's activation rows in the tensor map
  const int kb0 = split * p.kblocks / p.splits;
  const int nk = (split + 1) * p.kblocks / p.splits - kb0;
  const bool g_tile = E == kEpiQkv && tile >= p.n_main_tiles;
  const uint32_t x_bytes = (uint32_t)p.bpad * 2u * kRowBytes;
  const int mt = E == kEpiO ? p.mt : 1;  // weight tiles of this CTA, sharing each activation stage
  const uint32_t a_bytes = g_tile ? (uint32_t)p.g_rows * kRowBytes : kABytes * (uint32_t)mt;
  // sequences the epilogue covers: the up epilogue also zeroes the padded ones
  const int nrows = E == kEpiUp ? p.bpad : p.nb;
  float* const Y0 = reinterpret_cast<float*>(smem);
  volatile int* abort_v = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&done_bar, 1);
    abort_flag = 0;
    last_flag = 0;
    no_abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_w);
    prefetch_tensormap(&tm_x);
    if (g_tile || E == kEpiUp) prefetch_tensormap(&tm_g);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (threadIdx.x == 0) stamp(p, kTrStart);

  if (warp == 0) {
    // ---- producer: weights first (they do not depend on earlier kernels),
    // then the activations once the kernels before this one are done
    if (lane == 0) {
      int r0, r1;
      if (E == kEpiQkv && p.split_halves) {
        r0 = 2 * kMmaTileRows * (tile >> 1) + kBoxRows * (tile & 1);
        r1 = r0 + 2 * kBoxRows;
      } else {
        r0 = kMmaTileRows * tile;
        r1 = r0 + kBoxRows;
      }
      auto stage = [&](int s) { return smem + (size_t)s * p.stage_bytes; };
      auto load_w = [&](int s, int kb) {
        if (g_tile) {
          tma_load_2d(stage(s), &tm_g, &full_bar[s], kb * kKBlock, 0);
        } else if (E == kEpiUp) {  // gate rows, then the up rows of the same j
          tma_load_2d(stage(s), &tm_w, &full_bar[s], kb * kKBlock, kBoxRows * tile);
          tma_load_2d(stage(s) + kABytes / 2, &tm_g, &full_bar[s], kb * kKBlock, kBoxRows * tile);
        } else if (mt > 1) {  // tiles mt * tile .. + mt - 1, each as two 64-row boxes
          for (int h = 0; h < mt; ++h) {
            const int rr = kMmaTileRows * (mt * tile + h);
            tma_load_2d(stage(s) + h * kABytes, &tm_w, &full_bar[s], kb * kKBlock, rr);
            tma_load_2d(stage(s) + h * kABytes + kABytes / 2, &tm_w, &full_bar[s], kb * kKBlock, rr + kBoxRows);
          }
        } else {
          tma_load_2d(stage(s), &tm_w, &full_bar[s], kb * kKBlock, r0);
          tma_load_2d(stage(s) + kABytes / 2, &tm_w, &full_bar[s], kb * kKBlock, r1);
        }
      };
      const int pre = nk < p.stages ? nk : p.stages;
      const int pre_w = pre < kMmaPreW ? pre : kMmaPreW;  // weight stages requested before the wait
      for (int i = 0; i < pre; ++i) mbar_arrive_expect_tx(&full_bar[i], a_bytes + x_bytes);
      for (int i = 0; i < pre_w; ++i) load_w(i, kb0 + i);
      pdl_wait();
      pdl_trigger();
      fence_proxy_async_global();
      // the activations of the first stages, then the rest of their weights
      for (int i = 0; i < pre; ++i)
        tma_load_2d(stage(i) + kABytes * mt, &tm_x, &full_bar[i], (kb0 + i) * kKBlock, x_row);
      for (int i = pre_w; i < pre; ++i) load_w(i, kb0 + i);
      stamp(p, kTrXIssued);
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % p.stages;
        if (!mbar_wait_bounded(&empty_bar[s], ((i / p.stages) - 1) & 1, abort_v, kWaitLimitNs)) {
          raise_error(p.err, kErrWaitTimeout);
          *abort_v = 1;
          break;
        }
        mbar_arrive_expect_tx(&full_bar[s], a_bytes + x_bytes);
        load_w(s, kb0 + i);
        tma_load_2d(stage(s) + kABytes * mt, &tm_x, &full_bar[s], (kb0 + i) * kKBlock, x_row);
        issued = i + 1;
      }
      if (*abort_v) {
        // let the copies still in flight land before the CTA can exit
        for (int i = issued > p.stages ? issued - p.stages : 0; i < issued; ++i)
          mbar_wait_bounded(&full_bar[i % p.stages], (i / p.stages) & 1, &no_abort, kWaitLimitNs);
      }
    }
    __syncwarp();  // the other lanes wait only once lane 0 has issued its requests
    if (lane != 0) {
      pdl_wait();
      pdl_trigger();
    }
  } else if (warp == 1) {
    // ---- MMA issuer: 4 MMAs of K = 16 per stage, then free the stage
    pdl_wait();
    pdl_trigger();
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kMmaTileRows, 2 * p.bpad);
      for (int i = 0; i < nk; ++i) {
        const int s = i % p.stages;
        if (!mbar_wait_bounded(&full_bar[s], (i / p.stages) & 1, abort_v, kWaitLimitNs)) {
          raise_error(p.err, kErrWaitTimeout);
          *abort_v = 1;
          break;
        }
        tc_fence_after();
        if (i == 0) stamp(p, kTrFirstFull);
        if (i == nk - 1) stamp(p, kTrLastFull);
        const uint32_t a_addr = smem_u32(smem + (size_t)s * p.stage_bytes);
        const uint64_t dx = sw128_desc(a_addr + kABytes * mt);
        for (int h = 0; h < mt; ++h) {  // accumulator h at columns h * tmem_cols / mt
          const uint64_t da = sw128_desc(a_addr + h * kABytes);
          const uint32_t dt = tmem + (uint32_t)(h * (p.tmem_cols / mt));
#pragma unroll
          for (int k = 0; k < kKBlock / 16; ++k)
            mma_bf16(dt, da + 2u * k, dx + 2u * k, idesc, (i | k) != 0 ? 1u : 0u);
        }
        mma_commit(&empty_bar[s]);
      }
      mma_commit(&done_bar);
    }
    __syncwarp();
  } else {
    // ---- epilogue warps
    pdl_wait();
    pdl_trigger();
    const int quad = warp & 3;
    const int m = quad * 32 + lane;  // tile row (TMEM lane) of this thread
    const int et = threadIdx.x - 64;
    bool ok = mbar_wait_bounded(&done_bar, 0, abort_v, kWaitLimitNs);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
      raise_error(p.err, kErrWaitTimeout);
      *abort_v = 1;
    }
    tc_fence_after();
    if (et == 0) stamp(p, kTrDone);
    float* Y = reinterpret_cast<float*>(smem);  // [bpad][128] fp32, over the drained stages
    // this split's partial: to shared memory (cluster reduction, or the whole
    // sum when K is not split) or to the workspace
    float* P = (p.cluster || p.splits == 1) ? Y : p.part + (size_t)blockIdx.x * kMmaTileRows * p.bpad;
    if (ok) {
      const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16);
      for (int j = 0; j < p.bpad; j += 8) {
        float hi[8], lo[8];
        tmem_ld_8x2(trow + (uint32_t)j, trow + (uint32_t)(p.bpad + j), hi, lo);
#pragma unroll
        for (int c = 0; c < 8; ++c) P[(j + c) * kMmaTileRows + m] = hi[c] + lo[c];
      }
    }
  }
  if (p.cluster) {
    // Every split of the tile is a CTA of this cluster.  Once all partials
    // are in shared memory, CTA r adds up the sequences [r nb / S, (r+1) nb / S)
    // over the cluster (DSMEM, in split order) and runs their epilogue.
    const int S = p.splits, r = (int)cluster_rank();
    const int bb0 = r * nrows / S, bb1 = (r + 1) * nrows / S;
    float* Y = reinterpret_cast<float*>(smem);
    cluster_sync_all();  // every partial written
    if (warp >= 2) {
      const int et = threadIdx.x - 64;
      const int m4 = et & 31;
      // four sequences at a time, every remote read issued before any add
      for (int b0 = bb0 + (et >> 5); b0 < bb1; b0 += 16) {
        float4 v[4][kMaxSplits];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int q = 0; q < kMaxSplits; ++q)
            if (q < S && b0 + 4 * u < bb1)
              v[u][q] = ld_cluster_f4(Y + (size_t)(b0 + 4 * u) * kMmaTileRows + 4 * m4, (uint32_t)q);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          if (b0 + 4 * u >= bb1) break;
          float4 acc = v[u][0];
#pragma unroll
          for (int q = 1; q < kMaxSplits; ++q) {
            if (q < S) {
              acc.x += v[u][q].x;
              acc.y += v[u][q].y;
              acc.z += v[u][q].z;
              acc.w += v[u][q].w;
            }
          }
          *reinterpret_cast<float4*>(Y + (size_t)(b0 + 4 * u) * kMmaTileRows + 4 * m4) = acc;
        }
      }
    }
    cluster_sync_all();  // every remote read done: no CTA's memory is read after this
    if (warp >= 2) {
      const int et = threadIdx.x - 64;
      const int m = (warp & 3) * 32 + lane;
      if (et == 0) stamp(p, kTrReduced);
      epilogue<E, CT>(p, seq, tile, g_tile, Y, nullptr, bb0, bb1, m, et);
    }
  } else if (p.splits == 1) {
    if (warp >= 2) {
      const int et = threadIdx.x - 64;
      const int m = (warp & 3) * 32 + lane;
      named_bar_sync(kBarEpi, kEpiThreads);  // every row of Y written
      epilogue<E, CT>(p, seq, mt * tile, g_tile, Y0, nullptr, 0, nrows, m, et);
      // the CTA's further weight tiles: accumulator h into Y, then its epilogue
      for (int h = 1; h < mt; ++h) {
        named_bar_sync(kBarEpi, kEpiThreads);  // Y is free again
        if (!*abort_v) {
          const uint32_t trow = tmem + (uint32_t)(h * (p.tmem_cols / mt)) + ((uint32_t)((warp & 3) * 32) << 16);
          for (int j = 0; j < p.bpad; j += 8) {
            float hi[8], lo[8];
            tmem_ld_8x2(trow + (uint32_t)j, trow + (uint32_t)(p.bpad + j), hi, lo);
#pragma unroll
            for (int c = 0; c < 8; ++c) Y0[(j + c) * kMmaTileRows + m] = hi[c] + lo[c];
          }
        }
        named_bar_sync(kBarEpi, kEpiThreads);
        epilogue<E, CT>(p, seq, mt * tile + h, g_tile, Y0, nullptr, 0, nrows, m, et);
      }
    }
  } else if (warp >= 2) {
    const int et = threadIdx.x - 64;
    const int m = (warp & 3) * 32 + lane;
    float* Y = reinterpret_cast<float*>(smem);
    // the last CTA of the tile to finish (a ticket) adds the pieces
    const float* parts = p.part + (size_t)cta * p.splits * kMmaTileRows * p.bpad;
    __threadfence();
    named_bar_sync(kBarEpi, kEpiThreads);
    if (et == 0) {
      const uint32_t t = atomicAdd(&p.tickets[cta], 1u);
      const int last = t == (uint32_t)(p.splits - 1);
      if (last) p.tickets[cta] = 0u;  // every piece has arrived: ready for the next launch
      last_flag = last;
      stamp(p, kTrTicket);
    }
    named_bar_sync(kBarEpi, kEpiThreads);
    if (last_flag != 0) {
      __threadfence();
      epilogue<E, CT>(p, seq, tile, g_tile, Y, parts, 0, nrows, m, et);
    }
  }
  // every tensor-memory read is done before the owner frees the columns
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// [rows][cols] bf16 row-major matrix as a 2-D tensor map: boxes of 64
// columns (128 bytes) x box_rows rows, 128-byte swizzle; rows past the end
// read as zero.
bool make_bf16_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kKBlock, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct Plan {
  int splits, grid, stages, tmem_cols;
  uint32_t stage_bytes;
  size_t smem;
  bool cluster;  // the splits of a tile form a cluster (DSMEM reduction)
};

// Shape of a launch with `s` splits per tile: as many stages as fit.
Plan plan_with(int tiles, int kblocks, int bpad, int s) {
  Plan P;
  P.splits = s;
  P.grid = tiles * s;
  P.cluster = false;
  P.stage_bytes = kABytes + (uint32_t)bpad * 2u * kRowBytes;
  const int nk_max = (kblocks + s - 1) / s;
  int st = (int)(kStageBudget / P.stage_bytes);
  if (st > nk_max) st = nk_max;
  if (st > kMaxStages) st = kMaxStages;
  if (st < 1) st = 1;
  P.stages = st;
  size_t body = (size_t)st * P.stage_bytes;
  // after the pipeline drains: Y [bpad][128] fp32 and the rope table [bpad][64] float2
  const size_t y = (sizeof(float) * kMmaTileRows + sizeof(float2) * kBoxRows) * (size_t)bpad;
  if (y > body) body = y;
  P.smem = body + 1024;
  P.tmem_cols = 32;
  while (P.tmem_cols < 2 * bpad) P.tmem_cols *= 2;
  // No more CTAs on an SM than its tensor memory holds: a CTA whose
  // allocation had to wait for another's columns could wait on a cluster
  // peer that cannot start.  Enough shared memory keeps the extra CTA out.
  const size_t min_smem = kSmemPerSm / (kTmemCols / (uint32_t)P.tmem_cols + 1) + 1;
  if (P.smem < min_smem) P.smem = min_smem;
  return P;
}

// Split K so that the tiles cover the SMs once.  A launch of several chunks
// (compute-bound: hundreds of (tile, chunk) pairs) takes the split with the
// fewest K-blocks per SM over its waves, waves * ceil(kblocks / s), e.g. 80
// pairs of 64 K-blocks on 152 SMs: s = 3 (2 waves of 22) rather than 1 (64)
// or 2 (2 waves of 32).
int default_splits(int tiles, int kblocks, bool chunked) {
  const int sms = device_sm_count();
  if (chunked) {
    int best = 1;
    int64_t best_cost = INT64_MAX;
    for (int s = 1; s <= kMaxSplits && s <= kblocks; ++s) {
      if (s > 1 && s * tiles > kMmaMaxCtas) break;  // split partials and tickets are per CTA
      const int64_t waves = (int64_t)(tiles * s + sms - 1) / sms;
      const int64_t cost = waves * ((kblocks + s - 1) / s);
      if (cost < best_cost) {
        best_cost = cost;
        best = s;
      }
    }
    return best;
  }
  int s = sms / tiles;
  if (s > kMaxSplits) s = kMaxSplits;
  if (s > kblocks) s = kblocks;
  if (s * tiles > kMmaMaxCtas) s = kMmaMaxCtas / tiles;
  return s < 1 ? 1 : s;
}

cudaLaunchConfig_t launch_config(const Plan& P, cudaStream_t st, cudaLaunchAttribute (&attr)[2]) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(kMmaThreads);
  cfg.dynamicSmemBytes = P.smem;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)P.splits;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = P.cluster ? 2 : 1;
  return cfg;
}

// The launch shape of one projection: for 32 or more sequences, the most
// splits (2..8, at most the ticket path's) whose clusters all fit on the GPU
// at once, reducing through DSMEM (batch 64: 0.732 -> 0.718 ms per step,
// prefill of 512 tokens 0.832 -> 0.740 ms); otherwise, or if no cluster
// shape fits in one wave, the workspace-ticket reduction.
template <typename K>
Plan choose_plan_uncached(K kern, int tiles, int kblocks, int bpad, bool chunked, cudaStream_t st) {
  const int s0 = default_splits(tiles, kblocks, chunked);
  // Below kClusterMinBpad sequences the epilogue is short and the smaller
  // cluster grid streams weights more slowly (batch 8: qkv 15.4 -> 16.4 us).
  for (int s = s0; s >= 2 && bpad >= kClusterMinBpad; --s) {
    Plan P = plan_with(tiles, kblocks, bpad, s);
    if (P.smem > kMaxDynSmem) continue;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.smem) != cudaSuccess)
      continue;
    P.cluster = true;
    cudaLaunchAttribute attr[2];
    const cudaLaunchConfig_t cfg = launch_config(P, st, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= tiles) return P;
    cudaGetLastError();  // a refused query leaves no sticky error
  }
  return plan_with(tiles, kblocks, bpad, s0);
}

// choose_plan_uncached, remembered per kernel, device and shape; `tiles`
// counts (tile, chunk) pairs
template <typename K>
Plan choose_plan(K kern, int tiles, int kblocks, int bpad, bool chunked, cudaStream_t st) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int>, Plan> memo;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, tiles, kblocks, bpad, chunked ? 1 : 0);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) return it->second;
  }
  const Plan P = choose_plan_uncached(kern, tiles, kblocks, bpad, chunked, st);
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = P;
  return P;
}

template <int E, typename CT>
cudaError_t launch_gemm(const CUtensorMap& tw, const CUtensorMap& tg, const CUtensorMap& tx,
                        MmaParams p, const MmaSeq& seq, int tiles, cudaStream_t st) {
  auto kern = k_proj_mma<E, CT>;
  Plan P = choose_plan(kern, tiles * p.chunks, p.kblocks, p.bpad, p.chunks > 1, st);
  if (P.smem > kMaxDynSmem) return cudaErrorInvalidValue;
  // A grid of one to two CTAs per SM (the up GEMM's 160 tiles): a shallower
  // pipeline that lets two CTAs share an SM runs them all at once instead of
  // a second wave (batch 8: MLP 67 -> 53 us, batch 64: 71 -> 59 us).  Longer
  // grids (the head's 1024 tiles) keep the deep pipeline: measured faster.
  const int sms = device_sm_count();
  if (E != kEpiQkv && !P.cluster && P.grid > sms && P.grid <= 2 * sms && 2 * P.tmem_cols <= (int)kTmemCols) {
    const size_t cap = kSmemPerSm / 2 - 2048;  // two CTAs with their static and reserved shared memory
    const size_t y = (sizeof(float) * kMmaTileRows + sizeof(float2) * kBoxRows) * (size_t)p.bpad;
    const int st2 = (int)((cap - 1024) / P.stage_bytes);
    if (st2 >= 2 && y + 1024 <= cap) {
      if (st2 < P.stages) P.stages = st2;
      const size_t body = (size_t)P.stages * P.stage_bytes;
      P.smem = (body > y ? body : y) + 1024;
    }
  }
  // Grids of more than two waves of unsplit o tiles (the head's 1024): two
  // weight tiles per CTA share each activation stage, two accumulators, half
  // the CTAs, so the start-up of a CTA is paid once per 256 weight rows
  // (head at batch 8: 153 -> 145 us; at batch 64 in the decoder step 158 ->
  // 144 us).  Only with at least 4 stages: at 128 sequences (3) it was slower.
  p.mt = 1;
  if (E == kEpiO && P.splits == 1 && !P.cluster && P.grid > 2 * sms) {
    Plan Q = P;
    Q.stage_bytes = 2 * kABytes + (uint32_t)p.bpad * 2u * kRowBytes;
    int st2 = (int)(kStageBudget / Q.stage_bytes);
    if (st2 > kMaxStages) st2 = kMaxStages;
    if (st2 > p.kblocks) st2 = p.kblocks;
    const size_t y = (sizeof(float) * kMmaTileRows + sizeof(float2) * kBoxRows) * (size_t)p.bpad;
    if (st2 >= 4 && 2 * P.tmem_cols <= (int)kTmemCols) {
      Q.stages = st2;
      const size_t body = (size_t)st2 * Q.stage_bytes;
      Q.smem = (body > y ? body : y) + 1024;
      Q.tmem_cols = 2 * P.tmem_cols;
      const size_t min_smem = kSmemPerSm / (kTmemCols / (uint32_t)Q.tmem_cols + 1) + 1;  // TMEM per SM
      if (Q.smem < min_smem) Q.smem = min_smem;
      Q.grid = (tiles + 1) / 2 * p.chunks;
      if (Q.smem <= kMaxDynSmem) {
        P = Q;
        p.mt = 2;
      }
    }
  }
  p.splits = P.splits;
  p.stages = P.stages;
  p.stage_bytes = P.stage_bytes;
  p.tmem_cols = P.tmem_cols;
  p.cluster = P.cluster ? 1 : 0;
  static const bool tracing = getenv("SPARK_TRACE_MMA") != nullptr;
  if (!tracing || (size_t)P.grid * kTraceEvents > (size_t)kTraceWords) p.trace = nullptr;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = launch_config(P, st, attr);
  return cudaLaunchKernelEx(&cfg, kern, tw, tg, tx, p, seq);
}

}  // namespace

bool mma_mlp_supported(int wdtype, int hidden, int inter) {
  return wdtype == SPARK_BF16 && hidden % kKBlock == 0 && inter % 8 == 0 && tensor_map_encoder() != nullptr;
}

bool mma_projections_supported(int wdtype, int hidden, int n_q, int rotary_dim) {
  return wdtype == SPARK_BF16 && hidden % kKBlock == 0 && n_q <= kMmaTileRows &&
         (rotary_dim <= kMmaTileRows || rotary_dim == kHeadDim) && tensor_map_encoder() != nullptr;
}

// The sequences of a launch: chunks of kMmaMaxSeq (the 256 hi/lo columns of
// one MMA), padded to 8 when there is a single chunk.
struct Chunking {
  int chunks, bpad;
};
Chunking chunking(int batch) {
  Chunking c;
  c.chunks = (batch + kMmaMaxSeq - 1) / kMmaMaxSeq;
  c.bpad = c.chunks > 1 ? kMmaMaxSeq : (batch + 7) / 8 * 8;
  return c;
}

cudaError_t launch_qkv_mma(int cdtype, const float* h, const void* norm_w, const void* qkv_w,
                           const void* g_w, float* q_rot, void* kc, void* vc, float* g_out,
                           uint32_t* err, int hidden, int n_q, int n_kv, int batch, int64_t capacity,
                           int ring_capacity, int rotary_dim, double theta, float eps,
                           const int32_t* positions, const MmaWorkspace& ws, cudaStream_t st) {
  const int rows = (n_q + 2 * n_kv) * kHeadDim;
  CUtensorMap tw, tg, tx;
  const Chunking ch = chunking(batch);
  if (!make_bf16_map(&tw, qkv_w, hidden, rows, kBoxRows) || !make_bf16_map(&tg, g_w, hidden, n_q, n_q) ||
      !make_bf16_map(&tx, ws.x, hidden, (int64_t)ch.chunks * 2 * ch.bpad, 2 * ch.bpad))
    return cudaErrorInvalidValue;
  PrepArgs pa;
  for (int i = 0; i < kMaxPairs; ++i)
    pa.inv_freq[i] = i < rotary_dim / 2 ? pow(theta, -2.0 * i / (double)rotary_dim) : 0.0;
  MmaSeq seq;
  for (int b = 0; b < SPARK_MAX_BATCH; ++b) {
    pa.pos[b] = b < batch ? positions[b] : 0;
    seq.slot[b] = b < batch ? (int32_t)write_slot_of(positions[b], ring_capacity) : 0;
  }
  cudaError_t e = launch_pdl(k_prep_norm, dim3(ch.chunks * ch.bpad), dim3(kPrepThreads), 0, st, h,
                             static_cast<const __nv_bfloat16*>(norm_w), ws.x, ws.cs, hidden, batch, ch.bpad, eps,
                             rotary_dim, pa);
  if (e != cudaSuccess) return e;
  MmaParams p = {};
  p.n_main_tiles = rows / kMmaTileRows;
  p.kblocks = hidden / kKBlock;
  p.bpad = ch.bpad;
  p.nb = batch;
  p.chunks = ch.chunks;
  p.split_halves = rotary_dim == kHeadDim ? 1 : 0;
  p.g_rows = n_q;
  p.q_rot = q_rot;
  p.kc = kc;
  p.vc = vc;
  p.g_out = g_out;
  p.cs = ws.cs;
  p.n_q = n_q;
  p.n_kv = n_kv;
  p.rotary_dim = rotary_dim;
  p.capacity = capacity;
  p.hidden = hidden;
  p.part = ws.part;
  p.tickets = ws.tickets;
  p.err = err;
  p.trace = ws.trace;
  const int tiles = p.n_main_tiles + 1;
  return cdtype == SPARK_BF16 ? launch_gemm<kEpiQkv, __nv_bfloat16>(tw, tg, tx, p, seq, tiles, st)
                              : launch_gemm<kEpiQkv, float>(tw, tg, tx, p, seq, tiles, st);
}

cudaError_t launch_oproj_mma(const float* a, const float* g, const float* h, const void* o_w,
                             float* out, uint32_t* err, int hidden, int n_q, int batch,
                             const MmaWorkspace& ws, cudaStream_t st) {
  const int q_dim = n_q * kHeadDim;
  const Chunking ch = chunking(batch);
  CUtensorMap tw, tx;
  if (!make_bf16_map(&tw, o_w, q_dim, hidden, kBoxRows) ||
      !make_bf16_map(&tx, ws.x, q_dim, (int64_t)ch.chunks * 2 * ch.bpad, 2 * ch.bpad))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(k_prep_gate, dim3(ch.chunks * ch.bpad), dim3(kPrepThreads), 0, st, a, g, ws.x, q_dim,
                             n_q, batch, ch.bpad);
  if (e != cudaSuccess) return e;
  MmaParams p = {};
  p.n_main_tiles = (hidden + kMmaTileRows - 1) / kMmaTileRows;
  p.kblocks = q_dim / kKBlock;
  p.bpad = ch.bpad;
  p.nb = batch;
  p.chunks = ch.chunks;
  p.h = h;
  p.out = out;
  p.hidden = hidden;
  p.part = ws.part;
  p.tickets = ws.tickets;
  p.err = err;
  p.trace = ws.trace;
  MmaSeq seq = {};
  return launch_gemm<kEpiO, float>(tw, tw, tx, p, seq, p.n_main_tiles, st);
}

cudaError_t launch_mlp_mma(const float* h, const void* norm_w, const void* gate_w, const void* up_w,
                           const void* down_w, float* out, uint32_t* err, int hidden, int inter, int batch,
                           float eps, const MmaWorkspace& ws, __nv_bfloat16* xd, cudaStream_t st) {
  const Chunking ch = chunking(batch);
  CUtensorMap tg, tu, td, tx, txd;
  if (!make_bf16_map(&tg, gate_w, hidden, inter, kBoxRows) || !make_bf16_map(&tu, up_w, hidden, inter, kBoxRows) ||
      !make_bf16_map(&td, down_w, inter, hidden, kBoxRows) ||
      !make_bf16_map(&tx, ws.x, hidden, (int64_t)ch.chunks * 2 * ch.bpad, 2 * ch.bpad) ||
      !make_bf16_map(&txd, xd, inter, (int64_t)ch.chunks * 2 * ch.bpad, 2 * ch.bpad))
    return cudaErrorInvalidValue;
  PrepArgs pa = {};  // no rope table
  const int up_tiles = (inter + kBoxRows - 1) / kBoxRows;
  const int down_tiles = (hidden + kMmaTileRows - 1) / kMmaTileRows;
  cudaError_t e = launch_pdl(k_prep_norm, dim3(ch.chunks * ch.bpad), dim3(kPrepThreads), 0, st, h,
                             static_cast<const __nv_bfloat16*>(norm_w), ws.x, (float2*)nullptr, hidden, batch,
                             ch.bpad, eps, 0, pa);
  if (e != cudaSuccess) return e;
  MmaSeq seq = {};
  MmaParams p = {};
  p.n_main_tiles = up_tiles;
  p.kblocks = hidden / kKBlock;
  p.bpad = ch.bpad;
  p.nb = batch;
  p.chunks = ch.chunks;
  p.xd = xd;
  p.inter = inter;
  p.part = ws.part;
  p.tickets = ws.tickets;
  p.err = err;
  p.trace = ws.trace;
  e = launch_gemm<kEpiUp, float>(tg, tu, tx, p, seq, up_tiles, st);
  if (e != cudaSuccess) return e;
  MmaParams q = {};
  q.n_main_tiles = down_tiles;
  q.kblocks = (inter + kKBlock - 1) / kKBlock;  // the last block's columns past inter read as zero
  q.bpad = ch.bpad;
  q.nb = batch;
  q.chunks = ch.chunks;
  q.h = h;
  q.out = out;
  q.hidden = hidden;
  q.part = ws.part;
  q.tickets = ws.tickets;
  q.err = err;
  q.trace = ws.trace;
  return launch_gemm<kEpiO, float>(td, td, txd, q, seq, down_tiles, st);
}

cudaError_t launch_head_mma(const float* h, const void* norm_w, const void* embed, float* logits, uint32_t* err,
                            int hidden, int vocab, int batch, float eps, const MmaWorkspace& ws, cudaStream_t st) {
  const Chunking ch = chunking(batch);
  CUtensorMap te, tx;
  if (!make_bf16_map(&te, embed, hidden, vocab, kBoxRows) ||
      !make_bf16_map(&tx, ws.x, hidden, (int64_t)ch.chunks * 2 * ch.bpad, 2 * ch.bpad))
    return cudaErrorInvalidValue;
  PrepArgs pa = {};
  const int tiles = (vocab + kMmaTileRows - 1) / kMmaTileRows;
  cudaError_t e = launch_pdl(k_prep_norm, dim3(ch.chunks * ch.bpad), dim3(kPrepThreads), 0, st, h,
                             static_cast<const __nv_bfloat16*>(norm_w), ws.x, (float2*)nullptr, hidden, batch,
                             ch.bpad, eps, 0, pa);
  if (e != cudaSuccess) return e;
  MmaSeq seq = {};
  MmaParams p = {};
  p.n_main_tiles = tiles;
  p.kblocks = hidden / kKBlock;
  p.bpad = ch.bpad;
  p.nb = batch;
  p.chunks = ch.chunks;
  p.h = nullptr;  // no residual
  p.out = logits;
  p.hidden = vocab;
  p.part = ws.part;
  p.tickets = ws.tickets;
  p.err = err;
  p.trace = ws.trace;
  return launch_gemm<kEpiO, float>(te, te, tx, p, seq, tiles, st);
}

}  // namespace spark
