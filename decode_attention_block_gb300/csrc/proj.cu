// proj.cu -- the block's two weight-streaming projections, each fused with
// the small steps around it.
//
//  * qkv_rope: input RMSNorm + q_k_v_proj + g_proj + the split + per-class
//    NeoX rope + the cache-row write of k and v (turbospark-runtime 0.3.0,
//    src/families/spark/attn.rs, encode_attention_block: the fused
//    projection, the gate's projection reading the same normed x,
//    encode_split_qkv with k and v landing in their cache slots,
//    encode_rope_neox_subdim on q and on the k slot; module doc items 1-2;
//    src/families/spark/mod.rs, "One decoder layer, transcribed":
//    x = rms(h, w, 1e-6) with a plain w).
//  * oproj: the headwise sigmoid gate + o_proj + the raw residual add
//    (attn.rs: encode_sigmoid_head_gate_mul before o_proj; mod.rs:
//    encode_residual_add).
//
// Both are HBM-bound at small batch: every weight byte is read once and used
// for `nb` multiply-adds.  Each CTA (one per SM) owns an equal contiguous
// share of the weight rows and streams them with 1-D bulk copies
// (cp.async.bulk) into a pool of shared-memory stages, one row unit per
// stage; the pool holds the CTA's whole share when it fits (~200 KB at
// spark2_5's size), so every byte is requested at once, and the requests are
// issued before the kernel waits for its predecessor (programmatic dependent
// launch): the weight stream does not depend on the previous kernel.  Warps
// take units round-robin; the warp that frees a stage refills it.
//
// The rope angles' cos and sin come from the host, computed in double.
//
// The RMSNorm needs no pass before the GEMV: rms(h) scales every output of a
// row by the same 1/sqrt(mean(h^2) + eps), so the warps dot the rows with
// h * w and the scale is applied in the epilogue.
//
// qkv_rope processes rows in pairs.  For a rotated q or k head the pair is
// (i, i + r/2) -- the two rows NeoX rope mixes -- so the epilogue rotates the
// two finished dot products and writes q (fp32) or k (cache type) directly;
// v rows, rows past the rotary width and g rows are paired as neighbours.
#include <math.h>

#include "checks.h"
#include "gemv_parts.cuh"
#include "launch.h"
#include "partition.h"

namespace spark {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxPer = 8192 / 4 / kThreads;  // float4 of an activation vector per thread
// Shared memory per CTA for the activations and the weight stages (one CTA
// per SM).  Measured on GB300: a ~100 KB budget that lets the next kernel's
// CTAs co-reside gains less than the deeper pool loses.
#ifndef SPARK_GEMV_SMEM_KB
#define SPARK_GEMV_SMEM_KB 200
#endif
constexpr size_t kSmemBudget = SPARK_GEMV_SMEM_KB * 1024;
// q_k_v_proj units (row pairs) each CTA requests before the dependency wait;
// the rest go out once x is built.  Loads issued after a CTA-wide weight
// stream wait for it: with every stage requested up front, h arrived 4.3 us
// after the wait, with 6 (60 KB of 207 KB) after 2.5 us.  Swept again after
// o_proj's column path (its CTAs now leave the SMs sooner): 4 / 6 / 8 / 10 /
// 12 / 16 units give the 36-layer batch-1 step 783 / 762 / 751-754 / 753 /
// 759 / 768 us, and 8 is the best for the fp32 one-layer step too.
constexpr int kQkvPre = 8;
// o_proj rows per CTA whose residual is loaded with the activations
constexpr int kOprojHRows = 64;
// o_proj by columns (bf16 weights, every row of the share resident, up to 2 sequences):
// each thread keeps its own weight chunks' activations in registers, so the
// activation vector is read once instead of once per row pair
constexpr int kOprojColRows = 32;                 // most rows of a share
constexpr int kOprojColMaxQ = 4096;               // q_dim of the register slice
constexpr size_t kOprojEarlyBudget = 220 * 1024;  // shared memory of a CTA shaped to the free SMs


template <int NB>
struct QkvArgs {
  float2 cs[NB][kHeadDim / 2];  // (cos, sin) of the rope angle of pair i for sequence b
  int32_t pos[NB];
};

// ---------------------------------------------------------------------------
// RMSNorm + q_k_v_proj + g_proj + rope + cache write
// ---------------------------------------------------------------------------
template <typename WT, typename CT, int NB>
__global__ void __launch_bounds__(kThreads, 1)
    k_qkv_rope(const float* __restrict__ h, const WT* __restrict__ norm_w,
               const WT* __restrict__ qkv_w, const WT* __restrict__ g_w, float* __restrict__ q_rot,
               CT* __restrict__ kc, CT* __restrict__ vc, float* __restrict__ g_out, uint32_t* err,
               int hidden, int n_q, int n_kv, int nb, int64_t capacity, int ring_capacity,
               int rotary_dim, int stages, float eps, uint64_t* trace,
               const __grid_constant__ QkvArgs<NB> args) {
  constexpr int E = Chunk<WT>::kElems;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = hidden / E;
  const int xfloats = ((nchunk + 31) / 32) * 32 * E;  // one permuted activation vector
  const size_t row_bytes = (size_t)hidden * sizeof(WT);
  const size_t unit_bytes = 2 * row_bytes;
  float* xs = reinterpret_cast<float*>(smem);         // [NB][xfloats]
  unsigned char* pool = smem + sizeof(float) * NB * xfloats;  // [stages][2 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(pool + (size_t)stages * unit_bytes);
  __shared__ float red[kWarps][NB];
  __shared__ float inv_rms[NB];
  __shared__ int abort_flag;

  const int n_heads = n_q + 2 * n_kv;
  const int n_units = n_heads * (kHeadDim / 2) + n_q / 2;
  const int rows_qkv = n_heads * kHeadDim;
  const int u0 = (int)((int64_t)n_units * blockIdx.x / gridDim.x);
  const int u1 = (int)((int64_t)n_units * (blockIdx.x + 1) / gridDim.x);
  const int cnt = u1 - u0;  // this CTA's units: unit k goes to stage k % stages, warp k % nw
  const int nw = stages < kWarps ? stages : kWarps;  // warps that consume (a stage each at least)

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    abort_flag = 0;
    fence_mbar_init();
    cta_stamp(trace, 0);
  }
  __syncthreads();

  auto row_ptr = [&](int r) -> const WT* {
    return r < rows_qkv ? qkv_w + (int64_t)r * hidden : g_w + (int64_t)(r - rows_qkv) * hidden;
  };
  auto issue = [&](int k) {  // bring unit k of this CTA into stage k % stages
    const Unit un = unit_of(u0 + k, n_q, n_kv, rotary_dim);
    const int s = k % stages;
    unsigned char* dst = pool + (size_t)s * unit_bytes;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)unit_bytes);
    bulk_load(dst, row_ptr(un.row_a), (uint32_t)row_bytes, &bars[s]);
    bulk_load(dst + row_bytes, row_ptr(un.row_b), (uint32_t)row_bytes, &bars[s]);
  };

  // The weight stream does not depend on the previous kernel: request the
  // first kQkvPre stages now (each warp the units it will consume first),
  // the rest after x is built.
  auto issue_range = [&](int lo, int hi) {
    if (lane == 0 && warp < nw)
      for (int k = warp; k < hi && k < cnt; k += nw)
        if (k >= lo) issue(k);
  };
  // the norm weights first: after the wait only h is still to come
  float4 wv[kMaxPer];
  load_norm_w<WT, kThreads, kMaxPer>(norm_w, hidden, wv, threadIdx.x);
  issue_range(0, kQkvPre < stages ? kQkvPre : stages);
  __syncwarp();  // every lane waits only once its warp's requests are out
  pdl_wait();
  pdl_trigger();  // the next kernel starts only once the one before this has completed
  if (threadIdx.x == 0) cta_stamp(trace, 1);

  // activations: x = h * w (unscaled) and sum(h^2) per sequence
  float ss[NB];
  build_x_norm_w<E, NB, kThreads, kMaxPer>(h, wv, hidden, nb, xs, xfloats, ss, threadIdx.x);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const float v = warp_sum(ss[b]);
    if (lane == 0) red[warp][b] = v;
  }
  __syncthreads();
  if (threadIdx.x < NB) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += red[w][threadIdx.x];
    inv_rms[threadIdx.x] = 1.0f / sqrtf(t / (float)hidden + eps);
  }
  __syncthreads();
  if (threadIdx.x == 0) cta_stamp(trace, 2);
  issue_range(kQkvPre < stages ? kQkvPre : stages, stages);

  for (int k = warp; warp < nw && k < cnt; k += nw) {
    const int s = k % stages;
    const uint32_t parity = (uint32_t)((k / stages) & 1);
    const Unit un = unit_of(u0 + k, n_q, n_kv, rotary_dim);
    float2 acc_a[NB], acc_b[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc_a[b] = acc_b[b] = make_float2(0.f, 0.f);
    const bool ok = wait_stage(&bars[s], parity, &abort_flag, err);
    if (threadIdx.x == 0) cta_stamp(trace, k == 0 ? 3 : 4);
    if (ok) {
      const unsigned char* st = pool + (size_t)s * unit_bytes;
      row_dot2<WT, NB>(st, st + row_bytes, xs, xfloats, nchunk, acc_a, acc_b);
    }
    __syncwarp();
    // the stage is free again: refill it with the unit `stages` further on
    if (ok && lane == 0 && k + stages < cnt) issue(k + stages);
    if (!ok) continue;
    float va = 0.f, vb = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sa = warp_sum(acc_a[b].x + acc_a[b].y);
      const float sb = warp_sum(acc_b[b].x + acc_b[b].y);
      if (lane == b) {
        va = sa * inv_rms[b];
        vb = sb * inv_rms[b];
      }
    }
    if (lane < nb) {
      const int b = lane;
      if (un.pair >= 0) {
        const float2 cs = args.cs[b][un.pair];
        const float ra = va * cs.x - vb * cs.y;
        const float rb = vb * cs.x + va * cs.y;
        va = ra;
        vb = rb;
      }
      if (un.kind == kQ) {
        float* dst = q_rot + ((int64_t)b * n_q + un.head) * kHeadDim;
        dst[un.da] = va;
        dst[un.db] = vb;
      } else if (un.kind == kG) {
        g_out[(int64_t)b * n_q + un.da] = va;
        g_out[(int64_t)b * n_q + un.db] = vb;
      } else {
        const int64_t slot = write_slot_of(args.pos[b], ring_capacity);
        if (args.pos[b] < 0 || slot >= capacity) {  // rejected on the host; never write out of bounds
          if (err) atomicOr(err, kErrIndex);
        } else {
          CT* dst = (un.kind == kK ? kc : vc) + (((int64_t)b * capacity + slot) * n_kv + un.head) * kHeadDim;
          store_elem(dst + un.da, va);
          store_elem(dst + un.db, vb);
        }
      }
    }
  }
  if (trace != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) cta_stamp(trace, 5);
  }
}

// ---------------------------------------------------------------------------
// head gate + o_proj + residual
// ---------------------------------------------------------------------------

// o_proj of a share whose rows are all resident (row k in stage k, every
// row completing on one barrier), for up to two sequences.  Thread t owns
// weight chunks t + kThreads j of every row and holds their gated
// activations in registers; each row's dot product is its threads' terms
// added within the warp (warp_sums8, eight rows at a time) and then over the
// warps in warp order.  out = h + the sum, written by one thread per
// (row, sequence); h was read before any write (out may alias h).
// Measured at batch 1 against warps taking row pairs over an activation
// vector in shared memory: the work after the dependency wait 4.3 -> 2.6 us.
// A per-row barrier wait (17 waits in a row, ~0.9 us), a fully unrolled
// 32-row body and four rows per step with a branch per row were each slower
// than the row pairs.
template <typename WT, int NB, int J>
__device__ __forceinline__ void oproj_by_cols(const float* a, const float* g, const float* h,
                                              const unsigned char* pool, size_t row_bytes, uint64_t* bar,
                                              float* out, uint32_t* err, int hidden, int q_dim, int n_q, int nb,
                                              int r0, int cnt, volatile int* abort_flag, float* hs,
                                              uint64_t* trace) {
  constexpr int E = Chunk<WT>::kElems;
  constexpr int Q4 = E / 4;  // float4s of a chunk's activations
  constexpr int R = 8;       // rows per step
  __shared__ float red[kWarps][kOprojColRows * NB];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = q_dim / E;
  pdl_wait();
  pdl_trigger();  // the next kernel starts only once the one before this has completed
  if (threadIdx.x == 0) cta_stamp(trace, 1);
  // every load first: the residual rows, the attention output and its gates
  const int hk = threadIdx.x / NB, hb = threadIdx.x - hk * NB;
  float hv = 0.f;
  if (hk < cnt && hb < nb) hv = __ldcg(h + (int64_t)hb * hidden + r0 + hk);
  float4 x[NB][J][Q4];
  float gv[NB][J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    const int c = threadIdx.x + j * kThreads;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const bool live = c < nchunk && b < nb;
#pragma unroll
      for (int q = 0; q < Q4; ++q)
        x[b][j][q] = live ? __ldcg(reinterpret_cast<const float4*>(a + (int64_t)b * q_dim + c * E) + q)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
      gv[b][j] = live ? __ldcg(g + (int64_t)b * n_q + c * E / kHeadDim) : 0.f;
    }
  }
  if (hk < cnt && hb < nb) hs[hk * NB + hb] = hv;
  // a * sigmoid(g), one gate scalar per head (a chunk never straddles heads)
#pragma unroll
  for (int j = 0; j < J; ++j)
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sg = 1.0f / (1.0f + expf(-gv[b][j]));
#pragma unroll
      for (int q = 0; q < Q4; ++q)
        x[b][j][q] = make_float4(x[b][j][q].x * sg, x[b][j][q].y * sg, x[b][j][q].z * sg, x[b][j][q].w * sg);
    }
  if (threadIdx.x == 0) cta_stamp(trace, 2);
  const bool ok = __all_sync(0xffffffffu, wait_stage(bar, 0, abort_flag, err));  // every row (one barrier)
  if (threadIdx.x == 0) cta_stamp(trace, 3);
  // eight rows per step, their loads all issued before any use (a slot past
  // the share loads nothing and adds zero)
#pragma unroll 1
  for (int k0 = 0; ok && k0 < cnt; k0 += R) {
    uint4 w[R][J];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const bool live = k0 + i < cnt;
      const int k = live ? k0 + i : cnt - 1;
#pragma unroll
      for (int j = 0; j < J; ++j) {
        const int c = threadIdx.x + j * kThreads;
        w[i][j] = live && c < nchunk
                      ? *reinterpret_cast<const uint4*>(pool + (size_t)k * row_bytes + (size_t)c * 16)
                      : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float v[R];
#pragma unroll
      for (int i = 0; i < R; ++i) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < J; ++j) dot_chunk_reg<WT>(w[i][j], x[b][j], acc);
        v[i] = k0 + i < cnt ? acc.x + acc.y : 0.f;
      }
      warp_sums8(v);
      const int k = k0 + (lane >> 2);
      if ((lane & 3) == 0 && k < cnt) red[warp][k * NB + b] = v[0];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) cta_stamp(trace, 4);
  if (threadIdx.x < cnt * NB && ok && !*abort_flag) {
    const int k = threadIdx.x / NB, b = threadIdx.x - k * NB;
    if (b < nb) {
      float sum = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sum += red[w][threadIdx.x];
      out[(int64_t)b * hidden + r0 + k] = hs[threadIdx.x] + sum;
    }
  }
  if (trace != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) cta_stamp(trace, 5);
  }
}

template <typename WT, int NB>
__global__ void __launch_bounds__(kThreads, 1)
    k_oproj(const float* __restrict__ a, const float* __restrict__ g, const float* h,
            const WT* __restrict__ o_w, float* out, uint32_t* err, int hidden, int q_dim, int n_q,
            int nb, int stages, int early, int early_rows, uint64_t* trace) {
  constexpr int E = Chunk<WT>::kElems;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = q_dim / E;
  const int xfloats = ((nchunk + 31) / 32) * 32 * E;
  const size_t row_bytes = (size_t)q_dim * sizeof(WT);
  float* xs = reinterpret_cast<float*>(smem);  // [NB][xfloats]
  unsigned char* pool = smem + sizeof(float) * NB * xfloats;
  uint64_t* bars = reinterpret_cast<uint64_t*>(pool + (size_t)stages * row_bytes);
  __shared__ int abort_flag;
  __shared__ float hs[kOprojHRows * NB];  // the residual rows of the share, loaded with the activations

  int r0, r1;
  oproj_share(hidden, gridDim.x, early, early_rows, blockIdx.x, r0, r1);
  const int cnt = r1 - r0;
  const int nw = stages < kWarps ? stages : kWarps;
  // every row of the share resident: warps take rows in pairs, one pass over
  // the activations for both (at batch 1 the fp32 activation vector, twice the
  // bytes of a bf16 row, otherwise dominates the shared-memory reads)
  const bool pairs = stages >= cnt;
  const bool h_smem = cnt <= kOprojHRows;
  // or, for up to two sequences, by columns with the activations in registers
  constexpr int kColJ = kOprojColMaxQ / E / kThreads;  // chunks of a row per thread
  const bool by_cols = NB <= 2 && sizeof(WT) == 2 && pairs && cnt <= kOprojColRows && nchunk <= kColJ * kThreads;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    abort_flag = 0;
    fence_mbar_init();
    if (by_cols) mbar_arrive_expect_tx(&bars[0], (uint32_t)((size_t)cnt * row_bytes));
    cta_stamp(trace, 0);
  }
  __syncthreads();

  auto issue = [&](int k) {
    const int s = k % stages;
    if (by_cols) {  // every row completes on barrier 0, which expects them all
      bulk_load(pool + (size_t)s * row_bytes, o_w + (int64_t)(r0 + k) * q_dim, (uint32_t)row_bytes, &bars[0]);
      return;
    }
    mbar_arrive_expect_tx(&bars[s], (uint32_t)row_bytes);
    bulk_load(pool + (size_t)s * row_bytes, o_w + (int64_t)(r0 + k) * q_dim, (uint32_t)row_bytes,
              &bars[s]);
  };
  if (lane == 0 && warp < nw)
    for (int k = warp; k < stages && k < cnt; k += nw) issue(k);
  __syncwarp();  // every lane waits only once its warp's requests are out
  if constexpr (NB <= 2 && sizeof(WT) == 2) {  // fp32 rows never all fit beside each other at batch 1
    if (by_cols) {  // waits for the previous kernel itself
      oproj_by_cols<WT, NB, kColJ>(a, g, h, pool, row_bytes, &bars[0], out, err, hidden, q_dim, n_q, nb, r0, cnt,
                                   &abort_flag, hs, trace);
      return;
    }
  }
  pdl_wait();
  pdl_trigger();  // the next kernel starts only once the one before this has completed
  if (threadIdx.x == 0) cta_stamp(trace, 1);


  // the residual rows, requested with the activations so that the epilogue
  // needs no round trip of its own (out may alias h: every element is read
  // here, before this CTA writes it)
  const int hk = threadIdx.x / NB, hb = threadIdx.x - hk * NB;
  float hv = 0.f;
  if (h_smem && hk < cnt && hb < nb) hv = h[(int64_t)hb * hidden + r0 + hk];
  // gated attention output: a * sigmoid(g), one gate scalar per head
  build_x_gated<E, NB, kThreads, kMaxPer>(a, g, q_dim, n_q, nb, xs, xfloats, threadIdx.x);
  if (h_smem && hk < cnt && hb < nb) hs[hk * NB + hb] = hv;
  __syncthreads();
  if (threadIdx.x == 0) cta_stamp(trace, 2);

  auto finish = [&](int k, const float2 (&acc)[NB]) {  // out = h + the row's dot product
    float v = 0.f;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float sb = warp_sum(acc[b].x + acc[b].y);
      if (lane == b) v = sb;
    }
    if (lane < nb) {
      const int64_t idx = (int64_t)lane * hidden + r0 + k;
      out[idx] = (h_smem ? hs[k * NB + lane] : h[idx]) + v;  // read and written by the same thread
    }
  };
  if (pairs) {
    for (int p = warp; p < (cnt + 1) / 2; p += kWarps) {
      const int k0 = 2 * p, k1 = 2 * p + 1;
      float2 acc0[NB], acc1[NB];
#pragma unroll
      for (int b = 0; b < NB; ++b) acc0[b] = acc1[b] = make_float2(0.f, 0.f);
      bool ok = wait_stage(&bars[k0], 0, &abort_flag, err);
      if (k1 < cnt) ok = ok && wait_stage(&bars[k1], 0, &abort_flag, err);
      if (threadIdx.x == 0) cta_stamp(trace, p == 0 ? 3 : 4);
      if (!ok) continue;
      if (k1 < cnt) {
        row_dot2<WT, NB>(pool + (size_t)k0 * row_bytes, pool + (size_t)k1 * row_bytes, xs, xfloats, nchunk, acc0,
                         acc1);
        finish(k0, acc0);
        finish(k1, acc1);
      } else {
        row_dot<WT, NB>(pool + (size_t)k0 * row_bytes, xs, xfloats, nchunk, acc0);
        finish(k0, acc0);
      }
    }
  }
  for (int k = warp; !pairs && warp < nw && k < cnt; k += nw) {
    const int s = k % stages;
    const uint32_t parity = (uint32_t)((k / stages) & 1);
    float2 acc[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b] = make_float2(0.f, 0.f);
    const bool ok = wait_stage(&bars[s], parity, &abort_flag, err);
    if (threadIdx.x == 0) cta_stamp(trace, k == 0 ? 3 : 4);
    if (ok) row_dot<WT, NB>(pool + (size_t)s * row_bytes, xs, xfloats, nchunk, acc);
    __syncwarp();
    if (ok && lane == 0 && k + stages < cnt) issue(k + stages);
    if (!ok) continue;
    finish(k, acc);
  }
  if (trace != nullptr) {
    __syncthreads();
    if (threadIdx.x == 0) cta_stamp(trace, 5);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

int stages_for(size_t unit_bytes, size_t x_bytes, int max_units) {
  return gemv_stages(kSmemBudget, kWarps, unit_bytes, x_bytes, max_units);
}

template <typename WT>
size_t xbytes(int cols, int nb) {
  return gemv_xbytes<WT>(cols, nb);
}

template <typename WT, typename CT, int NB>
cudaError_t qkv_launch(const float* h, const void* norm_w, const void* qkv_w, const void* g_w,
                       float* q_rot, void* kc, void* vc, float* g_out, uint32_t* err, int hidden,
                       int n_q, int n_kv, int nb, int64_t capacity, int ring_capacity,
                       int rotary_dim, double theta, float eps, const int32_t* positions,
                       cudaStream_t st) {
  QkvArgs<NB> args;
  checks::fill_rope_table(&args.cs[0][0], kHeadDim / 2, nb, positions, rotary_dim, theta);
  for (int b = 0; b < NB; ++b) args.pos[b] = b < nb ? positions[b] : 0;
  const size_t row_bytes = (size_t)hidden * sizeof(WT);
  const size_t xb = xbytes<WT>(hidden, NB);
  const int n_units = (n_q + 2 * n_kv) * (kHeadDim / 2) + n_q / 2;
  int grid = device_sm_count();
  if (grid > n_units) grid = n_units;
  const int stages = stages_for(2 * row_bytes, xb, (n_units + grid - 1) / grid);
  if (stages == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = xb + (size_t)stages * (2 * row_bytes + 8);
  auto kern = k_qkv_rope<WT, CT, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, h, (const WT*)norm_w,
                    (const WT*)qkv_w, (const WT*)g_w, q_rot, (CT*)kc, (CT*)vc, g_out, err, hidden,
                    n_q, n_kv, nb, capacity, ring_capacity, rotary_dim, stages, eps, layer_trace(0), args);
}

template <typename WT, typename CT>
cudaError_t qkv_chunk(int nb, const float* h, const void* norm_w, const void* qkv_w,
                      const void* g_w, float* q_rot, void* kc, void* vc, float* g_out,
                      uint32_t* err, int hidden, int n_q, int n_kv, int64_t capacity,
                      int ring_capacity, int rotary_dim, double theta, float eps,
                      const int32_t* positions, cudaStream_t st) {
#define SPARK_QKV(NBV)                                                                           \
  return qkv_launch<WT, CT, NBV>(h, norm_w, qkv_w, g_w, q_rot, kc, vc, g_out, err, hidden, n_q, \
                                 n_kv, nb, capacity, ring_capacity, rotary_dim, theta, eps,     \
                                 positions, st)
  if (nb == 1) SPARK_QKV(1);
  if (nb == 2) SPARK_QKV(2);
  SPARK_QKV(4);
#undef SPARK_QKV
}

// free_sms > 0: SMs the kernel before this one leaves free while it runs (the
// rest are held by its CTAs until it ends).  A CTA that starts on one of them
// requests its whole share before its dependency wait; one that must wait for
// an SM streams its share after that kernel ends.  So for one sequence the
// grid is cut to the free SMs when they can hold every row, and otherwise the
// CTAs that start at once take as many rows as fit and the others share the
// rest (the per-CTA timeline shows CTAs dispatched in index order; the split
// is correct whatever the order).  Measured at batch 1, with the column
// path: the 36-layer step 798 -> 792 us, the two-layer step 46.4 -> 45.6 us.
template <typename WT, int NB>
cudaError_t oproj_launch(const float* a, const float* g, const float* h, const void* o_w,
                         float* out, uint32_t* err, int hidden, int n_q, int nb, int free_sms, cudaStream_t st) {
  const int q_dim = n_q * kHeadDim;
  const size_t row_bytes = (size_t)q_dim * sizeof(WT);
  const size_t xb = xbytes<WT>(q_dim, NB);
  int grid = device_sm_count();
  if (grid > hidden) grid = hidden;
  int early = 0, early_rows = 0, max_share = (hidden + grid - 1) / grid;
  size_t budget = kSmemBudget;
  if (NB == 1 && free_sms > 0 && free_sms < grid && xb < kOprojEarlyBudget) {
    int cap = (int)((kOprojEarlyBudget - xb) / (row_bytes + 8));  // rows that fit, all resident
    if (cap > kOprojColRows) cap = kOprojColRows;
    if (cap >= max_share) {
      if ((int64_t)free_sms * cap >= hidden) {
        grid = free_sms;
        max_share = (hidden + grid - 1) / grid;
      } else {
        early = free_sms;
        early_rows = cap;
        const int late = grid - early, rest = hidden - early * early_rows;
        max_share = cap > (rest + late - 1) / late ? cap : (rest + late - 1) / late;
      }
      budget = kOprojEarlyBudget;
    }
  }
  const int stages = gemv_stages(budget, kWarps, row_bytes, xb, max_share);
  if (stages == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = xb + (size_t)stages * (row_bytes + 8);
  auto kern = k_oproj<WT, NB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, a, g, h, (const WT*)o_w, out, err,
                    hidden, q_dim, n_q, nb, stages, early, early_rows, layer_trace(2));
}

template <typename WT>
cudaError_t oproj_chunk(int nb, const float* a, const float* g, const float* h, const void* o_w,
                        float* out, uint32_t* err, int hidden, int n_q, int free_sms, cudaStream_t st) {
  if (nb == 1) return oproj_launch<WT, 1>(a, g, h, o_w, out, err, hidden, n_q, nb, free_sms, st);
  if (nb == 2) return oproj_launch<WT, 2>(a, g, h, o_w, out, err, hidden, n_q, nb, -1, st);
  return oproj_launch<WT, 4>(a, g, h, o_w, out, err, hidden, n_q, nb, -1, st);
}

constexpr int kMaxChunk = 4;

}  // namespace

cudaError_t launch_qkv_rope(int wdtype, int cdtype, const float* h, const void* norm_w,
                            const void* qkv_w, const void* g_w, float* q_rot, void* kc, void* vc,
                            float* g_out, uint32_t* err, int hidden, int n_q, int n_kv, int batch,
                            int64_t capacity, int ring_capacity, int rotary_dim, double theta,
                            float eps, const int32_t* positions, cudaStream_t st) {
  const size_t ce = cdtype == SPARK_BF16 ? 2 : 4;
  for (int b0 = 0; b0 < batch; b0 += kMaxChunk) {
    const int nb = batch - b0 < kMaxChunk ? batch - b0 : kMaxChunk;
    const float* hb = h + (int64_t)b0 * hidden;
    float* qb = q_rot + (int64_t)b0 * n_q * kHeadDim;
    float* gb = g_out + (int64_t)b0 * n_q;
    const int64_t coff = (int64_t)b0 * capacity * n_kv * kHeadDim * ce;
    void* kb = static_cast<unsigned char*>(kc) + coff;
    void* vb = static_cast<unsigned char*>(vc) + coff;
    cudaError_t e;
    if (wdtype == SPARK_BF16 && cdtype == SPARK_BF16)
      e = qkv_chunk<__nv_bfloat16, __nv_bfloat16>(nb, hb, norm_w, qkv_w, g_w, qb, kb, vb, gb, err,
                                                  hidden, n_q, n_kv, capacity, ring_capacity,
                                                  rotary_dim, theta, eps, positions + b0, st);
    else if (wdtype == SPARK_BF16)
      e = qkv_chunk<__nv_bfloat16, float>(nb, hb, norm_w, qkv_w, g_w, qb, kb, vb, gb, err, hidden,
                                          n_q, n_kv, capacity, ring_capacity, rotary_dim, theta,
                                          eps, positions + b0, st);
    else if (cdtype == SPARK_BF16)
      e = qkv_chunk<float, __nv_bfloat16>(nb, hb, norm_w, qkv_w, g_w, qb, kb, vb, gb, err, hidden,
                                          n_q, n_kv, capacity, ring_capacity, rotary_dim, theta,
                                          eps, positions + b0, st);
    else
      e = qkv_chunk<float, float>(nb, hb, norm_w, qkv_w, g_w, qb, kb, vb, gb, err, hidden, n_q,
                                  n_kv, capacity, ring_capacity, rotary_dim, theta, eps,
                                  positions + b0, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_oproj(int wdtype, const float* a, const float* g, const float* h,
                         const void* o_w, float* out, uint32_t* err, int hidden, int n_q, int batch,
                         cudaStream_t st, int free_sms) {
  const int q_dim = n_q * kHeadDim;
  for (int b0 = 0; b0 < batch; b0 += kMaxChunk) {
    const int nb = batch - b0 < kMaxChunk ? batch - b0 : kMaxChunk;
    const float* ab = a + (int64_t)b0 * q_dim;
    const float* gb = g + (int64_t)b0 * n_q;
    const float* hb = h + (int64_t)b0 * hidden;
    float* ob = out + (int64_t)b0 * hidden;
    cudaError_t e = wdtype == SPARK_BF16
                        ? oproj_chunk<__nv_bfloat16>(nb, ab, gb, hb, o_w, ob, err, hidden, n_q,
                                                     batch == 1 ? free_sms : -1, st)
                        : oproj_chunk<float>(nb, ab, gb, hb, o_w, ob, err, hidden, n_q,
                                             batch == 1 ? free_sms : -1, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace spark
