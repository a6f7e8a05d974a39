// common.cuh -- device helpers shared by the block's kernels: inline PTX for
// mbarriers, TMA tensor loads, packed fp32x2 FMA and bounded waits; the
// per-sequence window arithmetic shared by host and device; the workspace
// layout.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/spark_attn.h"

namespace spark {

constexpr int kHeadDim = 256;        // the only head_dim the kernels are built for
constexpr int kGroup = 4;            // query heads per KV head
constexpr int kMaxAttnCtas = 1024;   // partial-result slots reserved for CTAs
constexpr int kPartFloats = 2 * kGroup + kGroup * kHeadDim;  // m[4], l[4], o[4][256]

// tensor-core projections (mma.cu): sequences per launch, CTAs a launch may use
constexpr int kMmaMaxSeq = 128;
constexpr int kMmaMaxCtas = 256;
constexpr int kMmaTileRows = 128;

// every bounded wait in the kernels gives up after this long
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// device error word bits
constexpr uint32_t kErrWaitTimeout = 1u;
constexpr uint32_t kErrIndex = 2u;

// ---------------------------------------------------------------------------
// window / ring arithmetic (attn.rs, encode_attention_block: the window set-up;
// the ring only addresses rows once seq_len exceeds its capacity)
// ---------------------------------------------------------------------------
struct Window {
  int64_t kv_start;   // first logical position read
  int64_t rows;       // number of positions read = seq_len - kv_start
  int64_t first_slot; // cache row of position kv_start
  int64_t len_a;      // rows from first_slot upwards before the ring wraps to row 0
};

__host__ __device__ inline Window window_of(int64_t position, bool full, int64_t window,
                                            int64_t ring_capacity) {
  Window w;
  const int64_t seq_len = position + 1;
  if (full) {
    w.kv_start = 0;
  } else {
    w.kv_start = seq_len > window ? seq_len - window : 0;
  }
  w.rows = seq_len - w.kv_start;
  const bool ring_active = !full && ring_capacity > 0 && seq_len > ring_capacity;
  if (ring_active) {
    w.first_slot = w.kv_start % ring_capacity;
    const int64_t to_end = ring_capacity - w.first_slot;
    w.len_a = w.rows < to_end ? w.rows : to_end;
  } else {
    w.first_slot = w.kv_start;
    w.len_a = w.rows;
  }
  return w;
}

// cache row that receives the token at `position` (kv_write.rs, kv_write_target)
__host__ __device__ inline int64_t write_slot_of(int64_t position, int64_t ring_capacity) {
  return ring_capacity > 0 ? position % ring_capacity : position;
}

// ---------------------------------------------------------------------------
// workspace layout (host computes, kernels receive the pieces as pointers)
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t err = 0;       // uint32 error word
  size_t gbar = 0;      // uint32 [2] grid barrier of the persistent decode kernel
  size_t counters = 0;  // uint32 [batch * n_kv] merge tickets
  size_t g = 0;         // f32 [batch][n_q] gate logits
  size_t q_rot = 0;     // f32 [batch][q_dim] rotated queries
  size_t a = 0;         // f32 [batch][q_dim] attention output
  size_t hbuf = 0;      // f32 [2][batch][hidden] residual stream between layers
  size_t part = 0;      // f32 [kMaxAttnCtas + batch * n_kv][kPartFloats]
  size_t mx = 0;        // bf16 [chunk][2][bpad][max(hidden, q_dim)] projection inputs (hi, lo)
  size_t mcs = 0;       // f32x2 [batch][head_dim / 2] rope (cos, sin) of each sequence
  size_t mpart = 0;     // f32 [kMmaMaxCtas][kMmaTileRows][min(batch, kMmaMaxSeq) rounded to 8]
  size_t mtick = 0;     // uint32 [kMmaMaxCtas] split-K tickets of the projection tiles
  size_t stage = 0;     // [2][batch][n_kv][head_dim] in the cache type (room for f32): a chunk's k, v rows
  size_t trace = 0;     // u64 [kTraceWords] phase timestamps of the persistent kernel (opt-in)
  size_t total = 0;
};

constexpr int kTraceWords = 8192;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Padded sequences of the tensor-core projections' activation rows: chunks
// of kMmaMaxSeq, or one chunk rounded up to 8.
inline size_t mma_padded_rows(int batch) {
  return batch > kMmaMaxSeq ? (size_t)(batch + kMmaMaxSeq - 1) / kMmaMaxSeq * kMmaMaxSeq
                            : (size_t)(batch + 7) / 8 * 8;
}

inline WsLayout ws_layout(int hidden, int n_q, int n_kv, int batch) {
  WsLayout L;
  L.err = 0;
  L.gbar = 64;
  size_t off = 256;
  L.counters = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)batch * n_kv, 256);
  L.g = off;
  off = align_up(off + sizeof(float) * (size_t)batch * n_q, 256);
  L.q_rot = off;
  off = align_up(off + sizeof(float) * (size_t)batch * n_q * kHeadDim, 256);
  L.a = off;
  off = align_up(off + sizeof(float) * (size_t)batch * n_q * kHeadDim, 256);
  L.hbuf = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)batch * hidden, 256);
  L.part = off;
  off = align_up(off + sizeof(float) * (size_t)(kMaxAttnCtas + (size_t)batch * n_kv) * kPartFloats, 256);
  const size_t kmax = (size_t)(hidden > n_q * kHeadDim ? hidden : n_q * kHeadDim);
  const size_t bpad = (size_t)((batch < kMmaMaxSeq ? batch : kMmaMaxSeq) + 7) / 8 * 8;
  L.mx = off;
  off = align_up(off + 2 * 2 * mma_padded_rows(batch) * kmax, 256);
  L.mcs = off;
  off = align_up(off + sizeof(float) * (size_t)batch * kHeadDim, 256);
  L.mpart = off;
  off = align_up(off + sizeof(float) * (size_t)kMmaMaxCtas * kMmaTileRows * bpad, 256);
  L.mtick = off;
  off = align_up(off + sizeof(uint32_t) * kMmaMaxCtas, 256);
  L.stage = off;
  off = align_up(off + sizeof(float) * 2 * (size_t)batch * n_kv * kHeadDim, 256);
  L.trace = off;
  off = align_up(off + sizeof(uint64_t) * kTraceWords, 256);
  L.total = off;
  return L;
}

// Workspace of the MLP half of a layer and of the head (spark_mlp_decode,
// spark_head_logits); the error word sits at offset 0 as in WsLayout, and the
// tickets right after it, at an offset that does not depend on the sizes: a
// workspace sized for one intermediate size serves the head too, and neither
// call's partial results land on the other's tickets.
struct MlpWsLayout {
  size_t err = 0;    // uint32 error word
  size_t mtick = 0;  // uint32 [kMmaMaxCtas] split-K tickets
  size_t m = 0;      // f32 [batch][inter] GELU products (GEMV path)
  size_t mx = 0;     // bf16 [chunk][2][bpad][hidden] normed activation rows (hi, lo)
  size_t md = 0;     // bf16 [chunk][2][bpad][inter] GELU product rows (hi, lo)
  size_t mpart = 0;  // f32 [kMmaMaxCtas][kMmaTileRows][bpad] split-K partials
  size_t trace = 0;  // u64 [kTraceWords] opt-in phase stamps
  size_t total = 0;
};

inline MlpWsLayout mlp_ws_layout(int hidden, int inter, int batch) {
  MlpWsLayout L;
  const size_t bpad = (size_t)((batch < kMmaMaxSeq ? batch : kMmaMaxSeq) + 7) / 8 * 8;
  L.mtick = 256;
  size_t off = align_up(L.mtick + sizeof(uint32_t) * kMmaMaxCtas, 256);
  L.m = off;
  off = align_up(off + sizeof(float) * (size_t)batch * inter, 256);
  L.mx = off;
  off = align_up(off + 2 * 2 * mma_padded_rows(batch) * (size_t)hidden, 256);
  L.md = off;
  off = align_up(off + 2 * 2 * mma_padded_rows(batch) * (size_t)inter, 256);
  L.mpart = off;
  off = align_up(off + sizeof(float) * (size_t)kMmaMaxCtas * kMmaTileRows * bpad, 256);
  L.trace = off;
  off = align_up(off + sizeof(uint64_t) * kTraceWords, 256);
  L.total = off;
  return L;
}

// Launch with programmatic dependent launch allowed: the kernel may start
// while its predecessor in the stream finishes; it calls pdl_wait() before
// touching anything the predecessor writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, at most `limit_ns`.  Returns
// false (and leaves the wait) if the time runs out or if another thread of the
// block raised `*abort`.  Every wait in these kernels goes through here, so no
// thread can spin forever.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

// 4-D tiled TMA load global -> shared, completing on `bar` (byte count).
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 2-D tiled TMA load global -> shared, completing on `bar` (byte count).
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// 1-D bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Hint: bring `bytes` (multiple of 16) of global memory into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

// Hint: bring one tile of a tensor map into L2.
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (a no-op without PDL) ...
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// ... and let the next grid in the stream start launching its prologue.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// order this thread's earlier generic-proxy view of global memory before its
// later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// d = a * b + c on two fp32 lanes at once (Blackwell packed FFMA2)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// bf16 pair packed in one 32-bit word -> two fp32 (exact widening)
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// 16-byte load of data read exactly once: not allocated in L1
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Opt-in timeline of the per-layer kernels: slot `ev` of this CTA's eight
// stamps (CTAs past kTraceCtas are not traced).
constexpr int kTraceCtas = 160;
constexpr int kTraceEvs = 8;
__device__ __forceinline__ void cta_stamp(uint64_t* trace, int ev) {
  if (trace != nullptr && blockIdx.x < kTraceCtas) trace[blockIdx.x * kTraceEvs + ev] = global_timer_ns();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

#endif  // __CUDACC__

}  // namespace spark
