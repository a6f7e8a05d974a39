// noalloc.cu -- the split-K attention for callers that cannot allocate device
// memory.
//
// The attention kernel needs scratch memory besides its inputs and outputs:
// one partial result (m, l, o) per piece of work a CTA finishes, the merge
// tickets that find the last CTA of each (sequence, KV head) group, and an
// error word.  spark_dbg_attention takes it from a workspace the caller
// allocates.  Some callers cannot allocate at all: code that runs while a
// stream is being captured into a CUDA graph (an allocation is not a
// capturable operation), hosts whose own memory pool owns every byte of the
// device and forbids allocations by plug-ins, and latency-critical loops that
// must not allocate mid-run.  For them, this file keeps the scratch in a
// fixed array of device memory inside the library and launches the very same
// kernel on it.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (about 2 MiB) until the process exits.  In host code its
// name is only a host-side stand-in, not a device address: the address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, and passed to the kernel.
#include <math.h>

#include <mutex>

#include "launch.h"

namespace spark {
namespace {

constexpr int kStaticGroups = 256;  // batch * n_kv a call may have
constexpr int kStaticCtas = 256;    // CTAs a call may use
constexpr int kMinRowsPerCta = 64;
constexpr size_t kErrOff = 0;
constexpr size_t kCounterOff = 256;
constexpr size_t kPartOff = kCounterOff + sizeof(uint32_t) * kStaticGroups;  // 1280, 256-aligned
constexpr size_t kScratchBytes =
    kPartOff + sizeof(float) * (size_t)(kStaticCtas + kStaticGroups) * kPartFloats;
static_assert(kPartOff % 256 == 0, "partials must stay aligned");

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device, looked up once.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The same argument rules as spark_dbg_attention: every row the kernel reads
// lies inside the cache buffers.
int check_args(const spark_geom* g, const float* q_rot, const spark_kv_layer* kv, int32_t cls,
               const int32_t* positions, int32_t batch, const float* a) {
  if (!g || !kv || !positions || !q_rot || !a) return SPARK_ERR_INVALID_ARG;
  if (g->head_dim != kHeadDim || g->n_kv < 1 || g->n_kv > 8 || g->n_q != kGroup * g->n_kv)
    return SPARK_ERR_UNSUPPORTED;
  if (g->window < 1 || !isfinite(g->scale)) return SPARK_ERR_INVALID_ARG;
  if (batch < 1 || batch > SPARK_MAX_BATCH) return SPARK_ERR_INVALID_ARG;
  if (cls != SPARK_FULL && cls != SPARK_SLIDING) return SPARK_ERR_INVALID_ARG;
  if (!aligned16(q_rot) || !aligned16(a)) return SPARK_ERR_INVALID_ARG;
  if (!kv->k || !kv->v || !aligned16(kv->k) || !aligned16(kv->v)) return SPARK_ERR_INVALID_ARG;
  if (kv->dtype != SPARK_F32 && kv->dtype != SPARK_BF16) return SPARK_ERR_INVALID_ARG;
  if (kv->capacity < 1 || kv->ring_capacity < 0) return SPARK_ERR_INVALID_ARG;
  if (kv->ring_capacity > 0) {
    if (cls == SPARK_FULL) return SPARK_ERR_BAD_RING;
    if (kv->ring_capacity > kv->capacity) return SPARK_ERR_INVALID_ARG;
    if (kv->ring_capacity < g->window) return SPARK_ERR_BAD_RING;
  }
  if ((int64_t)batch * kv->capacity >= ((int64_t)1 << 31)) return SPARK_ERR_UNSUPPORTED;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t p = positions[b];
    if (p < 0 || p >= INT32_MAX - 1) return SPARK_ERR_POSITION;
    if (kv->ring_capacity == 0 && (int64_t)p >= kv->capacity) return SPARK_ERR_POSITION;
  }
  return SPARK_OK;
}

}  // namespace
}  // namespace spark

using namespace spark;

extern "C" int spark_dbg_attention_noalloc(const spark_geom* g, const float* q_rot,
                                           const spark_kv_layer* kv, int32_t layer_class,
                                           const int32_t* positions, int32_t batch, float* a,
                                           void* stream) {
  int s = check_args(g, q_rot, kv, layer_class, positions, batch, a);
  if (s != SPARK_OK) return s;
  if (batch * g->n_kv > kStaticGroups) return SPARK_ERR_WORKSPACE;  // beyond the fixed scratch
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return SPARK_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  // the error word and the merge tickets must start at zero
  if (cudaMemsetAsync(scratch, 0, kPartOff, st) != cudaSuccess) return SPARK_ERR_CUDA;
  const bool full = layer_class == SPARK_FULL;
  int64_t rows = 0;
  for (int32_t b = 0; b < batch; ++b) rows += window_of(positions[b], full, g->window, kv->ring_capacity).rows;
  int64_t ctas = ((int64_t)g->n_kv * rows + kMinRowsPerCta - 1) / kMinRowsPerCta;
  if (ctas > device_sm_count()) ctas = device_sm_count();
  if (ctas > kStaticCtas) ctas = kStaticCtas;
  if (ctas < 1) ctas = 1;
  const cudaError_t e = launch_attention(
      kv->dtype, q_rot, kv->k, kv->v, g->n_kv, kv->capacity, kv->ring_capacity, full, g->window,
      g->scale, positions, batch, a, reinterpret_cast<float*>(scratch + kPartOff),
      reinterpret_cast<uint32_t*>(scratch + kCounterOff),
      reinterpret_cast<uint32_t*>(scratch + kErrOff), (int)ctas, nullptr, 0, st);
  return e == cudaSuccess ? SPARK_OK : SPARK_ERR_CUDA;
}
