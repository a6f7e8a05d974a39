// noalloc.cu -- the split-K attention for callers that cannot allocate device
// memory.
//
// The attention kernel needs scratch memory besides its inputs and outputs:
// one partial result (m, l, o) per piece of work a CTA finishes, the merge
// tickets that find the last CTA of each (sequence, KV head) group, and an
// error word.  spark_dbg_attention takes it from a workspace the caller
// allocates.  Some callers cannot allocate at all: hosts whose own memory
// pool owns every byte of the device and forbids allocations by plug-ins,
// and latency-critical loops that must not allocate mid-run.  For them, this
// file keeps the scratch in a fixed array of device memory inside the
// library and launches the very same kernel on it.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (about 2.4 MiB) until the process exits.  In host code its
// name is only a host-side stand-in, not a device address: the address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, and passed to the kernel.  The error word in the array collects
// the kernels' failure bits across calls until
// spark_dbg_attention_noalloc_error_word reads and clears it.
#include <math.h>

#include <mutex>

#include "checks.h"
#include "launch.h"

namespace spark {
namespace {

constexpr int kStaticGroups = 256;  // batch * n_kv a call may have
// CTAs a call may use: the automatic grid of the workspace entry point (two
// CTAs per SM on long histories) on GPUs of up to 160 SMs
constexpr int kStaticCtas = 320;
constexpr size_t kErrOff = 0;
constexpr size_t kCounterOff = 256;
constexpr size_t kPartOff = kCounterOff + sizeof(uint32_t) * kStaticGroups;  // 1280, 256-aligned
// a CTA c finishing group g writes partial slot c + g
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

}  // namespace
}  // namespace spark

using namespace spark;
using namespace spark::checks;

extern "C" int spark_dbg_attention_noalloc(const spark_geom* g, const float* q_rot,
                                           const spark_kv_layer* kv, int32_t layer_class,
                                           const int32_t* positions, int32_t batch, float* a,
                                           void* stream) {
  // the argument rules of spark_dbg_attention: every row the kernel reads
  // lies inside the cache buffers
  int s;
  if ((s = check_geom(g)) != SPARK_OK) return s;
  if ((s = check_batch(batch)) != SPARK_OK) return s;
  if ((s = check_kv(g, kv, layer_class, positions, batch)) != SPARK_OK) return s;
  if (!q_rot || !a || !aligned16(q_rot) || !aligned16(a)) return SPARK_ERR_INVALID_ARG;
  if (batch * g->n_kv > kStaticGroups) return SPARK_ERR_WORKSPACE;  // beyond the fixed scratch
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return SPARK_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  // the merge tickets must start at zero (a completed call leaves them so;
  // one that gave up on a wait may not); the error word keeps its bits
  if (cudaMemsetAsync(scratch + kCounterOff, 0, kPartOff - kCounterOff, st) != cudaSuccess)
    return SPARK_ERR_CUDA;
  // the grid spark_dbg_attention chooses by itself, within the array's CTAs
  const cudaError_t e = launch_attention(
      kv->dtype, q_rot, kv->k, kv->v, g->n_kv, kv->capacity, kv->ring_capacity,
      layer_class == SPARK_FULL, g->window, g->scale, positions, batch, a,
      reinterpret_cast<float*>(scratch + kPartOff), reinterpret_cast<uint32_t*>(scratch + kCounterOff),
      reinterpret_cast<uint32_t*>(scratch + kErrOff), 0, nullptr, 0, st, ChunkSrc(), kStaticCtas);
  return e == cudaSuccess ? SPARK_OK : SPARK_ERR_CUDA;
}

extern "C" int spark_dbg_attention_noalloc_error_word(uint32_t* word, void* stream) {
  if (!word) return SPARK_ERR_INVALID_ARG;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) return SPARK_ERR_CUDA;
  cudaStream_t st = (cudaStream_t)stream;
  uint32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, static_cast<unsigned char*>(base) + kErrOff, sizeof(uint32_t),
                                  cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(static_cast<unsigned char*>(base) + kErrOff, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  *word = host;
  return cuda_status(e);
}
