// kv_decode_attn_noalloc: decode attention whose split partials live in a
// fixed block of device memory that the library itself declares, so that the
// call needs no allocation of any kind from its caller or from this library.
//
// The block is a file-scope __device__ array. Every GPU that loads the
// library reserves it until the process exits. In host code its name stands
// for the symbol only; its device address comes from cudaGetSymbolAddress,
// taken once per device (with that device current) on the first call there.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

static_assert(KV_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");

// Split partials of the decode: [part_o | part_ml]. Nothing in it has to
// start at zero: each call writes every partial that its merge later reads.
static __device__ __align__(256) unsigned char g_decode_scratch[KV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch block on the current device (set up once).
kv_status scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::report(KV_ERR_CUDA, (std::string("cudaGetDevice: ") + cudaGetErrorString(e)).c_str());
  if (dev < 0 || dev >= kMaxDevices) return kvq::report(KV_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess || !p)
      return kvq::report(KV_ERR_CUDA,
                         (std::string("cudaGetSymbolAddress of the decode scratch: ") + cudaGetErrorString(e)).c_str());
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KV_OK;
}

}  // namespace

extern "C" kv_status kv_decode_attn_noalloc(kv_cache* cache, int layer, const void* q, float* out,
                                            float* lse_or_null, void* cuda_stream) {
  if (!cache) return kvq::report(KV_ERR_INVALID_ARG, "cache is NULL");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return kvq::report(KV_ERR_CUDA, (std::string("cudaGetDevice: ") + cudaGetErrorString(e)).c_str());
  if (dev != kvq::cache_device(cache))
    return kvq::report(KV_ERR_INVALID_ARG, "the cache's device must be the current device");
  void* scratch = nullptr;
  kv_status st = scratch_on_current_device(&scratch);
  if (st != KV_OK) return st;
  return kvq::decode_attn_impl(cache, layer, q, out, lse_or_null, cuda_stream, scratch, KV_NOALLOC_SCRATCH_BYTES);
}
