// Allocation-free decode entry point.
//
// Some callers cannot allocate device memory at the moment they decode: a
// serving process whose device memory is owned and fully pre-reserved by
// another framework's allocator, a real-time request thread on which any
// allocation (and the device-wide synchronisation cudaFree implies) is
// forbidden, or a runtime that plans all memory statically at start-up.
// zg_decode_static gives them the decode with its scratch taken from a fixed
// array in the library's own device memory instead of a caller workspace.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits.  In host code its name is only
// a host-side stand-in, so its device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and then passed on.
#include <mutex>

#include "zg_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = (size_t)ZG_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[64] = {};
unsigned long long g_static_ctx[64] = {};  // context the cached address belongs to

}  // namespace

extern "C" zg_status zg_decode_static(const zg_index* idx, const zg_plan* plan, const zg_model* model,
                                      const float* u, int32_t B, int32_t beam, int32_t K, int32_t* out_sids,
                                      float* out_scores, void* stream) {
  size_t need = 0;
  zg_status st = zg_decode_workspace_size(idx, plan, model, B, beam, K, &need);
  if (st != ZG_OK) return st;
  if (need > kStaticScratchBytes) {
    return zg::fail(ZG_ERR_INVALID_ARG,
                    "zg_decode_static: this decode needs " + std::to_string(need) +
                        " bytes of scratch, more than the library's static scratch of " +
                        std::to_string(kStaticScratchBytes) + " bytes; use zg_decode with a workspace");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return zg::cuda_fail(e, "zg_decode_static: cudaGetDevice");
  if (dev < 0 || dev >= 64) return zg::fail(ZG_ERR_UNSUPPORTED, "zg_decode_static: device ordinal >= 64");
  unsigned long long ctx = 0;
  e = zg::current_context_id(&ctx);
  if (e != cudaSuccess) return zg::cuda_fail(e, "zg_decode_static: current context");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_static_mu);
    // looked up once per device and context: a context created after
    // cudaDeviceReset holds a new copy of the array at a new address
    if (!g_static_ptr[dev] || g_static_ctx[dev] != ctx) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) return zg::cuda_fail(e, "zg_decode_static: cudaGetSymbolAddress of the static scratch");
      g_static_ptr[dev] = p;
      g_static_ctx[dev] = ctx;
    }
    scratch = g_static_ptr[dev];
  }
  // The decode writes every scratch word before it reads it, so the array
  // needs no clearing between calls.
  return zg_decode(idx, plan, model, u, B, beam, K, out_sids, out_scores, scratch, kStaticScratchBytes, stream);
}

extern "C" size_t zg_static_scratch_bytes(void) { return kStaticScratchBytes; }
