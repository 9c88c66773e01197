// fastgen_decode_attn_noalloc: the generation step for callers that cannot
// allocate device memory at decode time.
//
// Who needs it: a serving engine that hands all free device memory to its own
// pool allocator at start-up (a later cudaMalloc would fail, or carve memory
// out from under that pool), a plug-in hosted by a framework that owns every
// allocation, or a latency-bound loop that cannot afford cudaMalloc's
// implicit device synchronisation.  Such a caller still owns the inputs,
// outputs and caches; only the decode scratch (the split-K partial results)
// moves into a fixed array inside this library.
//
// The array is a file-scope __device__ variable of this file's own CUDA
// module.  CUDA sets it aside on a device when it loads that module there:
// under the default lazy module loading, that happens at the first address
// look-up below (the first call of the entry point on that device); with
// CUDA_MODULE_LOADING=EAGER, when the device's context is created.  From then
// on the device holds FASTGEN_NOALLOC_SCRATCH_BYTES until the process exits,
// so callers make their first call at set-up, before their own pool takes the
// free memory and before any stream capture.  Host code cannot use the
// array's name as a device address, so the address is looked up once per
// device with cudaGetSymbolAddress (with that device current) and cached for
// the life of the process (the device's primary context is assumed to live
// that long).  Every call shares the array: calls that overlap on the GPU
// race.  Each call writes every scratch entry it reads, so nothing needs
// clearing between calls.
#include <mutex>

#include "fg_common.cuh"
#include "fg_internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[FASTGEN_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
fg_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FG_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FG_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return FG_OK;
}

}  // namespace

extern "C" fg_status fastgen_decode_attn_noalloc(
    const fg_params* p, void* plan, const fg_plan_info* info, void* K_pool, void* V_pool,
    int32_t* pos_pool, const void* q, const void* k_new, const void* v_new,
    const int32_t* new_ids, const int32_t* special_ids, int32_t n_special,
    const int32_t* punct_ids, int32_t n_punct, int32_t pos, void* out, int32_t* dev_err,
    void* stream) {
  if (!p || !info) return FG_EINVAL;
  const size_t need = fastgen_decode_workspace_bytes(p, info);
  if (need == 0 && info->n_work != 0) return FG_EINVAL;  // parameters rejected
  if (need > (size_t)FASTGEN_NOALLOC_SCRATCH_BYTES) return FG_EWORKSPACE;
  void* scratch = nullptr;
  const fg_status st = scratch_address(&scratch);
  if (st != FG_OK) return st;
  return fastgen_decode_attn(p, plan, info, K_pool, V_pool, pos_pool, q, k_new, v_new, new_ids,
                             special_ids, n_special, punct_ids, n_punct, pos, out, scratch,
                             (size_t)FASTGEN_NOALLOC_SCRATCH_BYTES, dev_err, stream);
}
