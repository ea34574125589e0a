// attn_fwd_splitkv_noalloc: split-KV decode for callers that cannot allocate
// device memory.  The partial results live in a fixed scratch array that is
// part of the library's device image, so no call allocates anything.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/attn.h"
#include "launch.h"

namespace {

// Scratch for the split kernel's partial outputs and LSEs.  It is module
// memory: every GPU that loads this library holds it until the process
// exits.  Its name is a host-side stand-in in host code; the device address
// is looked up per device below.
static __device__ __align__(256) unsigned char g_splitkv_scratch[ATTN_SPLITKV_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_mutex;
void* g_addr[kMaxDevices];  // device address of the scratch, per device, once looked up

// Device address of the scratch on the current device (looked up once per
// device, with that device current, and kept for the life of the process:
// a device reset after that first lookup is not supported).  NULL if the
// lookup fails.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" attn_status attn_fwd_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                                const int* seqlens, int max_seqlen, void* o, float* lse, int B,
                                                int Hq, int Hkv, int d, float scale, int chunk, void* stream) {
  // every other argument is checked first, with the codes attn_fwd_splitkv
  // gives them; nothing here touches the GPU before the size check passes
  const attn_status st = attn::check_splitkv_args(q, k_cache, v_cache, seqlens, max_seqlen, nullptr, 0, o, lse, B,
                                                  Hq, Hkv, d, scale, chunk);
  if (st != ATTN_OK) return st;
  const size_t need = attn_splitkv_workspace_size(B, Hq, max_seqlen, d, chunk);
  if (need > static_cast<size_t>(ATTN_SPLITKV_NOALLOC_MAX_BYTES)) return ATTN_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (!scratch) return ATTN_ERR_LAUNCH;
  // Every partial the combine kernel reads is written by the split kernel of
  // the same call, so the scratch needs no clearing between calls.
  return attn_fwd_splitkv(q, k_cache, v_cache, seqlens, max_seqlen, o, lse, B, Hq, Hkv, d, scale, chunk, scratch,
                          static_cast<size_t>(ATTN_SPLITKV_NOALLOC_MAX_BYTES), stream);
}
