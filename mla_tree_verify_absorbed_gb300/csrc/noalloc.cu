// mla_verify_attn_noalloc: the verify call for callers that cannot allocate
// device memory when they call it -- for example a plugin running inside a
// host engine that owns every byte of the device memory pool, or a decode loop
// that must not pay the synchronisation cudaMalloc implies.  Such callers have
// no workspace to hand over, so this entry point uses a fixed scratch array
// that lives in the library image itself.
//
// The scratch is a file-scope __device__ array of MLA_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; later calls reuse the cached address.
//
// All calls share the one array and it keeps the previous call's contents.
// Nothing in it needs clearing by the caller: the metadata kernel zeroes the
// error word at the start of every call, and every other region is fully
// written before it is read within the same call.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and corrupt each other's results.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mla_verify.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
mla_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_verify_attn_noalloc(const mla_verify_args* args, int num_splits,
                                             mla_stream_t stream) {
  const size_t need = mla_verify_workspace_size(args, num_splits);
  if (need == 0) {
    // invalid arguments (or no device for num_splits == 0): let the regular
    // entry point report the precise status; it returns before any launch
    return mla_verify_attn(args, nullptr, 0, num_splits, stream);
  }
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  const mla_status st = scratch_address(&ws);
  if (st != MLA_OK) return st;
  return mla_verify_attn(args, ws, (size_t)MLA_NOALLOC_SCRATCH_BYTES, num_splits, stream);
}
