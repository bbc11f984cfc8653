// mla_verify_attn_noalloc: the verify call for callers that cannot allocate
// device memory when they call it -- for example a plugin running inside a
// host engine that owns every byte of the device memory pool, or a decode loop
// that must not pay the synchronisation cudaMalloc implies.  Such callers have
// no workspace to hand over, so this entry point uses a fixed scratch array
// that lives in the library image itself.
//
// The scratch is a file-scope __device__ array of MLA_NOALLOC_SCRATCH_BYTES.
// It is reserved on a device when the library's device code is loaded there:
// under lazy module loading (the CUDA default) that happens inside the first
// call on that device, which looks the array up, so that first call must come
// at start-up -- before a host engine claims the rest of the device memory,
// and before any stream capture.  It stays reserved until the process exits.
// Host code cannot use the array's name as a device address: each call looks
// the address up with cudaGetSymbolAddress (with the caller's device current)
// the first time it sees a CUDA context, and reuses it while that context
// lives; a new context on the device (after cudaDeviceReset, say) is looked up
// afresh.
//
// All calls share the one array and it keeps the previous call's contents.
// Nothing in it needs clearing by the caller: the metadata kernel zeroes the
// error word at the start of every call, and every other region is fully
// written before it is read within the same call.  Two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and corrupt each other's results.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mla_verify.h"

namespace mlav {
int plan_splits(const mla_verify_args* a, int num_splits);
}

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Identity of the current CUDA context, from the driver (0 when it cannot be
// had, in which case nothing is cached).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct Cached {
  unsigned long long ctx_id;
  void* addr;
};
std::mutex g_mutex;
Cached g_cache[kMaxDevices] = {};

// Device address of the scratch array in the current context.
mla_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  // 0 when the device has no context yet: the lookup below creates it, and
  // the next call caches
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (id != 0 && g_cache[dev].ctx_id == id && g_cache[dev].addr) {
    *out = g_cache[dev].addr;
    return MLA_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  g_cache[dev] = Cached{id, id ? p : nullptr};
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_verify_attn_noalloc(const mla_verify_args* args, int num_splits,
                                             mla_stream_t stream) {
  int splits = num_splits;
  size_t need = mla_verify_workspace_size(args, splits);
  if (need == 0) {
    // invalid arguments (or no device for num_splits == 0): let the regular
    // entry point report the precise status; it returns before any launch
    return mla_verify_attn(args, nullptr, 0, num_splits, stream);
  }
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) {
    if (num_splits != 0) return MLA_ERR_WORKSPACE;
    // automatic choice: the largest split count up to the automatic one whose
    // workspace fits the scratch (one split needs no partials, so it always fits)
    splits = mlav::plan_splits(args, 0);
    if (splits < 1) return MLA_ERR_INVALID_ARG;
    while (splits > 1 && mla_verify_workspace_size(args, splits) > (size_t)MLA_NOALLOC_SCRATCH_BYTES) --splits;
    need = mla_verify_workspace_size(args, splits);
    if (need == 0 || need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  }
  void* ws = nullptr;
  const mla_status st = scratch_address(&ws);
  if (st != MLA_OK) return st;
  return mla_verify_attn(args, ws, (size_t)MLA_NOALLOC_SCRATCH_BYTES, splits, stream);
}

extern "C" mla_status mla_verify_noalloc_check(mla_stream_t stream, uint32_t* bits) {
  void* ws = nullptr;
  const mla_status st = scratch_address(&ws);
  if (st != MLA_OK) return st;
  return mla_verify_check(ws, stream, bits);
}
