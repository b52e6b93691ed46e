// attn_bwd_noalloc: the backward without a caller workspace, for callers that
// cannot allocate device memory (include/attn.h says who they are).  The
// scratch lives in a fixed file-scope device array; its device address is
// looked up once per device and handed to attn_bwd as the workspace.
#include <mutex>
#include <cuda_runtime.h>
#include "../../include/attn.h"

namespace {

// The scratch.  In host code this name is only a host-side stand-in for the
// device array: never pass it to a kernel; use the looked-up address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device
std::mutex g_scratch_mu;

// Device address of the scratch on the current device, looked up on first use.
// The device is checked first, so that a GPU this library was not built for
// gets ATTN_ERR_DEVICE (as from attn_bwd) rather than a failed lookup.  The
// first lookup on a device loads this file's module there (module loading is
// lazy), which is when the array is reserved.
attn_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (major != 10 || minor != 3) return ATTN_ERR_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // leave no pending error behind for a later launch check
      return ATTN_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const void* q, const void* k, const void* v,
                                          const void* o, const void* dout, const float* lse,
                                          void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                                          int N, int d, float scale, const attn_mods_t* mods,
                                          void* stream) {
  // Size check first.  attn_workspace_size is 0 for invalid arguments; attn_bwd
  // then reports the argument error itself.
  const size_t need = attn_workspace_size(ATTN_OP_BWD, B, Hq, Hkv, N, d, mods);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const attn_status_t st = scratch_address(&scratch);
    if (st != ATTN_OK) return st;
  }
  return attn_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N, d, scale, mods, scratch,
                  need > 0 ? (size_t)ATTN_NOALLOC_SCRATCH_BYTES : 0, stream);
}
