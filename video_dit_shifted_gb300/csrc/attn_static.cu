// wp_window_attn_static: window attention without any caller-provided or
// library-allocated workspace.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code inside a runtime that owns a fixed memory pool and forbids
// allocation from plugins, latency-critical loops where cudaMalloc's implicit
// device synchronisation is unacceptable, or callers that simply have no
// allocator at hand.  For them this entry point takes its scratch (the status
// block and the per-window text outputs) from one fixed array that lives in
// the library's device image.  Every GPU that loads the library holds that
// array, WP_STATIC_SCRATCH_BYTES bytes, until the process exits.
//
// The array's name means something different on the host than on the
// device: host code only sees a stand-in symbol.  Its real device address is
// asked from the runtime (cudaGetSymbolAddress) the first time this entry
// point (or wp_read_status with a NULL workspace) runs on a device, with that
// device current, and is remembered per device; the kernels then receive
// that address like any workspace pointer.  Under CUDA's lazy module loading
// that first lookup is also when the runtime loads this module onto the
// device and reserves the array, so the first call is the set-up; every
// later call reuses the remembered address and allocates nothing.  A
// cudaDeviceReset unloads the module: the remembered address is then stale,
// and this entry point must not be used on that device again in the process.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "attn_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[WP_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

}  // namespace

namespace wp {

// Device address of g_static_scratch on the current device (looked up once).
int static_scratch_address(void** out) {
  int dev = -1;
  if (int rc = wp::cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return rc;
  if (dev < 0 || dev >= kMaxDevices)
    return wp::fail(WP_EUNSUPPORTED, "device ordinal %d is beyond the %d this entry point supports", dev,
                    kMaxDevices);
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      if (int rc = wp::cuda_check(cudaGetSymbolAddress(&p, g_static_scratch),
                                  "cudaGetSymbolAddress(static scratch)"))
        return rc;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return WP_OK;
}

}  // namespace wp

extern "C" int wp_window_attn_static(const wp_plan* plan, int layout, int heads, int head_dim, int L,
                                     int dtype, const void* q, const void* k, const void* v,
                                     int64_t vid_row_stride_B, const void* qt, const void* kt,
                                     const void* vt, int64_t txt_row_stride_B, void* o_vid,
                                     int64_t o_vid_row_stride_B, void* o_txt, float softmax_scale,
                                     void* stream) {
  size_t need = 0;
  if (int rc = wp_attn_workspace_bytes(plan, layout, heads, head_dim, L, dtype, &need)) return rc;
  if (need > static_cast<size_t>(WP_STATIC_SCRATCH_BYTES))
    return wp::fail(WP_EUNSUPPORTED,
                    "this call needs %zu bytes of scratch (256 + nwin*L*heads*head_dim*4) but the "
                    "allocation-free entry point has %zu; use wp_window_attn with a workspace",
                    need, static_cast<size_t>(WP_STATIC_SCRATCH_BYTES));
  void* scratch = nullptr;
  if (int rc = wp::static_scratch_address(&scratch)) return rc;
  // wp_window_attn clears the status block itself at the start of the call;
  // the text partials are fully overwritten before they are read.
  return wp_window_attn(plan, layout, heads, head_dim, L, dtype, q, k, v, vid_row_stride_B, qt, kt, vt,
                        txt_row_stride_B, o_vid, o_vid_row_stride_B, o_txt, scratch,
                        static_cast<size_t>(WP_STATIC_SCRATCH_BYTES), softmax_scale, stream);
}
