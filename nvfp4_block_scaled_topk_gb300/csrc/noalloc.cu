// megamoe_forward_static: the routed-expert forward for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc where they run the
// forward: plugins loaded into a host process that owns every device
// allocation (an inference server with its own memory pool, which forbids
// side allocations), embedded callers that link only this library and have no
// allocator of their own at hand, and hot loops that must never enter the
// driver's allocator.  For them this file keeps the forward's workspace in a
// file-scope device array of fixed size, MEGAMOE_STATIC_WS_BYTES (64 MiB),
// which every GPU that loads the library holds until the process exits.  The
// caller still passes the weights, the inputs and the outputs.
//
// The array's address is looked up once per device and driver context, with
// that device current, by the first call made there (cudaGetSymbolAddress);
// that first call should therefore come before any stream capture.  A later
// call under another context of the device (after cudaDeviceReset, or with a
// context the caller made current through the driver API) looks it up again.
// Every call shares the one array, so calls that overlap on the GPU (two
// streams, or two host threads on one device) race and must be serialised by
// the caller.  The forward itself clears what must start at zero (status
// word, amax accumulators) at the start of every call and rewrites every
// other region it reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/megamoe.h"
#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[MEGAMOE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
struct Slot {
  CUcontext ctx;  // the context the address was looked up in
  void* ptr;
};
Slot g_ws[kMaxDevices] = {};
std::mutex g_ws_mutex;

using CtxGetCurrent = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver (through the runtime's entry-point query,
// so the library needs no link against libcuda).
CtxGetCurrent ctx_get_current() {
  static CtxGetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrent>(p);
  });
  return fn;
}

// Device address of g_static_ws in the current device's current context
// (nullptr on failure).
void* static_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrent get = ctx_get_current();
  if (!get) return nullptr;
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS || !ctx) {
    // no context is current on this thread: the device's primary context
    // (a context the caller made current is kept as it is)
    if (cudaSetDevice(dev) != cudaSuccess) return nullptr;
    ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (!g_ws[dev].ptr || g_ws[dev].ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return nullptr;
    g_ws[dev].ctx = ctx;
    g_ws[dev].ptr = p;
  }
  return g_ws[dev].ptr;
}

}  // namespace

extern "C" megamoe_status megamoe_forward_static(const megamoe_weights* w, const uint16_t* x,
                                                  const int32_t* topk_ids,
                                                  const float* topk_weights, int T, int k,
                                                  int pad, uint16_t* out, uint32_t* status_out,
                                                  megamoe_stream_t stream) {
  // the forward's own argument and shape errors come first, so that a shape
  // the forward cannot take is never reported as a workspace limit
  megamoe_status st =
      megamoe::check_forward_args(w, x, topk_ids, topk_weights, T, k, pad, out, false);
  if (st != MEGAMOE_OK) return st;
  const size_t need =
      megamoe_workspace_size(T, k, w->num_experts, w->hidden, w->intermediate, pad);
  if (need == 0) return MEGAMOE_ERR_INVALID_ARG;
  if (need > MEGAMOE_STATIC_WS_BYTES) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;
  void* ws = static_workspace();
  if (!ws) return MEGAMOE_ERR_CUDA;
  st = megamoe_forward(w, x, topk_ids, topk_weights, T, k, pad, out, ws, MEGAMOE_STATIC_WS_BYTES,
                       stream);
  if (st != MEGAMOE_OK || !status_out) return st;
  // the workspace's first word is the forward's device status word
  if (cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MEGAMOE_ERR_CUDA;
  return MEGAMOE_OK;
}
