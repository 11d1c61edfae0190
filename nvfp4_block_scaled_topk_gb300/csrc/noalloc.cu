// megamoe_forward_static: the routed-expert forward for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc on the path where they
// run the forward: code running inside a CUDA stream capture whose graph must
// not contain allocation nodes, plugins loaded into a host process that owns
// every allocation (an inference server with its own pool, which forbids side
// allocations), or hot loops that must never enter the driver's allocator.
// For them this file keeps the forward's workspace in a file-scope device
// array of fixed size, MEGAMOE_STATIC_WS_BYTES (64 MiB), which every GPU that
// loads the library holds until the process exits.  The caller still passes
// the weights, the inputs and the outputs.
//
// The array's address is looked up once per device, with that device current,
// by the first call made on that device (cudaGetSymbolAddress); that first
// call should therefore come before any stream capture.  Every call shares the
// one array, so calls that overlap on the GPU (two streams, or two host
// threads on one device) race and must be serialised by the caller.  The
// forward itself clears what must start at zero (status word, amax
// accumulators) at the start of every call and rewrites every other region it
// reads.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/megamoe.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[MEGAMOE_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
void* g_ws_ptr[kMaxDevices] = {};
std::mutex g_ws_mutex;

// Device address of g_static_ws on the current device (nullptr on failure).
void* static_workspace(int* err) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = 1;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_ws_mutex);
  if (!g_ws_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) {
      *err = 1;
      return nullptr;
    }
    g_ws_ptr[dev] = p;
  }
  return g_ws_ptr[dev];
}

}  // namespace

extern "C" megamoe_status megamoe_forward_static(const megamoe_weights* w, const uint16_t* x,
                                                  const int32_t* topk_ids,
                                                  const float* topk_weights, int T, int k,
                                                  int pad, uint16_t* out, uint32_t* status_out,
                                                  megamoe_stream_t stream) {
  if (!w) return MEGAMOE_ERR_INVALID_ARG;
  const size_t need =
      megamoe_workspace_size(T, k, w->num_experts, w->hidden, w->intermediate, pad);
  if (need == 0) return MEGAMOE_ERR_INVALID_ARG;
  if (need > MEGAMOE_STATIC_WS_BYTES) return MEGAMOE_ERR_WORKSPACE_TOO_SMALL;
  int err = 0;
  void* ws = static_workspace(&err);
  if (!ws) return MEGAMOE_ERR_CUDA;
  const megamoe_status st =
      megamoe_forward(w, x, topk_ids, topk_weights, T, k, pad, out, ws, MEGAMOE_STATIC_WS_BYTES,
                      stream);
  if (st != MEGAMOE_OK || !status_out) return st;
  // the workspace's first word is the forward's device status word
  if (cudaMemcpyAsync(status_out, ws, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MEGAMOE_ERR_CUDA;
  return MEGAMOE_OK;
}
