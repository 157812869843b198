// noalloc.cu - rnn_forward_noalloc: the inference forward without any device
// allocation by the library.
//
// Who needs it: callers that cannot let a library call cudaMalloc - for
// example a serving process whose device memory is entirely pre-reserved and
// handed out by its own allocator or a framework's caching pool (a cudaMalloc
// from inside the library would fail or break that budget), or a latency-
// critical loop where the implicit device-wide synchronisation of cudaMalloc /
// cudaFree is not acceptable.  rnn_create allocates the handle's small device
// area and rnn_forward needs a caller-allocated workspace; this entry point
// needs neither.  The caller still passes (and owns) every input and output.
//
// Where the scratch lives: one file-scope __device__ array of
// RNN_NOALLOC_SCRATCH_BYTES, part of the library image, so every GPU that loads
// the library holds it until the process exits.  It holds the persistent
// kernels' step counters and status word followed by the forward's workspace
// (projection, packed weights, per-layer outputs).  Host code cannot use the
// array's name as a device address (it names a host-side stand-in), so the
// first call on each device resolves the real address with
// cudaGetSymbolAddress while that device is current, and caches it.
//
// Sharing: every call on a device uses the same array, which keeps whatever
// the last call left in it.  The counters and the status word are cleared at
// the start of each call (on its stream); everything else is written before it
// is read.  Calls whose executions overlap on the GPU (other streams, other
// threads) race on the array and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "handle.h"
#include "rnn.h"
#include "rnn_internal.h"

namespace {

constexpr size_t kScratchBytes = RNN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device, with that device current).
rnn_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_CUDA_ERROR;
  if (dev < 0 || dev >= kMaxDevices) return RNN_NOT_SUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return RNN_CUDA_ERROR;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return RNN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" rnn_status_t rnn_forward_noalloc(const rnn_desc_t* desc, const void* x, const void* hx,
                                            const void* cx, const void* w, void* y, void* hy, void* cy, int sync,
                                            void* stream) {
  if (!desc || !x || !w || !y) return RNN_BAD_PARAM;
  rnn_handle_s h;
  int rc = rnn::init_handle_host(&h, desc);
  if (rc != RNN_OK) return static_cast<rnn_status_t>(rc);
  const size_t area = align256(sizeof(rnn::DevArea));
  if (area + h.workspace_bytes > kScratchBytes) return RNN_NOT_SUPPORTED;   // too large for the fixed scratch
  void* base = nullptr;
  rnn_status_t rs = scratch_for_current_device(&base);
  if (rs != RNN_OK) return rs;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h.dev = static_cast<rnn::DevArea*>(base);
  // counters and status must start at zero; the last call left them as it ended
  if (cudaMemsetAsync(h.dev, 0, sizeof(rnn::DevArea), s) != cudaSuccess) return RNN_CUDA_ERROR;
  rs = rnn_forward(&h, x, hx, cx, w, y, hy, cy, static_cast<char*>(base) + area, nullptr, stream);
  if (rs != RNN_OK || !sync) return rs;
  return rnn_noalloc_status(stream);
}

extern "C" rnn_status_t rnn_noalloc_status(void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RNN_CUDA_ERROR;
  if (dev < 0 || dev >= kMaxDevices) return RNN_NOT_SUPPORTED;
  void* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    base = g_scratch_addr[dev];
  }
  if (!base) return RNN_OK;   // no call on this device yet
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return RNN_CUDA_ERROR;
  rnn::DevArea* area = static_cast<rnn::DevArea*>(base);
  unsigned int code = 0;
  if (cudaMemcpy(&code, &area->status, sizeof(code), cudaMemcpyDeviceToHost) != cudaSuccess)
    return RNN_CUDA_ERROR;
  if (code != 0 && cudaMemset(&area->status, 0, sizeof(code)) != cudaSuccess) return RNN_CUDA_ERROR;
  return static_cast<rnn_status_t>(code);
}
