// vpce_forward_static: the forward loss with no caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they need the
// loss: a plugin living inside a framework whose pooling allocator already
// owns (nearly) all of the GPU's memory, so a raw cudaMalloc fails or
// fragments that pool; code running on a path where cudaMalloc's implicit
// device synchronisation is not acceptable (a latency-bound evaluation loop);
// or deployments that forbid device allocation after start-up.  For them this
// entry point keeps its scratch in a fixed, file-scope device array instead.
//
// The array holds VPCE_STATIC_SCRATCH_BYTES on every GPU that loads this
// library, until the process exits.  Host code may not use the array's name as
// a device address (on the host it is only a stand-in), so the address is
// looked up once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device.
#include <mutex>

#include "vpce_kernels.cuh"

static __device__ __align__(256) unsigned char vpce_static_scratch[VPCE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxStaticDevices] = {};

// Device address of this device's copy of the scratch array.
vpce_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return VPCE_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxStaticDevices) return VPCE_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_addr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, vpce_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return VPCE_ERR_CUDA;
    }
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return VPCE_OK;
}

}  // namespace

extern "C" vpce_status vpce_forward_static(const void* const* shards, vpce_dtype dtype, int t, int64_t s,
                                           const int64_t* vocab_start, int64_t ld, const int64_t* targets,
                                           int64_t ignore_index, vpce_reduction reduction, float* loss_out,
                                           float* row_loss_out, vpce_stream_t stream) {
  if (t < 1 || t > VPCE_MAX_SHARDS || s < 0 || s > (int64_t(1) << 31)) return VPCE_ERR_INVALID_ARG;
  if (vpce::WsLayout(t, s).total > size_t(VPCE_STATIC_SCRATCH_BYTES)) return VPCE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const vpce_status st = static_scratch_address(&scratch);
  if (st != VPCE_OK) return st;
  // vpce_forward clears the scratch header (batch counter, error flag) in
  // stream order at the start of every call; everything else is written
  // before it is read.  A wait that gave up makes the loss NaN, so a caller
  // without access to the error flag still sees the failure.
  return vpce_forward(shards, dtype, t, s, vocab_start, ld, targets, ignore_index, reduction, loss_out,
                      row_loss_out, scratch, size_t(VPCE_STATIC_SCRATCH_BYTES), stream);
}
