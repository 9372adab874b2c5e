// tm_w4a16_gemm_host_static: the host-buffer product staged through a fixed
// device array instead of caller-provided device buffers.
//
// Some callers cannot allocate device memory at the point where they want a
// product: a plug-in loaded into a host application whose memory pool has
// already reserved the device (cudaMalloc fails or fragments that pool), or a
// latency-critical loop where cudaMalloc/cudaFree may block or synchronise the
// device.  For them the staging lives in one file-scope __device__ array that
// the module reserves when it loads on a device and keeps until the process
// exits; this call never allocates.
#include <cstdint>
#include <mutex>

#include "tm_common.cuh"

namespace w4 {

static_assert(TM_STATIC_STAGING_BYTES % 256 == 0, "the staging size must keep the 256-byte alignment");

// X at offset 0, Y at the next 256-byte boundary after X.  Shared by every
// call on a device; it holds whatever the last call left there.
static __device__ __align__(256) unsigned char s_static_staging[TM_STATIC_STAGING_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_staging_mu;
void* g_staging_ptr[kMaxDevices] = {};

// In host code s_static_staging names a host-side shadow, not device memory:
// the device address comes from the runtime, once per device, with that
// device current.
tm_status staging_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return TM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_staging_mu);
  if (!g_staging_ptr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, s_static_staging) != cudaSuccess || !ptr) return TM_ERR_CUDA;
    g_staging_ptr[device] = ptr;
  }
  *out = g_staging_ptr[device];
  return TM_OK;
}

}  // namespace
}  // namespace w4

using namespace w4;

extern "C" tm_status tm_w4a16_gemm_host_static(const void* X_host, const tm_packed* p, void* Y_host, int M,
                                               const tm_gemm_config* cfg, void* stream) {
  set_launch_count(0);
  if (!p || M < 0) return TM_ERR_INVALID_ARG;
  if (M == 0) return TM_OK;
  if (!X_host || !Y_host) return TM_ERR_INVALID_ARG;
  const size_t x_bytes = (size_t)M * (size_t)p->L.K * 2;
  const size_t y_off = (x_bytes + 255) & ~size_t(255);
  const size_t y_bytes = (size_t)M * (size_t)p->L.N * 2;
  if (y_off + y_bytes > (size_t)TM_STATIC_STAGING_BYTES) return TM_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TM_ERR_CUDA;
  if (dev != p->device) return TM_ERR_INVALID_ARG;  // the weights and the staging must share a device
  void* base = nullptr;
  const tm_status st = staging_address(dev, &base);
  if (st != TM_OK) return st;
  return tm_w4a16_gemm_host(X_host, p, Y_host, M, base, static_cast<unsigned char*>(base) + y_off, cfg, stream);
}
