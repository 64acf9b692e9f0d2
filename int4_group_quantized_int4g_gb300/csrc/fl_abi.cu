// Status, version and error strings of the C ABI; cached device attributes.
#include "fl_common.cuh"

namespace flh {

// Without a visible device (host-only size queries) the plan assumes a GB300
// (152 SMs); launches always use the real count of the current device.
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return 152;
  }
  if (dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
    cudaGetLastError();
    return 152;
  }
  if (dev < 64) cache[dev] = n;
  return n;
}

}  // namespace flh

extern "C" const char* fl_strerror(int status) {
  switch (status) {
    case FL_OK: return "ok";
    case FL_ERR_ARG: return "invalid argument";
    case FL_ERR_WORKSPACE: return "workspace too small";
    case FL_ERR_UNSUPPORTED: return "unsupported shape or group size";
    case FL_ERR_CUDA: return "CUDA launch or query failed";
    case FL_ERR_TIMEOUT: return "device-side wait ran out of time";
    case FL_ERR_DEVICE_CHECK: return "device-side check failed";
    case FL_ERR_RANGE: return "group scale overflows fp16";
    default: return "unknown status";
  }
}

extern "C" int fl_int4g_version(void) { return 100; }

extern "C" int fl_int4g_status(void* ws, fl_stream_t stream, int* out) {
  if (!ws || !out || !flh::aligned16(ws)) return FL_ERR_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t h[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return FL_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FL_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(h), s) != cudaSuccess) return FL_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FL_ERR_CUDA;
  *out = h[0];
  return FL_OK;
}
