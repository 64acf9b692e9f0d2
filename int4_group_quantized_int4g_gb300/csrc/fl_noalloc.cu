// Decode linear (M <= 32) that allocates nothing and takes no workspace.
//
// For callers that cannot allocate device memory at the point of the call:
// cudaMalloc may synchronize the whole device and can fail under memory
// pressure, so a latency-critical serving loop, a caller running inside a
// framework that owns every allocation, or host code that must not block
// cannot obtain a workspace for fl_int4g_linear.  This variant runs the same
// decode kernels, with the same dispatch, as fl_int4g_linear, with their
// split-K scratch (status block, ticket counters and fp32 partial sums) in a
// fixed device array that lives in the library.
#include <mutex>

#include "fl_common.cuh"

namespace {

// Maximum scratch of the variant.  Every GPU that loads the library holds
// this array until the process exits.
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB

// Status block and ticket counters of the decode workspace layout: they must
// be zero when a call starts.  The array starts zero-filled, and every
// successful call leaves them zero (each last arriver resets its counter).
constexpr size_t kCounterRegionBytes = fl::kScratchOff;
static_assert(kCounterRegionBytes <= kNoAllocScratchBytes, "the counter region must fit the scratch array");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (the host name of the array is only a stand-in, not a
// device address).  The cached address is that of the device's primary
// context: it is not refreshed after a device reset.
void* scratch_address(int dev) {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

int fl_linear_decode_workspace(int M, int N, int K, size_t* out);
int fl_linear_decode(const void* x, int M, int K, const void* w, int N, void* y, void* ws, size_t ws_bytes,
                     cudaStream_t s);

extern "C" int fl_int4g_linear_noalloc(const void* x, int M, int K, const void* w, int N, void* y,
                                       fl_stream_t stream) {
  if (!x || !w || !y || M < 1 || N < 1 || K < fl::kGroup || K % fl::kGroup) return FL_ERR_ARG;
  if (!flh::aligned16(x) || !flh::aligned16(w) || !flh::aligned16(y)) return FL_ERR_ARG;
  if (M > 32) return FL_ERR_UNSUPPORTED;
  size_t need = 0;
  if (fl_linear_decode_workspace(M, N, K, &need) != FL_OK) return FL_ERR_ARG;
  if (need > kNoAllocScratchBytes) return FL_ERR_WORKSPACE;   // shape needs more than the fixed scratch
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FL_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (!ws) return FL_ERR_CUDA;
  return fl_linear_decode(x, M, K, w, N, y, ws, kNoAllocScratchBytes, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fl_int4g_linear_noalloc_status(fl_stream_t stream, int* out) {
  if (!out) return FL_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FL_ERR_CUDA;
  void* ws = scratch_address(dev);
  if (!ws) return FL_ERR_CUDA;
  const int rc = fl_int4g_status(ws, stream, out);
  if (rc != FL_OK) return rc;
  // a call that gave up may have left ticket counters behind: clear them
  if (*out != FL_OK) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kCounterRegionBytes, s) != cudaSuccess) return FL_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FL_ERR_CUDA;
  }
  return FL_OK;
}
