// ep_debug.cu -- test hooks that reach device code of the dispatch without a
// dispatch: the FP8 payload's E4M3 conversion applied to any float32.
#include "ep_scatter.cuh"

// Test hook: the dispatch's E4M3 conversion (cvt_e4m3x4) applied to the
// float32 bit patterns first .. first + n - 1, four per thread.
namespace ep {
namespace {
__global__ void e4m3_range_kernel(uint32_t first, int64_t n4, uint32_t* out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const uint32_t b = first + (uint32_t)(4 * i);
  out[i] = cvt_e4m3x4(__uint_as_float(b), __uint_as_float(b + 1), __uint_as_float(b + 2),
                      __uint_as_float(b + 3));
}
}  // namespace
}  // namespace ep

extern "C" ep_status_t ep_debug_e4m3_range(uint32_t first, int64_t n, uint8_t* out,
                                           ep_stream_t stream) {
  if (n < 0 || n % 4 != 0 || (uint64_t)first + (uint64_t)n > (uint64_t(1) << 32))
    return EP_ERR_INVALID_ARG;
  if (n == 0) return EP_OK;
  if (!out || (reinterpret_cast<uintptr_t>(out) & 3) != 0) return EP_ERR_INVALID_ARG;
  const int64_t n4 = n / 4;
  const int64_t blocks = (n4 + 255) / 256;
  ep::e4m3_range_kernel<<<(unsigned)blocks, 256, 0, ep::to_cuda(stream)>>>(
      first, n4, reinterpret_cast<uint32_t*>(out));
  return ep::launch_status();
}
