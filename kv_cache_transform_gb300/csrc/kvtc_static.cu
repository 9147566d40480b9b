// Column mean of calibration rows with no device allocation at all.
//
// kvtc_calibrate allocates its working buffers with cudaMalloc.  Some
// callers cannot do that: serving engines that hand nearly all device memory
// to their own KV-cache pool at start-up (a later cudaMalloc fails or
// fragments that pool), and latency-sensitive paths where cudaMalloc and
// cudaFree would synchronise the device and stall every other stream.  This
// entry point gives them the first calibration statistic, the per-channel
// mean, computed into memory they own, with its own scratch taken from a
// fixed array that lives in the library image.
#include <mutex>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"

namespace {

constexpr int kStaticMaxD = 4096;   // widest row the scratch array holds
constexpr int kStaticChunks = 32;   // row chunks summed independently

// Partial column sums [chunk][channel].  Modules load lazily, so this
// 1 MiB comes into being on a device at the first call there and stays
// until the process exits.  All calls on a device share it; each call
// writes every entry it later reads, so nothing needs clearing, but two
// calls that run at the same time on the GPU race.
static __device__ __align__(256) double g_mean_partial[kStaticChunks *
                                                       kStaticMaxD];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
double* g_partial_addr[kMaxDevices] = {};

// Sum of rows [chunk * rows_per, min(N, (chunk + 1) * rows_per)) of column d.
__global__ void mean_partial_kernel(const uint16_t* x, int64_t N, int64_t ld,
                                    int D, int64_t rows_per,
                                    double* partial) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  const int chunk = blockIdx.y;
  if (d >= D) return;
  const int64_t r0 = (int64_t)chunk * rows_per;
  const int64_t r1 = r0 + rows_per < N ? r0 + rows_per : N;
  double s = 0.0;
  for (int64_t t = r0; t < r1; ++t)
    s += (double)__uint_as_float((uint32_t)x[t * ld + d] << 16);
  partial[(int64_t)chunk * D + d] = s;
}

__global__ void mean_finish_kernel(const double* partial, int64_t N, int D,
                                   double* mu) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  if (d >= D) return;
  double s = 0.0;
  for (int c = 0; c < kStaticChunks; ++c) s += partial[(int64_t)c * D + d];
  mu[d] = s / (double)N;
}

}  // namespace

extern "C" int kvtc_calib_mean_static(int cuda_device, const void* tokens,
                                      int64_t N, int64_t ld, int D,
                                      double* mu_out, void* cuda_stream) {
  if (!tokens || !mu_out || N < 1 || D < 1 || ld < D || cuda_device < 0 ||
      cuda_device >= kMaxDevices)
    return KVTC_EINVAL;
  if (D > kStaticMaxD) return KVTC_ESIZE;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return KVTC_ECUDA;
  if (prev != cuda_device && cudaSetDevice(cuda_device) != cudaSuccess)
    return KVTC_ECUDA;
  int ret = KVTC_OK;
  double* partial = nullptr;
  {
    // One-time set-up per device, with that device current: the device
    // address of the scratch array (the host-side name of the array is not
    // a device address).
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_partial_addr[cuda_device]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_mean_partial) != cudaSuccess || !p)
        ret = KVTC_ECUDA;
      else
        g_partial_addr[cuda_device] = static_cast<double*>(p);
    }
    partial = g_partial_addr[cuda_device];
  }
  if (ret == KVTC_OK) {
    cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
    const int64_t rows_per = (N + kStaticChunks - 1) / kStaticChunks;
    mean_partial_kernel<<<dim3((D + 127) / 128, kStaticChunks), 128, 0, st>>>(
        static_cast<const uint16_t*>(tokens), N, ld, D, rows_per, partial);
    mean_finish_kernel<<<(D + 127) / 128, 128, 0, st>>>(partial, N, D, mu_out);
    if (cudaGetLastError() != cudaSuccess) ret = KVTC_ECUDA;
    kvtc::count_launch();
    kvtc::count_launch();
  }
  if (prev != cuda_device) cudaSetDevice(prev);
  return ret;
}
