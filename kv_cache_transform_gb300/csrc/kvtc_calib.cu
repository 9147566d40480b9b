// One-time calibration on the GPU (kvtc page, technical summary 2A):
// per (layer, K|V) stream, the mean and PCA basis of calibration KV, the
// distortion of every group at every width measured with the codec's own
// quantiser, and the DP bit allocation under the budget.  Writes a
// calibration blob (format in include/kvtc.h).
//
// Arithmetic is fp64 throughout.  The covariance and the coefficient
// products are plain dense GEMMs (cuBLAS); the symmetric eigensolver is
// cuSOLVER's divide-and-conquer routine.  Mean, centring, the distortion
// table and the bit allocation are this library's own code.
#include <cublas_v2.h>
#include <cusolverDn.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <vector>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"

namespace {

constexpr int kGroupC = 16;
constexpr int kBmax = 8;
constexpr int kTokTile = 64;  // tokens per distortion-table block

__device__ __forceinline__ double bf16_to_f64(uint16_t b) {
  return (double)__uint_as_float((uint32_t)b << 16);
}

// mu[d] = mean over rows of x[:, d]
__global__ void column_mean_kernel(const uint16_t* x, int64_t N, int64_t ld,
                                   int D, double* mu) {
  const int d = blockIdx.x * blockDim.x + threadIdx.x;
  if (d >= D) return;
  double s = 0.0;
  for (int64_t t = 0; t < N; ++t) s += bf16_to_f64(x[t * ld + d]);
  mu[d] = s / (double)N;
}

// xc[t][d] = x[t][d] - mu[d]   (row-major, row stride D)
__global__ void centre_kernel(const uint16_t* x, int64_t N, int64_t ld, int D,
                              const double* mu, double* xc) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N * D) return;
  const int64_t t = i / D;
  const int d = (int)(i - t * D);
  xc[i] = bf16_to_f64(x[t * ld + d]) - mu[d];
}

// Directed fp64 -> fp16 roundings: fp64 -> fp32 and fp32 -> fp16 in the same
// direction compose to the single directed rounding.
__device__ __forceinline__ double rd16(double v) {
  return (double)__half2float(__float2half_rd(__double2float_rd(v)));
}
__device__ __forceinline__ double ru16(double v) {
  return (double)__half2float(__float2half_ru(__double2float_ru(v)));
}

// Partial distortion table: block (tile, g) sums, over its tokens, the
// squared error of group g at widths 0..8 -> part[tile][g][9].
__global__ void distortion_kernel(const double* c, int64_t N, int D,
                                  double* part) {
  const int G = D / kGroupC;
  const int g = blockIdx.y;
  const int64_t t = (int64_t)blockIdx.x * kTokTile + threadIdx.x;
  double e[kBmax + 1];
#pragma unroll
  for (int b = 0; b <= kBmax; ++b) e[b] = 0.0;
  if (t < N) {
    double v[kGroupC];
    double lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int i = 0; i < kGroupC; ++i) {
      v[i] = c[t * D + g * kGroupC + i];
      lo = fmin(lo, v[i]);
      hi = fmax(hi, v[i]);
      e[0] += v[i] * v[i];
    }
    const double shift = rd16(lo);
#pragma unroll
    for (int b = 1; b <= kBmax; ++b) {
      const double lev = (double)((1 << b) - 1);
      const double scale = ru16((hi - shift) / lev);
      double s = 0.0;
#pragma unroll
      for (int i = 0; i < kGroupC; ++i) {
        double q = 0.0;
        if (scale > 0.0) {
          q = floor((v[i] - shift) / scale + 0.5);
          q = fmin(fmax(q, 0.0), lev);
        }
        const double r = v[i] - (shift + q * scale);
        s += r * r;
      }
      e[b] = s;
    }
  }
  // deterministic block reduction over the tokens of this tile
  __shared__ double red[kTokTile][kBmax + 1];
#pragma unroll
  for (int b = 0; b <= kBmax; ++b) red[threadIdx.x][b] = e[b];
  __syncthreads();
  for (int s = kTokTile / 2; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s)
      for (int b = 0; b <= kBmax; ++b)
        red[threadIdx.x][b] += red[threadIdx.x + s][b];
    __syncthreads();
  }
  if (threadIdx.x == 0)
    for (int b = 0; b <= kBmax; ++b)
      part[((int64_t)blockIdx.x * G + g) * (kBmax + 1) + b] = red[0][b];
}

int cost_units(int b) { return b == 0 ? 0 : 2 + b; }

// DP over groups: least summed distortion within budget_bits / 16 units;
// ties keep the smaller width.
std::vector<uint8_t> allocate(const std::vector<double>& E, int G, int bmax,
                              int budget_bits) {
  const int U = budget_bits / 16;
  std::vector<double> F((size_t)(G + 1) * (U + 1), 0.0);
  std::vector<uint8_t> choice((size_t)(G + 1) * (U + 1), 0);
  for (int g = 1; g <= G; ++g)
    for (int u = 0; u <= U; ++u) {
      double best = std::numeric_limits<double>::infinity();
      int bb = 0;
      for (int b = 0; b <= bmax; ++b) {
        const int cu = cost_units(b);
        if (cu > u) break;
        const double v = F[(size_t)(g - 1) * (U + 1) + (u - cu)] +
                         E[(size_t)(g - 1) * (kBmax + 1) + b];
        if (v < best) {
          best = v;
          bb = b;
        }
      }
      F[(size_t)g * (U + 1) + u] = best;
      choice[(size_t)g * (U + 1) + u] = (uint8_t)bb;
    }
  std::vector<uint8_t> w(G);
  int u = U;
  for (int g = G; g >= 1; --g) {
    const int b = choice[(size_t)g * (U + 1) + u];
    w[g - 1] = (uint8_t)b;
    u -= cost_units(b);
  }
  return w;
}

struct Out {
  uint8_t* p;
  size_t cap, n = 0;
  bool ok = true;
  void put(const void* src, size_t bytes) {
    if (n + bytes > cap) ok = false;
    if (ok) std::memcpy(p + n, src, bytes);
    n += bytes;
  }
  void u32(uint32_t v) { put(&v, 4); }
};

}  // namespace

extern "C" {

int64_t kvtc_blob_max_bytes(int n, int D) {
  if (n <= 0 || D <= 0 || D % 16) return KVTC_EINVAL;
  const int64_t G = D / 16;
  const int64_t per = 16 + (G + 7) / 8 * 8 + 8LL * D + 8LL * D * D + 8LL * D;
  return 32 + per * n + 8;
}

int kvtc_calibrate(int cuda_device, int n, const int* layers, const int* kvs,
                   const void* const* tokens, int64_t N, int64_t ld, int D,
                   int sink, int window, int budget_bits, void* blob,
                   size_t capacity, size_t* blob_bytes, void* cuda_stream) {
  if (n <= 0 || !layers || !kvs || !tokens || !blob_bytes || N < 2 ||
      D <= 0 || D % 16 || ld < D || sink < 0 || window < 0 ||
      budget_bits < 0 || budget_bits > (1 << 24))
    return KVTC_EINVAL;
  for (int i = 0; i < n; ++i)
    if (!tokens[i] || kvs[i] < 0 || kvs[i] > 1 || layers[i] < 0)
      return KVTC_EINVAL;
  int prev = -1;
  cudaGetDevice(&prev);
  if (cudaSetDevice(cuda_device) != cudaSuccess) return KVTC_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int G = D / kGroupC;
  const int64_t tiles = (N + kTokTile - 1) / kTokTile;

  double *mu = nullptr, *xc = nullptr, *cov = nullptr, *w = nullptr,
         *V = nullptr, *coef = nullptr, *part = nullptr, *work = nullptr;
  int* info = nullptr;
  cublasHandle_t blas = nullptr;
  cusolverDnHandle_t solver = nullptr;
  int ret = KVTC_OK;
  auto cu = [&](cudaError_t e) {
    if (e != cudaSuccess && ret == KVTC_OK) ret = KVTC_ECUDA;
    return ret == KVTC_OK;
  };
  Out out{static_cast<uint8_t*>(blob), blob ? capacity : 0};
  out.put("KVTC", 4);
  const uint32_t hdr[7] = {1u, (uint32_t)n, 16u, 8u, (uint32_t)sink,
                           (uint32_t)window, (uint32_t)budget_bits};
  for (uint32_t v : hdr) out.u32(v);

  do {
    if (!cu(cudaMalloc(&mu, 8LL * D)) || !cu(cudaMalloc(&xc, 8LL * N * D)) ||
        !cu(cudaMalloc(&cov, 8LL * D * D)) || !cu(cudaMalloc(&w, 8LL * D)) ||
        !cu(cudaMalloc(&V, 8LL * D * D)) ||
        !cu(cudaMalloc(&coef, 8LL * N * D)) ||
        !cu(cudaMalloc(&part, 8LL * tiles * G * (kBmax + 1))) ||
        !cu(cudaMalloc(&info, sizeof(int)))) {
      ret = KVTC_ENOMEM;
      break;
    }
    if (cublasCreate(&blas) != CUBLAS_STATUS_SUCCESS ||
        cusolverDnCreate(&solver) != CUSOLVER_STATUS_SUCCESS ||
        cublasSetStream(blas, st) != CUBLAS_STATUS_SUCCESS ||
        cusolverDnSetStream(solver, st) != CUSOLVER_STATUS_SUCCESS) {
      ret = KVTC_ECUDA;
      break;
    }
    int lwork = 0;
    if (cusolverDnDsyevd_bufferSize(solver, CUSOLVER_EIG_MODE_VECTOR,
                                    CUBLAS_FILL_MODE_LOWER, D, cov, D, w,
                                    &lwork) != CUSOLVER_STATUS_SUCCESS ||
        !cu(cudaMalloc(&work, 8LL * std::max(lwork, 1)))) {
      ret = ret ? ret : KVTC_ECUDA;
      break;
    }
    std::vector<double> hcov((size_t)D * D), hw(D), hmu(D), hV((size_t)D * D);
    std::vector<double> hpart((size_t)tiles * G * (kBmax + 1));
    for (int i = 0; i < n && ret == KVTC_OK; ++i) {
      const uint16_t* x = static_cast<const uint16_t*>(tokens[i]);
      column_mean_kernel<<<(D + 127) / 128, 128, 0, st>>>(x, N, ld, D, mu);
      const int64_t tot = N * D;
      centre_kernel<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(x, N, ld, D,
                                                                   mu, xc);
      if (!cu(cudaGetLastError())) break;
      // covariance (column-major D x D, lower triangle) of the centred rows
      const double alpha = 1.0 / (double)N, beta = 0.0, one = 1.0;
      if (cublasDsyrk(blas, CUBLAS_FILL_MODE_LOWER, CUBLAS_OP_N, D, (int)N,
                      &alpha, xc, D, &beta, cov, D) != CUBLAS_STATUS_SUCCESS ||
          cusolverDnDsyevd(solver, CUSOLVER_EIG_MODE_VECTOR,
                           CUBLAS_FILL_MODE_LOWER, D, cov, D, w, work, lwork,
                           info) != CUSOLVER_STATUS_SUCCESS) {
        ret = KVTC_ECUDA;
        break;
      }
      int hinfo = 0;
      if (!cu(cudaMemcpyAsync(hcov.data(), cov, 8LL * D * D,
                              cudaMemcpyDeviceToHost, st)) ||
          !cu(cudaMemcpyAsync(hw.data(), w, 8LL * D, cudaMemcpyDeviceToHost,
                              st)) ||
          !cu(cudaMemcpyAsync(hmu.data(), mu, 8LL * D, cudaMemcpyDeviceToHost,
                              st)) ||
          !cu(cudaMemcpyAsync(&hinfo, info, sizeof(int),
                              cudaMemcpyDeviceToHost, st)) ||
          !cu(cudaStreamSynchronize(st)))
        break;
      if (hinfo != 0) {
        ret = KVTC_ECUDA;
        break;
      }
      // descending order; sign: largest-magnitude entry positive (first on
      // ties).  hV is column-major, column j = j-th principal vector.
      for (int j = 0; j < D; ++j) {
        const double* src = hcov.data() + (size_t)(D - 1 - j) * D;
        int arg = 0;
        for (int d = 1; d < D; ++d)
          if (std::fabs(src[d]) > std::fabs(src[arg])) arg = d;
        const double sgn = src[arg] < 0 ? -1.0 : 1.0;
        for (int d = 0; d < D; ++d) hV[(size_t)j * D + d] = sgn * src[d];
      }
      if (!cu(cudaMemcpyAsync(V, hV.data(), 8LL * D * D,
                              cudaMemcpyHostToDevice, st)))
        break;
      // coefficients, column-major D x N: coef = V^T xc
      if (cublasDgemm(blas, CUBLAS_OP_T, CUBLAS_OP_N, D, (int)N, D, &one, V,
                      D, xc, D, &beta, coef, D) != CUBLAS_STATUS_SUCCESS) {
        ret = KVTC_ECUDA;
        break;
      }
      distortion_kernel<<<dim3((unsigned)tiles, G), kTokTile, 0, st>>>(
          coef, N, D, part);
      if (!cu(cudaGetLastError()) ||
          !cu(cudaMemcpyAsync(hpart.data(), part, 8LL * hpart.size(),
                              cudaMemcpyDeviceToHost, st)) ||
          !cu(cudaStreamSynchronize(st)))
        break;
      std::vector<double> E((size_t)G * (kBmax + 1), 0.0);
      for (int64_t t = 0; t < tiles; ++t)
        for (size_t j = 0; j < E.size(); ++j)
          E[j] += hpart[(size_t)t * E.size() + j];
      const std::vector<uint8_t> widths = allocate(E, G, kBmax, budget_bits);
      int k = 0;
      for (int g = 0; g < G; ++g) k += widths[g] ? kGroupC : 0;
      out.u32((uint32_t)layers[i]);
      out.u32((uint32_t)kvs[i]);
      out.u32((uint32_t)D);
      out.u32((uint32_t)k);
      std::vector<uint8_t> wpad((G + 7) / 8 * 8, 0);
      std::copy(widths.begin(), widths.end(), wpad.begin());
      out.put(wpad.data(), wpad.size());
      out.put(hmu.data(), 8LL * D);
      for (int g = 0; g < G; ++g) {
        if (!widths[g]) continue;
        for (int j = g * kGroupC; j < (g + 1) * kGroupC; ++j)
          out.put(hV.data() + (size_t)j * D, 8LL * D);
      }
      for (int j = 0; j < D; ++j) {
        const double ev = hw[D - 1 - j];
        out.put(&ev, 8);
      }
    }
  } while (false);

  if (ret == KVTC_OK) {
    if (out.ok) {
      const uint32_t crc = kvtc::crc32_ieee(out.p, out.n);
      out.u32(crc);
      out.u32(0);
    } else {
      out.n += 8;
    }
    *blob_bytes = out.n;
    if (!out.ok) ret = KVTC_ESIZE;
  }
  if (solver) cusolverDnDestroy(solver);
  if (blas) cublasDestroy(blas);
  cudaFree(mu);
  cudaFree(xc);
  cudaFree(cov);
  cudaFree(w);
  cudaFree(V);
  cudaFree(coef);
  cudaFree(part);
  cudaFree(work);
  cudaFree(info);
  if (prev >= 0) cudaSetDevice(prev);
  return ret;
}

}  // extern "C"
