// One-time calibration on the GPU (kvtc page, technical summary 2A):
// per (layer, K|V) stream, the mean and PCA basis of calibration KV, the
// distortion of every group at every width measured with the codec's own
// quantiser, and the DP bit allocation under the budget.  Writes a
// calibration blob (format in include/kvtc.h).
//
// Arithmetic is fp64 throughout.  Mean, centring, the covariance (Gram
// matrix of the centred rows), the descending order and sign rule of the
// eigenvectors, the coefficient projection, the distortion table and the
// DP bit allocation are this library's own kernels; the symmetric
// eigensolver is cuSOLVER's divide-and-conquer routine (a one-time
// library step like a GEMM; a hand-written Jacobi iteration would be
// slower at D = 1024 and is not the hot path).
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

// fp64 tiles of 64 x 64 outputs, 256 threads, 4 x 4 outputs per thread,
// the contraction in steps of 16.
constexpr int kGT = 64;
constexpr int kGK = 16;

// Covariance of the centred rows xc [N][D] (row-major): for the tile pair
// (ti >= tj), C[i][j] = C[j][i] = alpha * sum_t xc[t][i] xc[t][j]; C is
// D x D and symmetric, so its storage order does not matter.
__global__ void __launch_bounds__(256) gram_kernel(const double* xc,
                                                   int64_t N, int D,
                                                   double alpha, double* C) {
  const int ti = blockIdx.y, tj = blockIdx.x;
  if (tj > ti) return;
  __shared__ double As[kGK][kGT + 1], Bs[kGK][kGT + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int i0 = ti * kGT, j0 = tj * kGT;
  double acc[4][4] = {};
  for (int64_t t0 = 0; t0 < N; t0 += kGK) {
    for (int e = threadIdx.x; e < kGK * kGT; e += 256) {
      const int tk = e / kGT, c = e - tk * kGT;
      const int64_t t = t0 + tk;
      As[tk][c] = (t < N && i0 + c < D) ? xc[t * D + i0 + c] : 0.0;
      Bs[tk][c] = (t < N && j0 + c < D) ? xc[t * D + j0 + c] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int tk = 0; tk < kGK; ++tk) {
      double a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = As[tk][ty * 4 + r];
        b[r] = Bs[tk][tx * 4 + r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fma(a[r], b[q], acc[r][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + ty * 4 + r, j = j0 + tx * 4 + q;
      if (i < D && j < D) {
        C[(int64_t)i * D + j] = alpha * acc[r][q];
        C[(int64_t)j * D + i] = alpha * acc[r][q];
      }
    }
}

// Eigenvectors in descending order of eigenvalue, each signed so that its
// largest-magnitude entry is positive (the first such entry on ties).
// evec: column j (contiguous, D entries) = eigenvector of the j-th smallest
// eigenvalue w[j].  Block j writes V column j (contiguous) = the (D-1-j)-th
// eigenvector times its sign, and ev[j] = w[D-1-j].
__global__ void __launch_bounds__(256) order_sign_kernel(const double* evec,
                                                         const double* w,
                                                         int D, double* V,
                                                         double* ev) {
  const int j = blockIdx.x;
  const double* src = evec + (int64_t)(D - 1 - j) * D;
  __shared__ double sv[256];
  __shared__ int si[256];
  double best = -1.0;
  int arg = D;
  for (int d = threadIdx.x; d < D; d += 256) {
    const double a = fabs(src[d]);
    if (a > best) {  // d ascends within a thread: ties keep the first
      best = a;
      arg = d;
    }
  }
  sv[threadIdx.x] = best;
  si[threadIdx.x] = arg;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) {
      const double ob = sv[threadIdx.x + s];
      const int oi = si[threadIdx.x + s];
      if (ob > sv[threadIdx.x] || (ob == sv[threadIdx.x] && oi < si[threadIdx.x])) {
        sv[threadIdx.x] = ob;
        si[threadIdx.x] = oi;
      }
    }
    __syncthreads();
  }
  const double sgn = src[si[0]] < 0.0 ? -1.0 : 1.0;
  for (int d = threadIdx.x; d < D; d += 256)
    V[(int64_t)j * D + d] = sgn * src[d];
  if (threadIdx.x == 0) ev[j] = w[D - 1 - j];
}

// Coefficients of every component: coef[t][j] = sum_d xc[t][d] V[d][j],
// xc [N][D] row-major, V stored by columns (column j contiguous).
__global__ void __launch_bounds__(256) project_kernel(const double* xc,
                                                      int64_t N, int D,
                                                      const double* V,
                                                      double* coef) {
  __shared__ double As[kGK][kGT + 1], Bs[kGK][kGT + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t r0 = (int64_t)blockIdx.y * kGT;
  const int j0 = blockIdx.x * kGT;
  double acc[4][4] = {};
  for (int d0 = 0; d0 < D; d0 += kGK) {
    for (int e = threadIdx.x; e < kGK * kGT; e += 256) {
      const int c = e / kGK, dk = e - c * kGK;  // dk fastest: contiguous d
      const int d = d0 + dk;
      const int64_t t = r0 + c;
      As[dk][c] = (t < N && d < D) ? xc[t * D + d] : 0.0;
      Bs[dk][c] = (j0 + c < D && d < D) ? V[(int64_t)(j0 + c) * D + d] : 0.0;
    }
    __syncthreads();
#pragma unroll
    for (int dk = 0; dk < kGK; ++dk) {
      double a[4], b[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        a[r] = As[dk][ty * 4 + r];
        b[r] = Bs[dk][tx * 4 + r];
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = fma(a[r], b[q], acc[r][q]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t t = r0 + ty * 4 + r;
      const int j = j0 + tx * 4 + q;
      if (t < N && j < D) coef[t * D + j] = acc[r][q];
    }
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

// Distortion table E[g][b] = sum over the token tiles of part[tile][g][b].
__global__ void distortion_sum_kernel(const double* part, int64_t tiles,
                                      int G, double* E) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= G * (kBmax + 1)) return;
  double s = 0.0;
  for (int64_t t = 0; t < tiles; ++t) s += part[t * G * (kBmax + 1) + i];
  E[i] = s;
}

__device__ __forceinline__ int cost_units(int b) { return b == 0 ? 0 : 2 + b; }

// DP over groups (one block): F[g][u] = least summed distortion of the
// first g groups within u units of 16 bits, choosing b = 0 .. bmax in
// ascending order with strict improvement only (ties keep the smaller
// width); then the widths by backtracking from u = U.  No allocation
// exceeds 10 units per group, so u is capped at 10 G: for larger u every
// F[g][u] equals F[g][10 g] and every choice equals the one there, so the
// widths are the same as with the full budget.  F: 2 x (U + 1) doubles of
// scratch, choice: G x (U + 1) bytes.
__global__ void __launch_bounds__(256) dp_kernel(const double* E, int G,
                                                 int bmax, int U, double* F,
                                                 uint8_t* choice,
                                                 uint8_t* widths) {
  double* prev = F;
  double* cur = F + (U + 1);
  for (int u = threadIdx.x; u <= U; u += 256) prev[u] = 0.0;
  __syncthreads();
  for (int g = 1; g <= G; ++g) {
    for (int u = threadIdx.x; u <= U; u += 256) {
      double best = INFINITY;
      int bb = 0;
      for (int b = 0; b <= bmax; ++b) {
        const int cu = cost_units(b);
        if (cu > u) break;
        const double v = prev[u - cu] + E[(g - 1) * (kBmax + 1) + b];
        if (v < best) {
          best = v;
          bb = b;
        }
      }
      cur[u] = best;
      choice[(int64_t)(g - 1) * (U + 1) + u] = (uint8_t)bb;
    }
    __syncthreads();
    double* t = prev;
    prev = cur;
    cur = t;
  }
  if (threadIdx.x == 0) {
    int u = U;
    for (int g = G; g >= 1; --g) {
      const int b = choice[(int64_t)(g - 1) * (U + 1) + u];
      widths[g - 1] = (uint8_t)b;
      u -= cost_units(b);
    }
  }
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
  // DP units: the budget's, capped where no allocation reaches (10 per group)
  const int U = std::min(budget_bits / 16, 10 * G);

  double *mu = nullptr, *xc = nullptr, *cov = nullptr, *w = nullptr,
         *V = nullptr, *ev = nullptr, *coef = nullptr, *part = nullptr,
         *E = nullptr, *F = nullptr, *work = nullptr;
  uint8_t *choice = nullptr, *dwidths = nullptr;
  int* info = nullptr;
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
        !cu(cudaMalloc(&V, 8LL * D * D)) || !cu(cudaMalloc(&ev, 8LL * D)) ||
        !cu(cudaMalloc(&coef, 8LL * N * D)) ||
        !cu(cudaMalloc(&part, 8LL * tiles * G * (kBmax + 1))) ||
        !cu(cudaMalloc(&E, 8LL * G * (kBmax + 1))) ||
        !cu(cudaMalloc(&F, 16LL * (U + 1))) ||
        !cu(cudaMalloc(&choice, (size_t)G * (U + 1))) ||
        !cu(cudaMalloc(&dwidths, (size_t)G)) ||
        !cu(cudaMalloc(&info, sizeof(int)))) {
      ret = KVTC_ENOMEM;
      break;
    }
    if (cusolverDnCreate(&solver) != CUSOLVER_STATUS_SUCCESS ||
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
    std::vector<double> hmu(D), hev(D), hV;
    std::vector<uint8_t> widths(G);
    const int nt = (D + kGT - 1) / kGT;
    for (int i = 0; i < n && ret == KVTC_OK; ++i) {
      const uint16_t* x = static_cast<const uint16_t*>(tokens[i]);
      column_mean_kernel<<<(D + 127) / 128, 128, 0, st>>>(x, N, ld, D, mu);
      const int64_t tot = N * D;
      centre_kernel<<<(unsigned)((tot + 255) / 256), 256, 0, st>>>(x, N, ld, D,
                                                                   mu, xc);
      // covariance (symmetric D x D) of the centred rows
      gram_kernel<<<dim3(nt, nt), 256, 0, st>>>(xc, N, D, 1.0 / (double)N,
                                                cov);
      if (!cu(cudaGetLastError())) break;
      if (cusolverDnDsyevd(solver, CUSOLVER_EIG_MODE_VECTOR,
                           CUBLAS_FILL_MODE_LOWER, D, cov, D, w, work, lwork,
                           info) != CUSOLVER_STATUS_SUCCESS) {
        ret = KVTC_ECUDA;
        break;
      }
      // descending order and sign rule; coefficients of every component;
      // distortion table; DP widths
      order_sign_kernel<<<D, 256, 0, st>>>(cov, w, D, V, ev);
      project_kernel<<<dim3(nt, (unsigned)((N + kGT - 1) / kGT)), 256, 0,
                       st>>>(xc, N, D, V, coef);
      distortion_kernel<<<dim3((unsigned)tiles, G), kTokTile, 0, st>>>(
          coef, N, D, part);
      distortion_sum_kernel<<<(G * (kBmax + 1) + 127) / 128, 128, 0, st>>>(
          part, tiles, G, E);
      dp_kernel<<<1, 256, 0, st>>>(E, G, kBmax, U, F, choice, dwidths);
      int hinfo = 0;
      if (!cu(cudaGetLastError()) ||
          !cu(cudaMemcpyAsync(hmu.data(), mu, 8LL * D, cudaMemcpyDeviceToHost,
                              st)) ||
          !cu(cudaMemcpyAsync(hev.data(), ev, 8LL * D, cudaMemcpyDeviceToHost,
                              st)) ||
          !cu(cudaMemcpyAsync(widths.data(), dwidths, (size_t)G,
                              cudaMemcpyDeviceToHost, st)) ||
          !cu(cudaMemcpyAsync(&hinfo, info, sizeof(int),
                              cudaMemcpyDeviceToHost, st)) ||
          !cu(cudaStreamSynchronize(st)))
        break;
      if (hinfo != 0) {
        ret = KVTC_ECUDA;
        break;
      }
      // the kept principal vectors: per active group its 16 columns of V
      int k = 0;
      for (int g = 0; g < G; ++g) k += widths[g] ? kGroupC : 0;
      hV.resize((size_t)k * D);
      int a = 0;
      for (int g = 0; g < G && ret == KVTC_OK; ++g) {
        if (!widths[g]) continue;
        cu(cudaMemcpyAsync(hV.data() + (size_t)a * D,
                           V + (size_t)g * kGroupC * D, 8LL * kGroupC * D,
                           cudaMemcpyDeviceToHost, st));
        a += kGroupC;
      }
      if (!cu(cudaStreamSynchronize(st))) break;
      out.u32((uint32_t)layers[i]);
      out.u32((uint32_t)kvs[i]);
      out.u32((uint32_t)D);
      out.u32((uint32_t)k);
      std::vector<uint8_t> wpad((G + 7) / 8 * 8, 0);
      std::copy(widths.begin(), widths.end(), wpad.begin());
      out.put(wpad.data(), wpad.size());
      out.put(hmu.data(), 8LL * D);
      out.put(hV.data(), 8LL * k * D);
      out.put(hev.data(), 8LL * D);
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
  cudaFree(mu);
  cudaFree(xc);
  cudaFree(cov);
  cudaFree(w);
  cudaFree(V);
  cudaFree(ev);
  cudaFree(coef);
  cudaFree(part);
  cudaFree(E);
  cudaFree(F);
  cudaFree(choice);
  cudaFree(dwidths);
  cudaFree(work);
  cudaFree(info);
  if (prev >= 0) cudaSetDevice(prev);
  return ret;
}

}  // extern "C"
