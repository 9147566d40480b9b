// Lossless field packing of codec streams: kernels and launchers.
//
// The kvtc page ("KV Cache Transform Coding for Compact Storage in LLM
// Inference", technical summary 2B) runs a lossless entropy stage after
// bit-packing.  This stage is our own: in each record only the high byte of
// every fp16 field (sign, exponent, two mantissa bits) carries redundancy,
// so its sign and exponent are stored as an offset from the stream's
// minimum for that field, in as many bits as the stream's range needs.
// The format is documented in include/kvtc.h.
//
// Pack, per launch group of streams:
//   fp_minmax_kernel  grid (kFpChunks, n): bytewise min / max of every
//                     field word over a chunk of each stream's records;
//   fp_layout_kernel  one block: per stream the slot table (vmin, dbits),
//                     the packed record size Rp and stream size; an
//                     exclusive scan gives the stream offsets; headers,
//                     tables and offsets are written;
//   fp_pack_kernel    persistent: raw-row chunks are copied, record tiles of
//                     128 tokens are bulk-loaded into shared memory, one
//                     warp packs one token at a time (lane s = field slot s,
//                     the slots' codes merged with warp OR-reductions), and
//                     the tile is bulk-stored.
// Unpack is one persistent kernel of the same shape that checks each
// stream's header against its calibration and offsets, then reverses the
// tile transform.
//
// Both tile kernels are HBM-bound byte shuffles; the per-token work is a
// few dozen instructions per warp, hidden behind three resident blocks per
// SM.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"
#include "ptx.cuh"

namespace kvtc {
namespace {

static_assert(kFpChunks == 8, "layout pass reads 8 chunks x 4 lanes");
static_assert(kMaxK / 16 <= 15, "at most 30 field slots (one warp)");
constexpr int kFpThreads = 256;
constexpr int kFpWarps = kFpThreads / 32;
constexpr int kFpLayoutThreads = 1024;
constexpr uint32_t kFpMagic = 0x5046564Bu;  // "KVFP", little-endian
constexpr int kFpInBytes = kFpTile * kMaxRecord;
constexpr int kFpOutBytes = kFpTile * kMaxRecord + 256;
constexpr int kFpSmem = kFpInBytes + kFpOutBytes + 16;  // + read slack

__device__ __forceinline__ int fp_table_bytes(int ga) {
  return (4 * ga + 15) & ~15;
}
__device__ __forceinline__ int64_t fp_align256(int64_t v) {
  return (v + 255) & ~int64_t(255);
}

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Stream of a work item: the last stream whose first item is <= item.
__device__ __forceinline__ int fp_find_stream(const FpParams& p, int item) {
  int lo = 0, hi = p.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.s[mid].item_begin <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Copy bytes [b0, b1) (16-byte multiples) with the whole block.
__device__ __forceinline__ void fp_block_copy(uint8_t* dst, const uint8_t* src,
                                              int64_t bytes) {
  const int64_t n = bytes >> 4;
  for (int64_t c = threadIdx.x; c < n; c += blockDim.x)
    reinterpret_cast<uint4*>(dst)[c] = ldg_nc(src + 16 * c);
}
__device__ __forceinline__ void fp_block_zero(uint8_t* dst, int64_t bytes) {
  const int64_t n = bytes >> 4;
  for (int64_t c = threadIdx.x; c < n; c += blockDim.x)
    reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
}

// Per-lane slot description: lane s < 2 G_a holds slot s's vmin, dbits and
// the bit position of its code; the warp also learns the code bits.
struct FpSlots {
  int vmin, d, pos, hbits;
};
__device__ __forceinline__ FpSlots fp_slots_from(int vmin, int d, int nslot) {
  const int lane = threadIdx.x & 31;
  const int w = lane < nslot ? d + 2 : 0;
  int incl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  FpSlots r;
  r.vmin = vmin;
  r.d = d;
  r.pos = incl - w;
  r.hbits = __shfl_sync(0xffffffffu, incl, 31);
  return r;
}

// ------------------------------------------------------------- pack pass 1
__global__ void __launch_bounds__(kFpThreads) fp_minmax_kernel(
    const __grid_constant__ FpParams p) {
  __shared__ uint32_t red[kFpWarps][kFpWorkWords];
  const int i = blockIdx.y, c = blockIdx.x;
  const FpStream& S = p.s[i];
  const int per = (S.tc + kFpChunks - 1) / kFpChunks;
  const int t0 = c * per;
  const int t1 = min(S.tc, t0 + per);
  const int nv = (S.ga + 3) >> 2;
  const uint8_t* rec = p.in + S.in_off + S.raw_bytes;
  uint32_t mn[16], mx[16];
#pragma unroll
  for (int a = 0; a < 16; ++a) {
    mn[a] = 0xffffffffu;
    mx[a] = 0u;
  }
  for (int t = t0 + (int)threadIdx.x; t < t1; t += kFpThreads) {
    const uint8_t* r = rec + (int64_t)t * S.R;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      if (v < nv) {
        const uint4 q = ldg_nc(r + 16 * v);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          mn[4 * v + e] = __vminu4(mn[4 * v + e], w[e]);
          mx[4 * v + e] = __vmaxu4(mx[4 * v + e], w[e]);
        }
      }
    }
  }
#pragma unroll
  for (int a = 0; a < 16; ++a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mn[a] = __vminu4(mn[a], __shfl_xor_sync(0xffffffffu, mn[a], o));
      mx[a] = __vmaxu4(mx[a], __shfl_xor_sync(0xffffffffu, mx[a], o));
    }
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
#pragma unroll
    for (int a = 0; a < 16; ++a) {
      red[warp][a] = mn[a];
      red[warp][16 + a] = mx[a];
    }
  }
  __syncthreads();
  if (threadIdx.x < kFpWorkWords) {
    const int a = threadIdx.x;
    uint32_t v = red[0][a];
    for (int w = 1; w < kFpWarps; ++w)
      v = a < 16 ? __vminu4(v, red[w][a]) : __vmaxu4(v, red[w][a]);
    p.work[((int64_t)i * kFpChunks + c) * kFpWorkWords + a] = v;
  }
}

// ------------------------------------------------------------- pack pass 2
// One block of 1024 threads: warp w handles streams w, w + 32, ...
__global__ void __launch_bounds__(kFpLayoutThreads) fp_layout_kernel(
    const __grid_constant__ FpParams p) {
  __shared__ int64_t size[kFpMaxStream];
  __shared__ int64_t excl[kFpMaxStream];
  __shared__ uint16_t table[kFpMaxStream][32];  // vmin | dbits << 8
  __shared__ int64_t base;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < p.n; i += kFpLayoutThreads / 32) {
    const FpStream& S = p.s[i];
    const int nslot = 2 * S.ga;
    // lane = chunk * 4 + q: q 0/1 min words [8q, 8q + 8), q 2/3 max words
    const int ch = lane >> 2, q = lane & 3;
    const uint32_t* src = p.work +
                          ((int64_t)i * kFpChunks + ch) * kFpWorkWords + 8 * q;
    const uint4 a = *reinterpret_cast<const uint4*>(src);
    const uint4 b = *reinterpret_cast<const uint4*>(src + 4);
    uint32_t r[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t v = __shfl_xor_sync(0xffffffffu, r[e], o);
        r[e] = q < 2 ? __vminu4(r[e], v) : __vmaxu4(r[e], v);
      }
    // slot s = lane: field word s >> 1, byte 1 (shift) or 3 (scale)
    const int fw = lane >> 1;
    uint32_t wmin = 0, wmax = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t v0 = __shfl_sync(0xffffffffu, r[e], fw >> 3);
      const uint32_t v1 = __shfl_sync(0xffffffffu, r[e], 2 + (fw >> 3));
      if ((fw & 7) == e) {
        wmin = v0;
        wmax = v1;
      }
    }
    const int sh = 8 + 16 * (lane & 1);
    int vmin = 0, d = 0;
    if (S.tc > 0 && lane < nslot) {
      vmin = (int)((wmin >> sh) & 0xffu) >> 2;
      const int vmax = (int)((wmax >> sh) & 0xffu) >> 2;
      d = 32 - __clz(vmax - vmin);
    }
    const FpSlots sl = fp_slots_from(vmin, d, nslot);
    const int hb2 = (sl.hbits + 15) >> 4;
    const int rp = 2 * S.ga + 2 * hb2 + (S.used - 4 * S.ga);
    table[i][lane] = (uint16_t)(vmin | (d << 8));
    if (lane == 0)
      size[i] = fp_align256(kFpHeader + fp_table_bytes(S.ga) + S.raw_bytes +
                            (int64_t)S.tc * rp);
  }
  if (threadIdx.x == 0) base = p.first == 0 ? 0 : p.offsets[p.first];
  __syncthreads();
  // exclusive scan of the sizes (n <= 256): warp 0, eight per lane
  if (warp == 0) {
    int64_t v[8], run = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = lane * 8 + e;
      v[e] = i < p.n ? size[i] : 0;
      run += v[e];
    }
    int64_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int64_t acc = base + incl - run;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = lane * 8 + e;
      if (i < p.n) excl[i] = acc;
      acc += v[e];
    }
  }
  __syncthreads();
  for (int i = warp; i < p.n; i += kFpLayoutThreads / 32) {
    const FpStream& S = p.s[i];
    const int64_t off = excl[i];
    uint8_t* o = p.out + off;
    const int tb = fp_table_bytes(S.ga);
    int hbits = 0;
    const int nslot = 2 * S.ga;
    if (lane < nslot) hbits = (table[i][lane] >> 8) + 2;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1)
      hbits += __shfl_xor_sync(0xffffffffu, hbits, k);
    const int rp = 2 * S.ga + 2 * ((hbits + 15) >> 4) + (S.used - 4 * S.ga);
    if (lane == 0) {
      uint32_t* h = reinterpret_cast<uint32_t*>(o);
      h[0] = kFpMagic;
      h[1] = (uint32_t)S.tc;
      h[2] = (uint32_t)rp | ((uint32_t)nslot << 16);
      h[3] = 0u;
      p.offsets[p.first + i + 1] = off + size[i];
      if (p.first == 0 && i == 0) p.offsets[0] = 0;
    }
    uint16_t* t = reinterpret_cast<uint16_t*>(o + kFpHeader);
    if (lane < tb / 2) t[lane] = lane < nslot ? table[i][lane] : 0;
    if (S.tc == 0 && S.raw_bytes == 0) {  // nothing else: pad here
      const int64_t from = kFpHeader + tb;
      for (int64_t b = from + 4 * lane; b < size[i]; b += 128)
        *reinterpret_cast<uint32_t*>(o + b) = 0u;
    }
  }
}

// ------------------------------------------------------------- pack pass 3
__global__ void __launch_bounds__(kFpThreads, 3) fp_pack_kernel(
    const __grid_constant__ FpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_in = smem;
  uint8_t* s_out = smem + kFpInBytes;
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  bool bad = false;
  for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
    const int i = fp_find_stream(p, item);
    const FpStream& S = p.s[i];
    const int local = item - S.item_begin;
    const int ga = S.ga, tb = fp_table_bytes(ga);
    const int64_t off = p.offsets[p.first + i];
    const int64_t end = p.offsets[p.first + i + 1];
    uint8_t* body = p.out + off + kFpHeader + tb;  // raw rows, then records
    if (local < S.nraw) {
      const int64_t b0 = (int64_t)local * kFpRawChunk;
      const int64_t b1 = min(S.raw_bytes, b0 + kFpRawChunk);
      fp_block_copy(body + b0, p.in + S.in_off + b0, b1 - b0);
      if (S.tc == 0 && local == S.nraw - 1)
        fp_block_zero(body + S.raw_bytes, end - (off + kFpHeader + tb) -
                                              S.raw_bytes);
      continue;
    }
    const int tile = local - S.nraw;
    const int t0 = tile * kFpTile;
    const int ntok = min(kFpTile, S.tc - t0);
    const int R = S.R, nslot = 2 * ga;
    // slot table from this stream's header (written by the layout pass)
    int vmin = 0, d = 0;
    if (lane < nslot) {
      const uint16_t e =
          reinterpret_cast<const uint16_t*>(p.out + off + kFpHeader)[lane];
      vmin = e & 0xff;
      d = e >> 8;
    }
    const FpSlots sl = fp_slots_from(vmin, d, nslot);
    const int hb2 = (sl.hbits + 15) >> 4;
    const int rp = 2 * ga + 2 * hb2 + (S.used - 4 * ga);
    const int p2 = (S.used - 4 * ga) >> 1;
    const int nw = (sl.hbits + 31) >> 5;
    uint8_t* gdst = body + S.raw_bytes + (int64_t)t0 * rp;
    const int len = tile == S.ntiles - 1 ? (int)(p.out + end - gdst)
                                         : ntok * rp;
    // the previous tile's store has read s_out; everyone is done with s_in
    if (tid == 0) bulk_wait_read<0>();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)(ntok * R);
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(s_in, p.in + S.in_off + S.raw_bytes + (int64_t)t0 * R, bytes,
               &bar);
    }
    for (int b = ntok * rp + tid; b < len; b += kFpThreads) s_out[b] = 0;
    const bool ok = mbar_wait(&bar, phase, &abort_flag);
    phase ^= 1u;
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(p.status, KVTC_FLAG_TIMEOUT);
        mbar_drain(&bar, phase ^ 1u);
      }
      break;
    }
    for (int tok = warp; tok < ntok; tok += kFpWarps) {
      const uint32_t* in32 = reinterpret_cast<const uint32_t*>(s_in + tok * R);
      uint8_t* ob = s_out + tok * rp;
      uint16_t* o16 = reinterpret_cast<uint16_t*>(ob);
      uint32_t clo = 0, chi = 0;
      int w0 = -2;
      if (lane < nslot) {
        const uint32_t w = in32[lane >> 1];
        const int sh = 16 * (lane & 1);
        const uint32_t lo = (w >> sh) & 0xffu, hi = (w >> (sh + 8)) & 0xffu;
        ob[lane] = (uint8_t)lo;
        const int u = (int)(hi >> 2) - sl.vmin;
        if (u < 0 || u >= (1 << sl.d)) bad = true;
        const uint32_t code = ((uint32_t)u & ((1u << sl.d) - 1)) |
                              ((hi & 3u) << sl.d);
        w0 = sl.pos >> 5;
        const int s5 = sl.pos & 31;
        clo = code << s5;
        chi = s5 ? code >> (32 - s5) : 0u;
      }
      uint32_t mine = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        if (w < nw) {
          const uint32_t v = __reduce_or_sync(
              0xffffffffu, (w0 == w ? clo : 0u) | (w0 + 1 == w ? chi : 0u));
          if ((lane >> 1) == w) mine = v;
        }
      }
      if (lane < hb2) o16[ga + lane] = (uint16_t)(mine >> (16 * (lane & 1)));
      const uint16_t* i16 =
          reinterpret_cast<const uint16_t*>(s_in + tok * R) + 2 * ga;
      uint16_t* q16 = o16 + ga + hb2;
      for (int j = lane; j < p2; j += 32) q16[j] = i16[j];
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(gdst, s_out, (uint32_t)len);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait<0>();
  if (bad) atomicOr(p.status, KVTC_FLAG_FORMAT);
}

// ------------------------------------------------------------------ unpack
__global__ void __launch_bounds__(kFpThreads, 3) fp_unpack_kernel(
    const __grid_constant__ FpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_in = smem;
  uint8_t* s_out = smem + kFpInBytes;
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  for (int item = blockIdx.x; item < p.total_items; item += gridDim.x) {
    const int i = fp_find_stream(p, item);
    const FpStream& S = p.s[i];
    const int local = item - S.item_begin;
    const int ga = S.ga, tb = fp_table_bytes(ga), nslot = 2 * ga;
    const int64_t off = p.offsets[p.first + i];
    const int64_t end = p.offsets[p.first + i + 1];
    // the header is read only once the offsets are known to frame it
    bool ok = off >= 0 && (off & 15) == 0 && end <= p.in_bytes &&
              end - off >= kFpHeader + tb;
    int vmin = 0, d = 0, rp = 0;
    FpSlots sl = {0, 0, 0, 0};
    if (ok) {
      const uint32_t* h = reinterpret_cast<const uint32_t*>(p.in + off);
      const uint32_t h0 = h[0], h1 = h[1], h2 = h[2];
      if (lane < nslot) {
        const uint16_t e =
            reinterpret_cast<const uint16_t*>(p.in + off + kFpHeader)[lane];
        vmin = e & 0xff;
        d = e >> 8;
      }
      const bool slot_ok = lane >= nslot || (d <= 6 && vmin <= 63);
      sl = fp_slots_from(vmin, d, nslot);
      rp = 2 * ga + 2 * ((sl.hbits + 15) >> 4) + (S.used - 4 * ga);
      ok = __all_sync(0xffffffffu, slot_ok) && h0 == kFpMagic &&
           h1 == (uint32_t)S.tc && (h2 & 0xffffu) == (uint32_t)rp &&
           (h2 >> 16) == (uint32_t)nslot &&
           end - off == fp_align256(kFpHeader + tb + S.raw_bytes +
                                    (int64_t)S.tc * rp);
    }
    if (!ok) {
      if (tid == 0) atomicOr(p.status, KVTC_FLAG_FORMAT);
      continue;
    }
    const uint8_t* body = p.in + off + kFpHeader + tb;
    uint8_t* obase = p.out + S.out_off;
    const int64_t out_end =
        S.out_off + fp_align256(S.raw_bytes + (int64_t)S.tc * S.R);
    if (local < S.nraw) {
      const int64_t b0 = (int64_t)local * kFpRawChunk;
      const int64_t b1 = min(S.raw_bytes, b0 + kFpRawChunk);
      fp_block_copy(obase + b0, body + b0, b1 - b0);
      if (S.tc == 0 && local == S.nraw - 1)
        fp_block_zero(obase + S.raw_bytes, out_end - S.out_off - S.raw_bytes);
      continue;
    }
    const int tile = local - S.nraw;
    const int t0 = tile * kFpTile;
    const int ntok = min(kFpTile, S.tc - t0);
    const int R = S.R, R2 = R >> 1, u2 = S.used >> 1;
    const int hb2 = (sl.hbits + 15) >> 4;
    uint8_t* gdst = obase + S.raw_bytes + (int64_t)t0 * R;
    const int len = tile == S.ntiles - 1 ? (int)(p.out + out_end - gdst)
                                         : ntok * R;
    if (tid == 0) bulk_wait_read<0>();
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)((ntok * rp + 15) & ~15);
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(s_in, body + S.raw_bytes + (int64_t)t0 * rp, bytes, &bar);
    }
    for (int b = ntok * R + tid; b < len; b += kFpThreads) s_out[b] = 0;
    const bool got = mbar_wait(&bar, phase, &abort_flag);
    phase ^= 1u;
    if (__syncthreads_or(!got)) {
      if (tid == 0) {
        atomicOr(p.status, KVTC_FLAG_TIMEOUT);
        mbar_drain(&bar, phase ^ 1u);
      }
      break;
    }
    for (int tok = warp; tok < ntok; tok += kFpWarps) {
      const uint8_t* ib = s_in + tok * rp;
      const uint16_t* i16 = reinterpret_cast<const uint16_t*>(ib);
      uint16_t* o16 = reinterpret_cast<uint16_t*>(s_out + tok * R);
      if (lane < nslot) {
        const int k = sl.pos >> 4;
        const uint32_t bits =
            (uint32_t)i16[ga + k] | ((uint32_t)i16[ga + k + 1] << 16);
        const uint32_t code = (bits >> (sl.pos & 15)) & ((4u << sl.d) - 1);
        const uint32_t u = code & ((1u << sl.d) - 1), m2 = code >> sl.d;
        const uint32_t hi = (((u + sl.vmin) << 2) | m2) & 0xffu;
        o16[lane] = (uint16_t)(ib[lane] | (hi << 8));
      }
      for (int j = 2 * ga + lane; j < R2; j += 32)
        o16[j] = j < u2 ? i16[hb2 - ga + j] : (uint16_t)0;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      bulk_s2g(gdst, s_out, (uint32_t)len);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait<0>();
}

int fp_blocks(int items) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int cap = 3 * (sms > 0 ? sms : 1);
  return items < cap ? (items > 0 ? items : 1) : cap;
}

}  // namespace

cudaError_t launch_fields_pack(const FpParams& p, cudaStream_t st) {
  if (p.n == 0) return cudaSuccess;
  fp_minmax_kernel<<<dim3(kFpChunks, p.n), kFpThreads, 0, st>>>(p);
  count_launch();
  fp_layout_kernel<<<1, kFpLayoutThreads, 0, st>>>(p);
  count_launch();
  if (p.total_items > 0) {
    cudaFuncSetAttribute((const void*)fp_pack_kernel,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, kFpSmem);
    fp_pack_kernel<<<fp_blocks(p.total_items), kFpThreads, kFpSmem, st>>>(p);
    count_launch();
  }
  return cudaGetLastError();
}

cudaError_t launch_fields_unpack(const FpParams& p, cudaStream_t st) {
  if (p.n == 0 || p.total_items == 0) return cudaSuccess;
  cudaFuncSetAttribute((const void*)fp_unpack_kernel,
                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFpSmem);
  fp_unpack_kernel<<<fp_blocks(p.total_items), kFpThreads, kFpSmem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvtc
