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
//   fp_tile_kernel<true>  persistent: raw-row chunks are copied, record
//                     tiles of up to 32 KB are bulk-loaded into shared
//                     memory, each warp packs four tokens per step (lane s =
//                     field slot s, the slots' codes merged with warp
//                     OR-reductions), and the tile is bulk-stored.
// Unpack is fp_tile_kernel<false>, the same pipeline, which checks each
// stream's header against its calibration and offsets and then reverses
// the tile transform.
//
// Each block keeps two 32 KB loads in flight ahead of the tile it
// transforms, so memory latency is hidden; what bounds both directions is
// the per-token instruction count of the transform (about 50 warp
// instructions per token to unpack, 100 to pack), not HBM.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"
#include "ptx.cuh"

namespace kvtc {
namespace {

static_assert(kFpChunks == 8, "layout pass reads 8 chunks x 4 lanes");
static_assert(kNarrowK / 16 <= 15, "at most 30 field slots (one warp)");
constexpr int kFpThreads = 256;
constexpr int kFpWarps = kFpThreads / 32;
constexpr int kFpLayoutThreads = 1024;
constexpr int kFpBuf = kFpRawChunk;              // one input buffer
constexpr int kFpSmem = 3 * kFpBuf + 256 + 16;   // 2 in, 1 out + padding

__device__ __forceinline__ int fp_table_bytes(int ga) {
  return fp_prefix_bytes(ga) - kFpHeader;
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
    const int rp = fp_record_bytes(S.ga, hb2, S.used);
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
    const int rp = fp_record_bytes(S.ga, (hbits + 15) >> 4, S.used);
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
    for (int j = lane; j < tb / 2; j += 32)
      t[j] = j < nslot ? table[i][j] : 0;
    if (S.tc == 0 && S.raw_bytes == 0) {  // nothing else: pad here
      const int64_t from = kFpHeader + tb;
      for (int64_t b = from + 4 * lane; b < size[i]; b += 128)
        *reinterpret_cast<uint32_t*>(o + b) = 0u;
    }
  }
}

// ---------------------------------------------------- pack pass 3, unpack
// One persistent kernel for both directions.  Block b takes a contiguous
// range of work items; warp 0 resolves items (the stream's header is read
// once per stream) and bulk-loads each into one of two input buffers two
// items ahead of the block; all warps then transform a record tile into the
// output buffer and one thread bulk-stores it.  A raw-row chunk goes out of
// its input buffer unchanged.
struct FpInfo {
  const uint8_t* gsrc;    // bulk-load source
  uint8_t* gdst;          // bulk-store destination
  uint8_t* zero_dst;      // stream padding to clear after raw rows (or null)
  int32_t kind;           // 0 skip, 1 raw chunk, 2 record tile
  int32_t load_bytes;
  int32_t store_bytes;    // tile: packed / codec bytes plus trailing padding
  int32_t zero_bytes;
  int32_t ntok, ga, used, R, rp, hb2;
  uint16_t table[32];     // slot s: vmin | dbits << 8
};

template <bool kPack>
__global__ void __launch_bounds__(kFpThreads, 2) fp_tile_kernel(
    const __grid_constant__ FpParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_out = smem + 2 * kFpBuf;
  __shared__ uint64_t full[2];
  __shared__ FpInfo info[2];
  __shared__ int abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nb = gridDim.x, bid = blockIdx.x;
  const int q = p.total_items / nb, r = p.total_items % nb;
  const int ib = bid * q + min(bid, r);
  const int ie = ib + q + (bid < r ? 1 : 0);
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---- producer state (warp 0): the stream whose header it holds
  int c_i = -1, c_rp = 0, c_hb2 = 0;
  int64_t c_off = 0, c_end = 0;
  bool c_ok = false;
  uint32_t c_tab = 0;
  auto produce = [&](int j, int bsel) {
    const int i = fp_find_stream(p, j);
    const FpStream& S = p.s[i];
    const int ga = S.ga, nslot = 2 * ga, tb = fp_table_bytes(ga);
    if (i != c_i) {
      c_i = i;
      c_off = p.offsets[p.first + i];
      c_end = p.offsets[p.first + i + 1];
      const uint8_t* hbase = kPack ? p.out : p.in;
      // unpack: read the header only once the offsets are known to frame it
      c_ok = kPack || (c_off >= 0 && (c_off & 15) == 0 &&
                       c_end <= p.in_bytes && c_end - c_off >= kFpHeader + tb);
      int vmin = 0, d = 0;
      c_tab = 0;
      if (c_ok) {
        if (lane < nslot) {
          c_tab = reinterpret_cast<const uint16_t*>(hbase + c_off +
                                                    kFpHeader)[lane];
          vmin = c_tab & 0xff;
          d = c_tab >> 8;
        }
        const FpSlots sl = fp_slots_from(vmin, d, nslot);
        c_hb2 = (sl.hbits + 15) >> 4;
        c_rp = fp_record_bytes(ga, c_hb2, S.used);
        if (!kPack) {
          const uint32_t* h = reinterpret_cast<const uint32_t*>(p.in + c_off);
          const uint32_t h0 = h[0], h1 = h[1], h2 = h[2];
          const bool slot_ok = lane >= nslot || (d <= 6 && vmin <= 63);
          c_ok = __all_sync(0xffffffffu, slot_ok) && h0 == kFpMagic &&
                 h1 == (uint32_t)S.tc && (h2 & 0xffffu) == (uint32_t)c_rp &&
                 (h2 >> 16) == (uint32_t)nslot &&
                 c_end - c_off == fp_align256(kFpHeader + tb + S.raw_bytes +
                                              (int64_t)S.tc * c_rp);
          if (!c_ok && lane == 0) atomicOr(p.status, KVTC_FLAG_FORMAT);
        }
      }
    }
    const int local = j - S.item_begin;
    // byte positions of this stream in the packed and the codec buffers
    const int64_t pbody = c_off + kFpHeader + tb;    // raw rows, then records
    const int64_t cbody = kPack ? S.in_off : S.out_off;
    const int64_t cend = cbody + fp_align256(S.raw_bytes + (int64_t)S.tc * S.R);
    const uint8_t* pin = p.in;
    uint8_t* pout = p.out;
    FpInfo inf;
    inf.zero_dst = nullptr;
    inf.zero_bytes = 0;
    inf.ntok = 0;
    inf.ga = ga;
    inf.used = S.used;
    inf.R = S.R;
    inf.rp = c_rp;
    inf.hb2 = c_hb2;
    if (!c_ok) {
      inf.kind = 0;
      inf.load_bytes = inf.store_bytes = 0;
      inf.gsrc = nullptr;
      inf.gdst = nullptr;
    } else if (local < S.nraw) {
      const int64_t b0 = (int64_t)local * kFpRawChunk;
      const int64_t b1 = min(S.raw_bytes, b0 + kFpRawChunk);
      inf.kind = 1;
      inf.load_bytes = inf.store_bytes = (int32_t)(b1 - b0);
      inf.gsrc = kPack ? pin + cbody + b0 : pin + pbody + b0;
      inf.gdst = kPack ? pout + pbody + b0 : pout + cbody + b0;
      if (S.tc == 0 && local == S.nraw - 1) {
        inf.zero_dst = kPack ? pout + pbody + S.raw_bytes
                             : pout + cbody + S.raw_bytes;
        inf.zero_bytes = kPack ? (int32_t)(c_end - pbody - S.raw_bytes)
                               : (int32_t)(cend - cbody - S.raw_bytes);
      }
    } else {
      const int tile = local - S.nraw;
      const int t0 = tile * S.tile;
      const int ntok = min((int)S.tile, S.tc - t0);
      const int64_t prec = pbody + S.raw_bytes + (int64_t)t0 * c_rp;
      const int64_t crec = cbody + S.raw_bytes + (int64_t)t0 * S.R;
      const bool last = tile == S.ntiles - 1;
      inf.kind = 2;
      inf.ntok = ntok;
      if (kPack) {
        inf.gsrc = pin + crec;
        inf.load_bytes = ntok * S.R;
        inf.gdst = pout + prec;
        inf.store_bytes = last ? (int32_t)(c_end - prec) : ntok * c_rp;
      } else {
        inf.gsrc = pin + prec;
        inf.load_bytes = (ntok * c_rp + 15) & ~15;
        inf.gdst = pout + crec;
        inf.store_bytes = last ? (int32_t)(cend - crec) : ntok * S.R;
      }
    }
    uint16_t tab[32];
#pragma unroll
    for (int s = 0; s < 32; ++s)
      tab[s] = (uint16_t)__shfl_sync(0xffffffffu, c_tab, s);
    if (lane == 0) {
      FpInfo& f = info[bsel];
      f.gsrc = inf.gsrc;
      f.gdst = inf.gdst;
      f.zero_dst = inf.zero_dst;
      f.kind = inf.kind;
      f.load_bytes = inf.load_bytes;
      f.store_bytes = inf.store_bytes;
      f.zero_bytes = inf.zero_bytes;
      f.ntok = inf.ntok;
      f.ga = inf.ga;
      f.used = inf.used;
      f.R = inf.R;
      f.rp = inf.rp;
      f.hb2 = inf.hb2;
#pragma unroll
      for (int s = 0; s < 32; ++s) f.table[s] = tab[s];
      if (inf.kind == 0) {
        mbar_arrive(&full[bsel]);
      } else {
        mbar_arrive_expect_tx(&full[bsel], (uint32_t)inf.load_bytes);
        bulk_g2s(smem + bsel * kFpBuf, inf.gsrc, (uint32_t)inf.load_bytes,
                 &full[bsel]);
      }
    }
    __syncwarp();
  };

  if (warp == 0) {
    if (ib < ie) produce(ib, 0);
    if (ib + 1 < ie) produce(ib + 1, 1);
  }
  uint32_t phase = 0;  // bit b: parity to wait for on full[b]
  bool bad = false;
  for (int it = ib; it < ie; ++it) {
    const int bsel = (it - ib) & 1;
    const bool got = mbar_wait(&full[bsel], (phase >> bsel) & 1u, &abort_flag);
    phase ^= 1u << bsel;
    if (__syncthreads_or(!got)) {
      if (tid == 0) {
        atomicOr(p.status, KVTC_FLAG_TIMEOUT);
        mbar_drain(&full[bsel], ((phase >> bsel) & 1u) ^ 1u);
        if (it + 1 < ie)
          mbar_drain(&full[bsel ^ 1], (phase >> (bsel ^ 1)) & 1u);
      }
      break;
    }
    const FpInfo& f = info[bsel];
    const int kind = f.kind;
    uint8_t* s_in = smem + bsel * kFpBuf;
    if (kind == 2) {
      const int ntok = f.ntok, ga = f.ga, nslot = 2 * ga, R = f.R;
      const int rp = f.rp, hb2 = f.hb2, used = f.used;
      const int store_bytes = f.store_bytes;
      int vmin = 0, d = 0;
      if (lane < nslot) {
        vmin = f.table[lane] & 0xff;
        d = f.table[lane] >> 8;
      }
      const FpSlots sl = fp_slots_from(vmin, d, nslot);
      if (tid == 0) bulk_wait_read<0>();  // s_out read by the last store
      __syncthreads();
      const int body = kPack ? ntok * rp : ntok * R;
      for (int b = body + tid; b < store_bytes; b += kFpThreads) s_out[b] = 0;
      if (kPack) {
        // four tokens per warp step: their loads issue back to back
        const int nw = (sl.hbits + 31) >> 5, p2 = (used - 4 * ga) >> 1;
        const int w0 = lane < nslot ? sl.pos >> 5 : -2;
        const int s5 = sl.pos & 31, fsh = 16 * (lane & 1);
        const uint32_t umask = (1u << sl.d) - 1;
        for (int tok0 = 4 * warp; tok0 < ntok; tok0 += 4 * kFpWarps) {
          const int nt = min(4, ntok - tok0);
          uint32_t wv[4], clo[4], chi[4], mine[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            wv[u] = (u < nt && lane < nslot)
                        ? reinterpret_cast<const uint32_t*>(
                              s_in + (tok0 + u) * R)[lane >> 1]
                        : 0u;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            clo[u] = chi[u] = mine[u] = 0u;
            if (u < nt && lane < nslot) {
              const uint32_t lo = (wv[u] >> fsh) & 0xffu;
              const uint32_t hi = (wv[u] >> (fsh + 8)) & 0xffu;
              s_out[(tok0 + u) * rp + lane] = (uint8_t)lo;
              const int v = (int)(hi >> 2) - sl.vmin;
              if (v < 0 || v > (int)umask) bad = true;
              // h - 4 vmin: the low 2 bits of h, then v - vmin
              const uint32_t code = (hi - 4u * (uint32_t)sl.vmin) &
                                    ((4u << sl.d) - 1u);
              clo[u] = code << s5;
              chi[u] = s5 ? code >> (32 - s5) : 0u;
            }
          }
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            if (w < nw) {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const uint32_t v = __reduce_or_sync(
                    0xffffffffu,
                    (w0 == w ? clo[u] : 0u) | (w0 + 1 == w ? chi[u] : 0u));
                if ((lane >> 1) == w) mine[u] = v;
              }
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (u < nt && lane < hb2)
              reinterpret_cast<uint16_t*>(s_out + (tok0 + u) * rp)[ga + lane] =
                  (uint16_t)(mine[u] >> fsh);
          for (int j = lane; j < p2; j += 32) {
            uint16_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              v[u] = u < nt ? reinterpret_cast<const uint16_t*>(
                                  s_in + (tok0 + u) * R)[2 * ga + j]
                            : (uint16_t)0;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (u < nt)
                reinterpret_cast<uint16_t*>(
                    s_out + (tok0 + u) * rp)[ga + hb2 + j] = v[u];
          }
          // the record's zero padding to a multiple of 4 bytes
          if (lane < nt && 2 * (ga + hb2 + p2) < rp)
            reinterpret_cast<uint16_t*>(s_out + (tok0 + lane) * rp)[ga + hb2 +
                                                                    p2] = 0;
        }
      } else {
        const int R2 = R >> 1, u2 = used >> 1;
        const int k = sl.pos >> 4, sh = sl.pos & 15;
        const uint32_t cmask = (4u << sl.d) - 1;
        for (int tok0 = 4 * warp; tok0 < ntok; tok0 += 4 * kFpWarps) {
          const int nt = min(4, ntok - tok0);
          uint32_t bits[4], lob[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            bits[u] = lob[u] = 0u;
            if (u < nt && lane < nslot) {
              const uint8_t* ibp = s_in + (tok0 + u) * rp;
              const uint16_t* i16 = reinterpret_cast<const uint16_t*>(ibp);
              bits[u] = (uint32_t)i16[ga + k] | ((uint32_t)i16[ga + k + 1] << 16);
              lob[u] = ibp[lane];
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (u < nt && lane < nslot) {
              const uint32_t code = (bits[u] >> sh) & cmask;
              const uint32_t hi = (code + 4u * (uint32_t)sl.vmin) & 0xffu;
              reinterpret_cast<uint16_t*>(s_out + (tok0 + u) * R)[lane] =
                  (uint16_t)(lob[u] | (hi << 8));
            }
          }
          for (int j = 2 * ga + lane; j < R2; j += 32) {
            uint16_t v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
              v[u] = (u < nt && j < u2)
                         ? reinterpret_cast<const uint16_t*>(
                               s_in + (tok0 + u) * rp)[hb2 - ga + j]
                         : (uint16_t)0;
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (u < nt)
                reinterpret_cast<uint16_t*>(s_out + (tok0 + u) * R)[j] = v[u];
          }
        }
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        bulk_s2g(f.gdst, s_out, (uint32_t)store_bytes);
        bulk_commit();
      }
    } else if (kind == 1) {
      if (tid == 0) {
        bulk_s2g(f.gdst, s_in, (uint32_t)f.load_bytes);
        bulk_commit();
      }
      const int nz = f.zero_bytes >> 4;
      for (int c = tid; c < nz; c += kFpThreads)
        reinterpret_cast<uint4*>(f.zero_dst)[c] = make_uint4(0, 0, 0, 0);
    }
    // refill this buffer with the item two ahead
    if (it + 2 < ie) {
      if (kind == 1 && tid == 0) bulk_wait_read<0>();
      __syncthreads();
      if (warp == 0) produce(it + 2, bsel);
    }
  }
  if (tid == 0) bulk_wait<0>();
  if (bad) atomicOr(p.status, KVTC_FLAG_FORMAT);
}

// Per-device launch facts, looked up once: SM count, and whether the tile
// kernels' shared-memory limit has been raised on the device.
constexpr int kFpMaxDev = 64;
int g_fp_sms[kFpMaxDev];
bool g_fp_smem_set[kFpMaxDev][2];

int fp_device() {
  int dev = 0;
  cudaGetDevice(&dev);
  return dev >= 0 && dev < kFpMaxDev ? dev : 0;
}

void fp_allow_smem(const void* func) {
  const int dev = fp_device();
  const int which = func == (const void*)fp_tile_kernel<true> ? 0 : 1;
  if (!g_fp_smem_set[dev][which]) {
    cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kFpSmem);
    g_fp_smem_set[dev][which] = true;
  }
}

int fp_blocks(int items) {
  const int dev = fp_device();
  if (g_fp_sms[dev] == 0) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_fp_sms[dev] = sms > 0 ? sms : 1;
  }
  const int cap = 2 * g_fp_sms[dev];
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
    fp_allow_smem((const void*)fp_tile_kernel<true>);
    fp_tile_kernel<true>
        <<<fp_blocks(p.total_items), kFpThreads, kFpSmem, st>>>(p);
    count_launch();
  }
  return cudaGetLastError();
}

cudaError_t launch_fields_unpack(const FpParams& p, cudaStream_t st) {
  if (p.n == 0 || p.total_items == 0) return cudaSuccess;
  fp_allow_smem((const void*)fp_tile_kernel<false>);
  fp_tile_kernel<false>
      <<<fp_blocks(p.total_items), kFpThreads, kFpSmem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvtc
