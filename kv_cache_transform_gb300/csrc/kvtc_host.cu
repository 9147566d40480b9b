// Host side of the C ABI declared in include/kvtc.h: calibration blob
// parsing, device operand preparation, argument validation and launches.
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"

using namespace kvtc;

namespace kvtc {
static std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

uint32_t crc32_ieee(const uint8_t* p, size_t n) {
  // CRC-32 of IEEE 802.3 (reflected polynomial 0xEDB88320, init and final
  // xor 0xFFFFFFFF), table driven.
  static uint32_t table[256];
  static std::once_flag once;
  std::call_once(once, [] {
    for (uint32_t i = 0; i < 256; ++i) {
      uint32_t c = i;
      for (int k = 0; k < 8; ++k) c = (c & 1u) ? 0xEDB88320u ^ (c >> 1) : c >> 1;
      table[i] = c;
    }
  });
  uint32_t c = 0xFFFFFFFFu;
  for (size_t i = 0; i < n; ++i) c = table[(c ^ p[i]) & 0xFFu] ^ (c >> 8);
  return c ^ 0xFFFFFFFFu;
}
}  // namespace kvtc

namespace {

// Nearest (ties to even) bf16 of a finite double, rounded once: keep 8
// significant bits (quantum 2^-133 below the normal range).
uint16_t bf16_bits_rne(double x) {
  int e;
  std::frexp(x, &e);
  if (x == 0.0) e = 0;
  const int ee = e < -125 ? -125 : e;
  const double r = std::nearbyint(std::ldexp(x, 8 - ee));
  const float f = (float)std::ldexp(r, ee - 8);  // exact
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// Nearest (ties to even) fp16 of a finite double, rounded once: keep 11
// significant bits (quantum 2^-24 below the normal range), then assemble
// the binary16 fields.  Values beyond 65504 after rounding become inf.
uint16_t fp16_bits_rne(double x) {
  uint16_t sign = std::signbit(x) ? 0x8000u : 0u;
  double a = std::fabs(x);
  if (a == 0.0) return sign;
  int e;
  std::frexp(a, &e);
  const int ee = e < -13 ? -13 : e;
  const double r = std::nearbyint(std::ldexp(a, 11 - ee));
  const double v = std::ldexp(r, ee - 11);
  if (v > 65504.0) return sign | 0x7C00u;
  if (v < std::ldexp(1.0, -14)) {  // subnormal: v = m * 2^-24
    return sign | (uint16_t)std::ldexp(v, 24);
  }
  int ev;
  const double mant = std::frexp(v, &ev);  // v = mant * 2^ev, mant in [.5,1)
  const int exp_field = ev - 1 + 15;
  const uint16_t frac = (uint16_t)((mant * 2.0 - 1.0) * 1024.0);
  return sign | (uint16_t)(exp_field << 10) | frac;
}

struct Reader {
  const uint8_t* p;
  size_t n, off;
  bool ok = true;
  template <class T>
  T get() {
    T v{};
    if (off + sizeof(T) > n) {
      ok = false;
      return v;
    }
    std::memcpy(&v, p + off, sizeof(T));
    off += sizeof(T);
    return v;
  }
  const uint8_t* take(size_t bytes) {
    if (off + bytes > n) {
      ok = false;
      return nullptr;
    }
    const uint8_t* r = p + off;
    off += bytes;
    return r;
  }
};

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// K-block-major operand [nblk][rows][64] (16-bit elements): 3-D map
// {64, rows, nblk}, box {64, box_rows, box_blk}, 128-byte swizzle; a box
// lands in shared memory as box_blk [box_rows][64] tiles.
bool encode_blocked_3d(CUtensorMap* m, CUtensorMapDataType dt,
                       const void* base, uint64_t rows, uint64_t nblk,
                       uint32_t box_rows, uint32_t box_blk) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, rows, nblk};
  cuuint64_t strides[2] = {128, 128ull * rows};
  cuuint32_t box[3] = {64u, box_rows, box_blk};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 rows [rows][cols] (row stride row_bytes) viewed as
// {64 columns, rows, cols / 64 column blocks}: one box {64, 128 rows, 2}
// brings 128 rows of two consecutive 64-column K blocks, landing in shared
// memory as two [128][64] tiles; 128-byte swizzle.
bool encode_rows_kblocks(CUtensorMap* m, const void* base, uint64_t cols,
                         uint64_t rows, uint64_t row_bytes, uint32_t kblocks) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, rows, cols / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64u, (cuuint32_t)kTileM, kblocks};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map for the reconstruction epilogue: bf16 rows [rows][cols] with a
// stride of row_bytes, box {64 columns, 32 rows}, 128-byte swizzle.
bool encode_store_2d(CUtensorMap* m, const void* base, uint64_t cols,
                     uint64_t rows, uint64_t row_bytes) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {64u, 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A paged pool bf16 [num_blocks][16][D] as {D, 16, num_blocks}: box {64,
// 16, 1} is one block's rows of a 64-column slab, 128-byte swizzle.
bool encode_pool_3d(CUtensorMap* m, const void* base, uint64_t D,
                    uint64_t num_blocks) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {D, 16, num_blocks};
  cuuint64_t strides[2] = {D * 2, D * 2 * 16};
  cuuint32_t box[3] = {64u, 16u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev)
      cudaSetDevice(prev);
  }
};

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
inline bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

// ---------------------------------------------------------------- calib
struct HostStream {
  int layer, kv, D, k, Ga, R;
  std::vector<uint8_t> widths;
};

struct kvtc_calib {
  int device = 0;
  int sm_count = 0;
  int group = 16, bmax = 8, sink = 0, window = 0, budget_bits = 0;
  std::vector<HostStream> hs;
  std::map<std::pair<int, int>, int> index;  // (layer, kv) -> stream
  void* pool = nullptr;                      // all device operands
  DevStream* d_streams = nullptr;
  unsigned* d_status = nullptr;
};

namespace {

int record_bytes(int budget_bits) { return 16 * ((budget_bits + 127) / 128); }

// Row of V_enc (K-block major [D/64][k][64]) that holds kept component a.
// CTA r of a pair loads rows [r k/2, (r + 1) k/2).  Up to k = 256 one MMA
// of N = k reads them in order.  Above, two MMAs per K step read rows
// [0, 128) (N = 256, output columns [0, 256)) and rows [128, k/2)
// (N = k - 256, columns [256, k)) of each CTA, so the rows are stored in
// the order that puts component j in output column j.
int venc_row(int a, int k) {
  if (k <= 256) return a;
  const int half = k / 2, h2 = (k - 256) / 2;
  if (a < 128) return a;
  if (a < 256) return half + (a - 128);
  if (a < 256 + h2) return 128 + (a - 256);
  return half + 128 + (a - 256 - h2);
}

void split_tokens(int64_t T, int s, int w, int64_t* s_, int64_t* w_,
                  int64_t* tc) {
  *s_ = std::min<int64_t>(s, T);
  *w_ = std::min<int64_t>(w, T - *s_);
  *tc = T - *s_ - *w_;
}

int64_t stream_bytes_of(const kvtc_calib* c, const HostStream& h, int64_t T) {
  int64_t s_, w_, tc;
  split_tokens(T, c->sink, c->window, &s_, &w_, &tc);
  return align_up((s_ + w_) * h.D * 2 + tc * h.R, 256);
}

int find_stream(const kvtc_calib* c, int layer, int kv) {
  auto it = c->index.find({layer, kv});
  return it == c->index.end() ? -1 : it->second;
}

// Selected (layer, kv) streams of a call in storage order.
int select_streams(const kvtc_calib* c, int layer0, int nlayers, int kv_mask,
                   std::vector<int>* cs, std::vector<int>* slot) {
  if (nlayers < 0 || kv_mask < 1 || kv_mask > 3) return KVTC_EINVAL;
  for (int l = 0; l < nlayers; ++l)
    for (int kv = 0; kv < 2; ++kv) {
      if (!(kv_mask & (1 << kv))) continue;
      const int i = find_stream(c, layer0 + l, kv);
      if (i < 0) return KVTC_EINVAL;
      cs->push_back(i);
      slot->push_back(2 * l + kv);
    }
  return KVTC_OK;
}

// CTA pairs for `items` super-tiles, at most what can be resident at once.
// Append a row segment to the raw-row list a tensor-core kernel copies
// while it runs (src null: zeros).  False when the list is full.
bool raw_list_add(RawList& r, const char* s, char* d, int64_t sld,
                  int64_t dld, int64_t rows, int64_t row_bytes) {
  if (rows <= 0 || row_bytes <= 0) return true;
  if (r.nseg == kRawListMax) return false;
  RawListSeg& g = r.seg[r.nseg++];
  g.src = s;
  g.dst = d;
  g.src_ld = sld;
  g.dst_ld = dld;
  g.rows = (int32_t)rows;
  g.row_bytes = (int32_t)row_bytes;
  g.chunk_begin = r.total_chunks;
  g.pk = -1;
  g.pk_tc = 0;
  g.pk_off = 0;
  r.total_chunks += rows * (row_bytes / 16);
  return true;
}

// The same for rows of packed stream `pk` (r.pk_offs), `at` bytes from its
// start, whose header must hold T_c = tc; the kernel checks both.
bool raw_list_add_packed(RawList& r, int pk, int tc, int64_t at, char* d,
                         int64_t dld, int64_t rows, int64_t row_bytes) {
  if (!raw_list_add(r, nullptr, d, row_bytes, dld, rows, row_bytes))
    return false;
  if (rows <= 0 || row_bytes <= 0) return true;
  RawListSeg& g = r.seg[r.nseg - 1];
  g.pk = pk;
  g.pk_tc = tc;
  g.pk_off = at;
  return true;
}

int pairs_for(int max_pairs, int items) {
  return std::max(1, std::min(items, max_pairs));
}

// The compressed input of a restore may sit in device memory, or in pinned
// host memory, which is mapped into the device's address space: the kernels
// then read it over the host link themselves, with no staging copy.
// Pageable host memory cannot be read by the kernels and is refused.
int resolve_input(const void* p, const void** dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return KVTC_EINVAL;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *dev = p;
    return KVTC_OK;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *dev = a.devicePointer;
    return KVTC_OK;
  }
  return KVTC_EINVAL;
}

// Restore of codec streams (pk_offs null), or of the packed streams that
// kvtc_fields_pack wrote (pk_offs: their offsets), whose records the restore
// kernel unpacks as it reads them.
int decompress_impl(const kvtc_calib* c, int layer0, int nlayers, int kv_mask,
                    const void* src, int64_t src_bytes,
                    const int64_t* pk_offs, int64_t T, void* const* dst,
                    int64_t ld, void* cuda_stream,
                    void* const* layer_events) {
  const bool packed = pk_offs != nullptr;
  if (!c || !dst || (!src && src_bytes) || T < 0 || T > (1LL << 31) - 1)
    return KVTC_EINVAL;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  int64_t s_, w_, tc;
  split_tokens(T, c->sink, c->window, &s_, &w_, &tc);
  int64_t need = 0;
  std::vector<int64_t> off(cs.size());
  for (size_t i = 0; i < cs.size(); ++i) {
    const HostStream& h = c->hs[cs[i]];
    if (!dst[slot[i]] && T > 0) return KVTC_EINVAL;
    if (ld < h.D) return KVTC_ESIZE;
    if (ld % 8 || !aligned16(dst[slot[i]])) return KVTC_EALIGN;
    // field packing holds at most 15 active groups a stream
    if (packed && h.Ga > 15) return KVTC_ENOTSUP;
    off[i] = need;
    need += stream_bytes_of(c, h, T);
  }
  // a packed stream is at least 256 bytes; its length is in the offsets,
  // which the kernels check against src_bytes
  if (packed) need = (int64_t)cs.size() * 256;
  if (src_bytes < need) return KVTC_ESIZE;
  if (!aligned16(src)) return KVTC_EALIGN;
  if (packed && (reinterpret_cast<uintptr_t>(pk_offs) & 7u))
    return KVTC_EALIGN;
  if (layer_events)
    for (int l = 0; l < nlayers; ++l)
      if (!layer_events[l]) return KVTC_EINVAL;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  if (need > 0) {
    st = resolve_input(src, &src);
    if (st != KVTC_OK) return st;
  }
  if (packed && !cs.empty()) {
    const void* o = pk_offs;
    st = resolve_input(pk_offs, &o);
    if (st != KVTC_OK) return st;
    pk_offs = static_cast<const int64_t*>(o);
  }
  const char* in = static_cast<const char*>(src);

  // Launch groups: all streams at once, or one layer at a time when the
  // caller wants per-layer completion events.
  std::vector<std::pair<size_t, size_t>> groups;
  if (layer_events) {
    size_t i = 0;
    for (int l = 0; l < nlayers; ++l) {
      size_t j = i;
      while (j < cs.size() && slot[j] / 2 == l) ++j;
      groups.push_back({i, j});
      i = j;
    }
  } else {
    for (size_t i = 0; i < cs.size(); i += kDecMaxSeg)
      groups.push_back({i, std::min(cs.size(), i + (size_t)kDecMaxSeg)});
  }
  RawParams* rp = new (std::nothrow) RawParams;
  DecParams* p = new (std::nothrow) DecParams;
  if (!rp || !p) {
    delete rp;
    delete p;
    return KVTC_ENOMEM;
  }
  int ret = KVTC_OK;
  for (size_t gi = 0; gi < groups.size() && ret == KVTC_OK; ++gi) {
    const size_t i0 = groups[gi].first, i1 = groups[gi].second;
    // raw rows back to their places: by the decompress kernel while it
    // runs, or by a copy kernel when there are no coded tokens
    std::memset(rp, 0, sizeof(*rp));
    std::memset(p, 0, sizeof(*p));
    if (packed) {
      p->raw.pk_base = reinterpret_cast<const uint8_t*>(in);
      p->raw.pk_offs = pk_offs;
      p->raw.pk_bytes = src_bytes;
    }
    for (size_t i = i0; i < i1; ++i) {
      const HostStream& h = c->hs[cs[i]];
      const int64_t rb = 2LL * h.D;
      const char* so = in + off[i];
      char* x = static_cast<char*>(dst[slot[i]]);
      const int64_t rows[2] = {s_, w_};
      const char* s2[2] = {so, so + s_ * rb};
      char* d2[2] = {x, x + (T - w_) * 2 * ld};
      for (int k2 = 0; k2 < 2; ++k2) {
        if (rows[k2] <= 0) continue;
        if (packed) {
          // the rows follow the header and the slot table
          const int64_t at = fp_prefix_bytes(h.Ga) + (k2 ? s_ * rb : 0);
          if (!raw_list_add_packed(p->raw, (int)i, (int)tc, at, d2[k2],
                                   2 * ld, rows[k2], rb))
            ret = KVTC_EINVAL;
          continue;
        }
        if (tc > 0) {
          if (!raw_list_add(p->raw, s2[k2], d2[k2], rb, 2 * ld, rows[k2], rb))
            ret = KVTC_EINVAL;
          continue;
        }
        if (rp->nseg == kRawMaxSeg) {
          if (launch_raw_copy(*rp, stream) != cudaSuccess) ret = KVTC_ECUDA;
          rp->nseg = 0;
          rp->total_chunks = 0;
        }
        RawSeg& g = rp->seg[rp->nseg++];
        g.src = s2[k2];
        g.dst = d2[k2];
        g.src_ld = rb;
        g.dst_ld = 2 * ld;
        g.rows = (int32_t)rows[k2];
        g.row_bytes = (int32_t)rb;
        g.chunk_begin = rp->total_chunks;
        rp->total_chunks += rows[k2] * (rb / 16);
      }
    }
    if (rp->nseg && launch_raw_copy(*rp, stream) != cudaSuccess)
      ret = KVTC_ECUDA;
    if (packed && tc == 0 &&
        launch_raw_list(p->raw, c->d_status, stream) != cudaSuccess)
      ret = KVTC_ECUDA;
    if (ret != KVTC_OK) break;
    if (tc > 0) {
      int tiles = 0;
      for (size_t i = i0; i < i1; ++i) {
        const HostStream& h = c->hs[cs[i]];
        DecSeg& g = p->seg[i - i0];
        // packed input: the kernel finds the records through the offsets
        g.rec = reinterpret_cast<const uint8_t*>(
            packed ? in : in + off[i] + (s_ + w_) * 2LL * h.D);
        g.dst = static_cast<char*>(dst[slot[i]]) + s_ * 2 * ld;
        g.ld_bytes = 2 * ld;
        g.tc = (int32_t)tc;
        g.cs = cs[i];
        if (!encode_store_2d(&p->tm_out[i - i0], g.dst, (uint64_t)h.D,
                             (uint64_t)tc, 2ull * ld)) {
          ret = KVTC_ECUDA;
          break;
        }
        tiles += (int)((tc + kPairM - 1) / kPairM);
      }
      if (ret != KVTC_OK) break;
      p->streams = c->d_streams;
      p->status = c->d_status;
      p->nseg = (int32_t)(i1 - i0);
      p->total_tiles = tiles;
      p->tiles_per_seg = (int32_t)((tc + kPairM - 1) / kPairM);
      int rmax = 0, kmax = 0;
      for (size_t i = i0; i < i1; ++i) {
        rmax = std::max(rmax, c->hs[cs[i]].R);
        kmax = std::max(kmax, c->hs[cs[i]].k);
      }
      p->rec_words = rmax / 4;
      p->wide = kmax > kNarrowK;
      p->packed = packed;
      p->pk_first = (int32_t)i0;
      p->pk_raw_rows = (int32_t)(s_ + w_);
      p->nstages = decompress_stages(p->rec_words);
      const int mp = max_pairs_decompress(
          decompress_smem_bytes(p->nstages, p->rec_words));
      if (tiles && (mp < 1 || launch_decompress(*p, pairs_for(mp, tiles),
                                                stream) != cudaSuccess))
        ret = KVTC_ECUDA;
    }
    if (ret == KVTC_OK && layer_events &&
        cudaEventRecord(static_cast<cudaEvent_t>(layer_events[gi]), stream) !=
            cudaSuccess)
      ret = KVTC_ECUDA;
  }
  delete rp;
  delete p;
  return ret;
}

}  // namespace

extern "C" {

uint64_t kvtc_launch_count(void) {
  return kvtc::g_launches.load(std::memory_order_relaxed);
}

const char* kvtc_strerror(int s) {
  switch (s) {
    case KVTC_OK: return "ok";
    case KVTC_EINVAL: return "invalid argument";
    case KVTC_EFORMAT: return "malformed calibration blob";
    case KVTC_ESIZE: return "buffer size or token count inconsistent";
    case KVTC_ENOMEM: return "device allocation failed";
    case KVTC_ECUDA: return "CUDA call failed";
    case KVTC_ERANGE: return "fp16 field out of range";
    case KVTC_EDEVICE: return "device-side fault flag";
    case KVTC_EALIGN: return "pointer or stride misaligned";
    case KVTC_ENOTSUP: return "shape not supported by the kernels";
    default: return "unknown status";
  }
}

int kvtc_calib_load(const void* blob, size_t blob_bytes, int cuda_device,
                    kvtc_calib** out) {
  if (!blob || !out || cuda_device < 0) return KVTC_EINVAL;
  *out = nullptr;
  const uint8_t* b = static_cast<const uint8_t*>(blob);
  if (blob_bytes < 4 + 28 + 8 || std::memcmp(b, "KVTC", 4) != 0)
    return KVTC_EFORMAT;
  uint32_t crc, zero;
  std::memcpy(&crc, b + blob_bytes - 8, 4);
  std::memcpy(&zero, b + blob_bytes - 4, 4);
  if (zero != 0 || crc32_ieee(b, blob_bytes - 8) != crc) return KVTC_EFORMAT;
  Reader r{b, blob_bytes - 8, 4};
  const uint32_t version = r.get<uint32_t>(), n = r.get<uint32_t>();
  const uint32_t group = r.get<uint32_t>(), bmax = r.get<uint32_t>();
  const uint32_t sink = r.get<uint32_t>(), window = r.get<uint32_t>();
  const uint32_t budget = r.get<uint32_t>();
  if (!r.ok || version != 1 || group != 16 || bmax < 1 || bmax > 8 || n == 0 ||
      n > 65536 || sink > (1u << 30) || window > (1u << 30) ||
      budget > (1u << 24))
    return KVTC_EFORMAT;

  kvtc_calib* c = new (std::nothrow) kvtc_calib();
  if (!c) return KVTC_ENOMEM;
  c->device = cuda_device;
  c->group = (int)group;
  c->bmax = (int)bmax;
  c->sink = (int)sink;
  c->window = (int)window;
  c->budget_bits = (int)budget;
  const int R = record_bytes((int)budget);

  struct Raw {
    const double* mu;
    const double* V;
  };
  std::vector<Raw> raw;
  int status = KVTC_OK;
  for (uint32_t i = 0; i < n && status == KVTC_OK; ++i) {
    HostStream h;
    h.layer = (int)r.get<uint32_t>();
    h.kv = (int)r.get<uint32_t>();
    h.D = (int)r.get<uint32_t>();
    h.k = (int)r.get<uint32_t>();
    if (!r.ok || h.kv > 1 || h.D <= 0 || h.D % 16 || h.k < 0 || h.k > h.D) {
      status = KVTC_EFORMAT;
      break;
    }
    const int G = h.D / 16;
    const uint8_t* w = r.take((size_t)((G + 7) / 8 * 8));
    const uint8_t* mu = r.take((size_t)h.D * 8);
    const uint8_t* V = r.take((size_t)h.k * h.D * 8);
    const uint8_t* ev = r.take((size_t)h.D * 8);
    (void)ev;
    if (!r.ok) {
      status = KVTC_EFORMAT;
      break;
    }
    h.widths.assign(w, w + G);
    for (int d = 0; d < h.D; ++d) {
      double m;
      std::memcpy(&m, mu + 8LL * d, 8);
      if (!std::isfinite(m) || std::fabs(m) > 60000.0) status = KVTC_ENOTSUP;
    }
    if (status != KVTC_OK) break;
    int ga = 0, cost = 0;
    for (int g = 0; g < G; ++g) {
      if (h.widths[g] > bmax) status = KVTC_EFORMAT;
      if (h.widths[g]) {
        ++ga;
        cost += 32 + 16 * h.widths[g];
      }
    }
    if (status != KVTC_OK || 16 * ga != h.k || cost > (int)budget) {
      status = KVTC_EFORMAT;
      break;
    }
    h.Ga = ga;
    h.R = R;
    // the projection's ring (at least one stage: x tile and this CTA's
    // V_enc half, two K blocks each) and its record staging must fit shared
    // memory (always so for k <= 496 and R <= 256)
    const bool smem_ok =
        compress_smem_bytes(1, 2 * kTileM * 128 + h.k * 128, R / 4) <= 232448;
    if (h.D % 64 || h.D > kMaxD || h.k > kMaxK || h.k == 0 || R > kMaxRecord ||
        !smem_ok || find_stream(c, h.layer, h.kv) >= 0) {
      status = find_stream(c, h.layer, h.kv) >= 0 ? KVTC_EFORMAT : KVTC_ENOTSUP;
      break;
    }
    c->index[{h.layer, h.kv}] = (int)c->hs.size();
    c->hs.push_back(h);
    raw.push_back({reinterpret_cast<const double*>(mu),
                   reinterpret_cast<const double*>(V)});
  }
  if (status == KVTC_OK && r.off != r.n) status = KVTC_EFORMAT;
  if (status != KVTC_OK) {
    delete c;
    return status;
  }

  DeviceGuard guard(cuda_device);
  if (!guard.ok ||
      cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount,
                             cuda_device) != cudaSuccess) {
    delete c;
    return KVTC_ECUDA;
  }

  // One pool: [DevStream x n][status][per stream: mu, m, bits, poff, venc,
  // vdec], each piece 256-byte aligned.
  struct Off {
    int64_t mu, m, bits, poff, venc, vdec;
  };
  std::vector<Off> offs(c->hs.size());
  int64_t total = align_up((int64_t)sizeof(DevStream) * n, 256);
  const int64_t status_off = total;
  total += 256;
  for (size_t i = 0; i < c->hs.size(); ++i) {
    const HostStream& h = c->hs[i];
    Off& o = offs[i];
    o.mu = total; total = align_up(total + 4LL * h.D, 256);
    o.m = total; total = align_up(total + 4LL * h.k, 256);
    o.bits = total; total = align_up(total + h.Ga, 256);
    o.poff = total; total = align_up(total + 2LL * h.Ga, 256);
    o.venc = total; total = align_up(total + 2LL * h.k * h.D, 256);
    o.vdec = total;
    total = align_up(total + 2LL * ((h.k + 16 + 63) / 64 * 64) * h.D, 256);
  }
  std::vector<uint8_t> host((size_t)total, 0);
  if (cudaMalloc(&c->pool, (size_t)total) != cudaSuccess) {
    delete c;
    return KVTC_ENOMEM;
  }
  uint8_t* dev = static_cast<uint8_t*>(c->pool);
  std::vector<DevStream> ds(c->hs.size());
  for (size_t i = 0; i < c->hs.size(); ++i) {
    const HostStream& h = c->hs[i];
    const Off& o = offs[i];
    const double* mu = raw[i].mu;
    const double* V = raw[i].V;  // [k][D]
    float* hmu = reinterpret_cast<float*>(host.data() + o.mu);
    float* hm = reinterpret_cast<float*>(host.data() + o.m);
    uint8_t* hb = host.data() + o.bits;
    uint16_t* hp = reinterpret_cast<uint16_t*>(host.data() + o.poff);
    uint16_t* venc = reinterpret_cast<uint16_t*>(host.data() + o.venc);
    uint16_t* vdec = reinterpret_cast<uint16_t*>(host.data() + o.vdec);
    std::vector<double> muv(h.D);
    const int kp = h.k + 16;
    // V_dec is stored K-block major, [kb][d][64], so that one 3-D TMA box
    // brings all K blocks of a run of output channels
    auto vd = [&](int d, int col) -> uint16_t& {
      return vdec[((size_t)(col >> 6) * h.D + d) * 64 + (col & 63)];
    };
    for (int d = 0; d < h.D; ++d) {
      std::memcpy(&muv[d], mu + d, 8);
      hmu[d] = (float)muv[d];
      // the reconstruction adds mu through one more K step: columns k and
      // k + 1 of V_dec hold mu split into two fp16 terms (the A operand
      // holds 1.0 there), the other 14 columns of that step are zero
      const uint16_t hi = fp16_bits_rne(muv[d]);
      const double hiv = (double)__half2float(__ushort_as_half(hi));
      vd(d, h.k) = hi;
      vd(d, h.k + 1) = fp16_bits_rne(muv[d] - hiv);
    }
    for (int a = 0; a < h.k; ++a) {
      double acc = 0.0;
      for (int d = 0; d < h.D; ++d) {
        double v;
        std::memcpy(&v, V + (size_t)a * h.D + d, 8);
        const uint16_t eb = bf16_bits_rne(v);
        venc[((size_t)(d >> 6) * h.k + venc_row(a, h.k)) * 64 + (d & 63)] =
            eb;
        vd(d, a) = fp16_bits_rne(v);
        uint32_t u = (uint32_t)eb << 16;
        float ef;
        std::memcpy(&ef, &u, 4);
        acc += (double)ef * muv[d];
      }
      hm[a] = (float)acc;
    }
    int ga = 0, bitsum = 0;
    for (int g = 0; g < h.D / 16; ++g) {
      if (!h.widths[g]) continue;
      hb[ga] = h.widths[g];
      hp[ga] = 0;  // filled below
      ++ga;
    }
    for (int a = 0; a < h.Ga; ++a) {
      hp[a] = (uint16_t)(4 * h.Ga + 2 * bitsum);
      bitsum += hb[a];
    }
    DevStream& s = ds[i];
    std::memset(&s, 0, sizeof(s));
    s.mu = reinterpret_cast<const float*>(dev + o.mu);
    s.m = reinterpret_cast<const float*>(dev + o.m);
    s.bits = dev + o.bits;
    s.poff = reinterpret_cast<const uint16_t*>(dev + o.poff);
    s.D = h.D;
    s.k = h.k;
    s.Ga = h.Ga;
    s.R = h.R;
    s.nc = (h.D % 256 == 0) ? 256 : (h.D % 128 == 0) ? 128 : 64;
    s.kp = kp;
    // the reconstruction's B operand comes in one ring stage per chunk
    // (every K block, at most four) or in two
    const int nkb = (kp + 63) / 64;
    s.nbs = nkb <= 4 ? 1 : 2;
    s.kbs = (nkb + s.nbs - 1) / s.nbs;
    // each CTA of a pair loads half of the N rows of the B operand, several K
    // blocks at once (V_dec: kbs K blocks of a chunk half; V_enc: two K
    // blocks of the component half)
    if (!encode_blocked_3d(&s.tm_vdec, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           dev + o.vdec, (uint64_t)h.D, (uint64_t)nkb,
                           (uint32_t)(s.nc / 2), (uint32_t)s.kbs) ||
        !encode_blocked_3d(&s.tm_venc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           dev + o.venc, (uint64_t)h.k, (uint64_t)(h.D / 64),
                           (uint32_t)(h.k / 2), 2u) ||
        !encode_blocked_3d(&s.tm_venc1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                           dev + o.venc, (uint64_t)h.k, (uint64_t)(h.D / 64),
                           (uint32_t)(h.k / 2), 1u)) {
      cudaFree(c->pool);
      delete c;
      return KVTC_ECUDA;
    }
  }
  std::memcpy(host.data(), ds.data(), sizeof(DevStream) * ds.size());
  if (cudaMemcpy(c->pool, host.data(), (size_t)total, cudaMemcpyHostToDevice) !=
      cudaSuccess) {
    cudaFree(c->pool);
    delete c;
    return KVTC_ECUDA;
  }
  c->d_streams = reinterpret_cast<DevStream*>(dev);
  c->d_status = reinterpret_cast<unsigned*>(dev + status_off);
  *out = c;
  return KVTC_OK;
}

void kvtc_calib_free(kvtc_calib* c) {
  if (!c) return;
  DeviceGuard guard(c->device);
  if (c->pool) cudaFree(c->pool);
  delete c;
}

int kvtc_calib_query(const kvtc_calib* c, int layer, int kv, int* D, int* k,
                     int* s, int* w, int* R) {
  if (!c) return KVTC_EINVAL;
  const int i = find_stream(c, layer, kv);
  if (i < 0) return KVTC_EINVAL;
  const HostStream& h = c->hs[i];
  if (D) *D = h.D;
  if (k) *k = h.k;
  if (s) *s = c->sink;
  if (w) *w = c->window;
  if (R) *R = h.R;
  return KVTC_OK;
}

int64_t kvtc_stream_bytes(const kvtc_calib* c, int layer, int kv, int64_t T) {
  if (!c || T < 0 || T > (1LL << 31) - 1) return KVTC_EINVAL;
  const int i = find_stream(c, layer, kv);
  if (i < 0) return KVTC_EINVAL;
  return stream_bytes_of(c, c->hs[i], T);
}

int kvtc_compress(const kvtc_calib* c, int layer0, int nlayers, int kv_mask,
                  const void* const* src, int64_t ld, int64_t T, void* dst,
                  int64_t dst_bytes, void* cuda_stream) {
  if (!c || !src || (!dst && dst_bytes) || T < 0 || T > (1LL << 31) - 1)
    return KVTC_EINVAL;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  if (cs.empty()) return KVTC_OK;
  int64_t s_, w_, tc;
  split_tokens(T, c->sink, c->window, &s_, &w_, &tc);
  int64_t need = 0;
  std::vector<int64_t> off(cs.size());
  for (size_t i = 0; i < cs.size(); ++i) {
    const HostStream& h = c->hs[cs[i]];
    if (!src[slot[i]] && T > 0) return KVTC_EINVAL;
    if (ld < h.D) return KVTC_ESIZE;
    if (ld % 8 || !aligned16(src[slot[i]])) return KVTC_EALIGN;
    off[i] = need;
    need += stream_bytes_of(c, h, T);
  }
  if (dst_bytes < need) return KVTC_ESIZE;
  if (!aligned16(dst)) return KVTC_EALIGN;
  if (T == 0) return KVTC_OK;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  char* out = static_cast<char*>(dst);

  // With no coded tokens the raw sink/window rows and the zero padding go
  // by a copy kernel; otherwise the compress kernel copies them while it
  // runs (below).
  if (tc == 0) {
    RawParams rp;
    std::memset(&rp, 0, sizeof(rp));
    auto flush = [&]() -> int {
      if (!rp.nseg) return KVTC_OK;
      if (launch_raw_copy(rp, stream) != cudaSuccess) return KVTC_ECUDA;
      rp.nseg = 0;
      rp.total_chunks = 0;
      return KVTC_OK;
    };
    auto add = [&](const char* s, char* d, int64_t sld, int64_t dld,
                   int64_t rows, int64_t row_bytes) -> int {
      if (rows <= 0 || row_bytes <= 0) return KVTC_OK;
      if (rp.nseg == kRawMaxSeg) {
        int e = flush();
        if (e) return e;
      }
      RawSeg& g = rp.seg[rp.nseg++];
      g.src = s;
      g.dst = d;
      g.src_ld = sld;
      g.dst_ld = dld;
      g.rows = (int32_t)rows;
      g.row_bytes = (int32_t)row_bytes;
      g.chunk_begin = rp.total_chunks;
      rp.total_chunks += rows * (row_bytes / 16);
      return KVTC_OK;
    };
    for (size_t i = 0; i < cs.size(); ++i) {
      const HostStream& h = c->hs[cs[i]];
      const char* x = static_cast<const char*>(src[slot[i]]);
      char* so = out + off[i];
      const int64_t rb = 2LL * h.D;
      int e = add(x, so, 2 * ld, rb, s_, rb);
      if (!e) e = add(x + (T - w_) * 2 * ld, so + s_ * rb, 2 * ld, rb, w_, rb);
      if (e) return e;
    }
    if (flush()) return KVTC_ECUDA;
    // zero the tail padding of every stream (records end 16-byte aligned)
    for (size_t i = 0; i < cs.size(); ++i) {
      const HostStream& h = c->hs[cs[i]];
      const int64_t used = (s_ + w_) * 2LL * h.D + tc * h.R;
      const int64_t pad = stream_bytes_of(c, h, T) - used;
      if (pad > 0 &&
          cudaMemsetAsync(out + off[i] + used, 0, (size_t)pad, stream) !=
              cudaSuccess)
        return KVTC_ECUDA;
    }
    return KVTC_OK;
  }

  // Tensor-core projection + quantise/pack, up to kCompMaxSeg streams per
  // launch, with those streams' raw rows and padding.
  CompParams* p = new (std::nothrow) CompParams;
  if (!p) return KVTC_ENOMEM;
  int ret = KVTC_OK;
  for (size_t i0 = 0; i0 < cs.size() && ret == KVTC_OK; i0 += kCompMaxSeg) {
    std::memset(p, 0, sizeof(*p));
    const size_t i1 = std::min(cs.size(), i0 + kCompMaxSeg);
    int tiles = 0, kmax = 0, rmax = 0;
    for (size_t i = i0; i < i1; ++i) {
      kmax = std::max(kmax, c->hs[cs[i]].k);
      rmax = std::max(rmax, c->hs[cs[i]].R);
    }
    // A ring stage holds two K blocks (x tile and this CTA's V_enc half of
    // each), or one where two such stages do not fit beside the record
    // staging (k > 382 at 256-byte records); then the ring is as deep as
    // fits
    p->kps = 2;
    if (compress_smem_bytes(2, 2 * (kTileM * 128 + kmax * 64), rmax / 4) >
        232448)
      p->kps = 1;
    for (size_t i = i0; i < i1; ++i) {
      const HostStream& h = c->hs[cs[i]];
      CompSeg& g = p->seg[i - i0];
      if (!encode_rows_kblocks(&g.tm_x, src[slot[i]], (uint64_t)h.D,
                               (uint64_t)(s_ + tc), 2ull * ld,
                               (uint32_t)p->kps)) {
        ret = KVTC_ECUDA;
        break;
      }
      g.rec = reinterpret_cast<uint8_t*>(out + off[i] + (s_ + w_) * 2LL * h.D);
      g.tc = (int32_t)tc;
      g.row0 = (int32_t)s_;
      g.cs = cs[i];
      const char* x = static_cast<const char*>(src[slot[i]]);
      char* so = out + off[i];
      const int64_t rb = 2LL * h.D;
      const int64_t used = (s_ + w_) * rb + tc * h.R;
      const int64_t pad = stream_bytes_of(c, h, T) - used;
      if (!raw_list_add(p->raw, x, so, 2 * ld, rb, s_, rb) ||
          !raw_list_add(p->raw, x + (T - w_) * 2 * ld, so + s_ * rb, 2 * ld,
                        rb, w_, rb) ||
          !raw_list_add(p->raw, nullptr, so + used, 0, pad, 1, pad)) {
        ret = KVTC_EINVAL;
        break;
      }
      tiles += (int)((tc + kPairM - 1) / kPairM);
      kmax = std::max(kmax, h.k);
      rmax = std::max(rmax, h.R);
    }
    if (ret != KVTC_OK) break;
    p->wide = kmax > 256;
    p->streams = c->d_streams;
    p->status = c->d_status;
    p->nseg = (int32_t)(i1 - i0);
    p->total_tiles = tiles;
    p->tiles_per_seg = (int32_t)((tc + kPairM - 1) / kPairM);
    // a stage holds kps K blocks: x [kps][128][64] and this CTA's half of
    // V_enc's k rows [kps][k/2][64]
    p->b_bytes_max = p->kps * kmax * 64;
    p->stage_bytes = p->kps * kTileM * 128 + p->b_bytes_max;
    p->rec_stg_words = rmax / 4;
    int nst = 6;
    while (nst > 1 && compress_smem_bytes(nst, p->stage_bytes,
                                          p->rec_stg_words) > 232448)
      --nst;
    p->nstages = nst;
    const int mp = max_pairs_compress(
        compress_smem_bytes(nst, p->stage_bytes, p->rec_stg_words));
    if (mp < 1 || launch_compress(*p, pairs_for(mp, tiles), stream) !=
                      cudaSuccess)
      ret = KVTC_ECUDA;
  }
  delete p;
  return ret;
}

int kvtc_decompress(const kvtc_calib* c, int layer0, int nlayers, int kv_mask,
                    const void* src, int64_t src_bytes, int64_t T,
                    void* const* dst, int64_t ld, void* cuda_stream,
                    void* const* layer_events) {
  return decompress_impl(c, layer0, nlayers, kv_mask, src, src_bytes, nullptr,
                         T, dst, ld, cuda_stream, layer_events);
}

int kvtc_decompress_packed(const kvtc_calib* c, int layer0, int nlayers,
                           int kv_mask, const void* src, int64_t src_bytes,
                           const int64_t* offsets, int64_t T, void* const* dst,
                           int64_t ld, void* cuda_stream,
                           void* const* layer_events) {
  if (!offsets) return KVTC_EINVAL;
  return decompress_impl(c, layer0, nlayers, kv_mask, src, src_bytes, offsets,
                         T, dst, ld, cuda_stream, layer_events);
}

int kvtc_decompress_paged(const kvtc_calib* c, int layer0, int nlayers,
                          int kv_mask, const void* const* src, const int64_t* T,
                          int R, const int32_t* block_table, int max_blocks,
                          int block_size, void* const* cache,
                          int64_t num_blocks, void* cuda_stream) {
  if (!c || !src || !T || R < 0 || R > 4096 || !block_table || !cache ||
      max_blocks <= 0 || num_blocks <= 0)
    return KVTC_EINVAL;
  if (block_size != 16) return KVTC_ENOTSUP;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  if (cs.empty() || R == 0) return KVTC_OK;
  const int D = c->hs[cs[0]].D;
  for (size_t i = 0; i < cs.size(); ++i) {
    if (c->hs[cs[i]].D != D) return KVTC_ENOTSUP;
    if (!cache[slot[i]]) return KVTC_EINVAL;
    if (!aligned16(cache[slot[i]])) return KVTC_EALIGN;
  }
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0) return KVTC_EALIGN;
  for (int r = 0; r < R; ++r) {
    if (!src[r] || T[r] < 0 || T[r] > (1LL << 31) - 1) return KVTC_EINVAL;
    if (!aligned16(src[r])) return KVTC_EALIGN;
    if ((T[r] + block_size - 1) / block_size > max_blocks) return KVTC_ESIZE;
  }
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  std::vector<const void*> in(R);
  for (int r = 0; r < R; ++r) {
    st = resolve_input(src[r], &in[r]);
    if (st != KVTC_OK) return st;
  }
  PagedParams* p = new (std::nothrow) PagedParams;
  if (!p) return KVTC_ENOMEM;
  const HostStream& h0 = c->hs[cs[0]];
  int ret = KVTC_OK;
  // launches over groups of up to kPagedMaxReq requests and kPagedMaxStream
  // streams (each stream of a group has its own pool tensor map)
  for (size_t j0 = 0; j0 < cs.size() && ret == KVTC_OK; j0 += kPagedMaxStream) {
    const size_t j1 = std::min(cs.size(), j0 + (size_t)kPagedMaxStream);
    const int ns = (int)(j1 - j0);
    for (int r0 = 0; r0 < R && ret == KVTC_OK; r0 += kPagedMaxReq) {
      const int r1 = std::min(R, r0 + kPagedMaxReq);
      std::memset(p, 0, sizeof(*p));
      int64_t tiles = 0;
      int64_t raw_chunks = 0;
      const int cpr = 2 * D / 16;
      for (int r = r0; r < r1; ++r) {
        int64_t s_, w_, tc;
        split_tokens(T[r], c->sink, c->window, &s_, &w_, &tc);
        const int i = r - r0;
        p->src[i] = static_cast<const uint8_t*>(in[r]);
        p->sbytes[i] = stream_bytes_of(c, h0, T[r]);
        p->tc[i] = (int32_t)tc;
        p->s_[i] = (int32_t)s_;
        p->raw_rows[i] = (int32_t)(s_ + w_);
        p->tile_begin[i] = (int32_t)tiles;
        p->raw_begin[i] = raw_chunks;
        p->req_index[i] = r;
        tiles += paged_tiles((int)s_, (int)tc);
        raw_chunks += (int64_t)ns * (s_ + w_) * cpr;
      }
      // stream-major: every stream of the launch has the same tiles
      if (tiles * ns > INT32_MAX) {
        ret = KVTC_ESIZE;
        break;
      }
      p->tile_begin[r1 - r0] = (int32_t)tiles;
      p->raw_begin[r1 - r0] = raw_chunks;
      tiles *= ns;
      int rmax = 0, kmax = 0;
      for (size_t j = j0; j < j1; ++j) {
        const int jl = (int)(j - j0);
        p->cache[jl] = static_cast<char*>(cache[slot[j]]);
        p->cs[jl] = cs[j];
        p->sidx[jl] = (int32_t)j;
        rmax = std::max(rmax, c->hs[cs[j]].R);
        kmax = std::max(kmax, c->hs[cs[j]].k);
        if (!encode_pool_3d(&p->tm_cache[jl], cache[slot[j]], (uint64_t)D,
                            (uint64_t)num_blocks))
          ret = KVTC_ECUDA;
      }
      if (ret != KVTC_OK) break;
      p->streams = c->d_streams;
      p->status = c->d_status;
      p->block_table = block_table;
      p->num_blocks = num_blocks;
      p->max_blocks = max_blocks;
      p->block_size = block_size;
      p->nreq = r1 - r0;
      p->nstream = ns;
      p->total_tiles = (int32_t)tiles;
      p->D = D;
      p->total_raw_chunks = raw_chunks;
      p->rec_words = rmax / 4;
      p->wide = kmax > kNarrowK;
      p->nstages = decompress_stages(p->rec_words);
      if (launch_paged_raw(*p, stream) != cudaSuccess) ret = KVTC_ECUDA;
      const int mp =
          max_pairs_decompress(decompress_smem_bytes(p->nstages, p->rec_words));
      if (ret == KVTC_OK && tiles &&
          (mp < 1 ||
           launch_decompress_paged(*p, pairs_for(mp, (int)tiles), stream) !=
               cudaSuccess))
        ret = KVTC_ECUDA;
    }
  }
  delete p;
  return ret;
}

// ------------------------------------------------------------ field packing
namespace {

// Used bytes of a codec record: per active group its two fp16 fields and
// its b bit-planes of two bytes.
int record_used(const HostStream& h) {
  int u = 0;
  for (uint8_t b : h.widths)
    if (b) u += 4 + 2 * b;
  return u;
}

// Worst-case packed bytes of one stream (every slot needing 6 offset bits
// gives the longest packed record: the used bytes, padded to 4).
int64_t fp_bound_of(const kvtc_calib* c, const HostStream& h, int64_t T) {
  int64_t s_, w_, tc;
  split_tokens(T, c->sink, c->window, &s_, &w_, &tc);
  return align_up(fp_prefix_bytes(h.Ga) + (s_ + w_) * h.D * 2 +
                      tc * align_up(record_used(h), 4),
                  256);
}

// Fill the launch parameters of streams [i0, i1) of a field-packing call.
void fp_fill(FpParams* p, const kvtc_calib* c, const std::vector<int>& cs,
             const std::vector<int64_t>& codec_off, size_t i0, size_t i1,
             int64_t T) {
  std::memset(p, 0, sizeof(*p));
  int64_t s_, w_, tc;
  split_tokens(T, c->sink, c->window, &s_, &w_, &tc);
  int items = 0;
  for (size_t i = i0; i < i1; ++i) {
    const HostStream& h = c->hs[cs[i]];
    FpStream& f = p->s[i - i0];
    f.in_off = codec_off[i];
    f.out_off = codec_off[i];
    f.raw_bytes = (s_ + w_) * h.D * 2;
    f.tc = (int32_t)tc;
    f.tile = (int16_t)((kFpRawChunk / h.R) & ~15);
    f.ntiles = (int32_t)((tc + f.tile - 1) / f.tile);
    f.nraw = (int32_t)((f.raw_bytes + kFpRawChunk - 1) / kFpRawChunk);
    f.ga = (int16_t)h.Ga;
    f.used = (int16_t)record_used(h);
    f.R = (int16_t)h.R;
    f.item_begin = items;
    items += f.ntiles + f.nraw;
  }
  p->n = (int32_t)(i1 - i0);
  p->first = (int32_t)i0;
  p->total_items = items;
}

// Field packing holds one field slot per lane of a warp: at most 15 active
// groups (30 slots) per stream.
int fp_supported(const kvtc_calib* c, const std::vector<int>& cs) {
  for (int i : cs)
    if (c->hs[i].Ga > 15) return KVTC_ENOTSUP;
  return KVTC_OK;
}

}  // namespace

int64_t kvtc_fields_bound(const kvtc_calib* c, int layer0, int nlayers,
                          int kv_mask, int64_t T) {
  if (!c || T < 0 || T > (1LL << 31) - 1) return KVTC_EINVAL;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  if ((st = fp_supported(c, cs)) != KVTC_OK) return st;
  int64_t n = 0;
  for (int i : cs) n += fp_bound_of(c, c->hs[i], T);
  return n;
}

int64_t kvtc_fields_workspace_bytes(const kvtc_calib* c, int layer0,
                                    int nlayers, int kv_mask) {
  if (!c) return KVTC_EINVAL;
  std::vector<int> cs, slot;
  const int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  const int64_t n = std::min<int64_t>((int64_t)cs.size(), kFpMaxStream);
  return std::max<int64_t>(n, 1) * kFpChunks * kFpWorkWords * 4;
}

int kvtc_fields_pack(const kvtc_calib* c, int layer0, int nlayers,
                     int kv_mask, const void* src, int64_t src_bytes,
                     int64_t T, void* dst, int64_t dst_capacity,
                     int64_t* offsets, void* workspace,
                     int64_t workspace_bytes, void* cuda_stream) {
  if (!c || !dst || !offsets || !workspace || T < 0 || T > (1LL << 31) - 1)
    return KVTC_EINVAL;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  if (cs.empty()) return KVTC_EINVAL;
  if ((st = fp_supported(c, cs)) != KVTC_OK) return st;
  std::vector<int64_t> off(cs.size());
  int64_t need = 0, bound = 0;
  for (size_t i = 0; i < cs.size(); ++i) {
    off[i] = need;
    need += stream_bytes_of(c, c->hs[cs[i]], T);
    bound += fp_bound_of(c, c->hs[cs[i]], T);
  }
  if (!src && need) return KVTC_EINVAL;
  if (src_bytes < need || dst_capacity < bound) return KVTC_ESIZE;
  const int64_t ws = std::min<int64_t>((int64_t)cs.size(), kFpMaxStream) *
                     kFpChunks * kFpWorkWords * 4;
  if (workspace_bytes < ws) return KVTC_ESIZE;
  if (!aligned16(src) || !aligned16(dst) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(offsets) & 7u))
    return KVTC_EALIGN;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  FpParams* p = new (std::nothrow) FpParams;
  if (!p) return KVTC_ENOMEM;
  int ret = KVTC_OK;
  for (size_t i0 = 0; i0 < cs.size() && ret == KVTC_OK; i0 += kFpMaxStream) {
    const size_t i1 = std::min(cs.size(), i0 + (size_t)kFpMaxStream);
    fp_fill(p, c, cs, off, i0, i1, T);
    p->in = static_cast<const uint8_t*>(src);
    p->out = static_cast<uint8_t*>(dst);
    p->offsets = offsets;
    p->work = static_cast<uint32_t*>(workspace);
    p->status = c->d_status;
    p->in_bytes = src_bytes;
    if (launch_fields_pack(*p, static_cast<cudaStream_t>(cuda_stream)) !=
        cudaSuccess)
      ret = KVTC_ECUDA;
  }
  delete p;
  return ret;
}

int kvtc_fields_unpack(const kvtc_calib* c, int layer0, int nlayers,
                       int kv_mask, const void* src, int64_t src_bytes,
                       const int64_t* offsets, int64_t T, void* dst,
                       int64_t dst_bytes, void* cuda_stream) {
  if (!c || !src || !offsets || T < 0 || T > (1LL << 31) - 1)
    return KVTC_EINVAL;
  std::vector<int> cs, slot;
  int st = select_streams(c, layer0, nlayers, kv_mask, &cs, &slot);
  if (st != KVTC_OK) return st;
  if (cs.empty()) return KVTC_EINVAL;
  if ((st = fp_supported(c, cs)) != KVTC_OK) return st;
  std::vector<int64_t> off(cs.size());
  int64_t need = 0;
  for (size_t i = 0; i < cs.size(); ++i) {
    off[i] = need;
    need += stream_bytes_of(c, c->hs[cs[i]], T);
  }
  if (!dst && need) return KVTC_EINVAL;
  if (dst_bytes < need) return KVTC_ESIZE;
  if (src_bytes < (int64_t)cs.size() * 256) return KVTC_ESIZE;
  if (!aligned16(src) || !aligned16(dst) ||
      (reinterpret_cast<uintptr_t>(offsets) & 7u))
    return KVTC_EALIGN;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  FpParams* p = new (std::nothrow) FpParams;
  if (!p) return KVTC_ENOMEM;
  int ret = KVTC_OK;
  for (size_t i0 = 0; i0 < cs.size() && ret == KVTC_OK; i0 += kFpMaxStream) {
    const size_t i1 = std::min(cs.size(), i0 + (size_t)kFpMaxStream);
    fp_fill(p, c, cs, off, i0, i1, T);
    p->in = static_cast<const uint8_t*>(src);
    p->out = static_cast<uint8_t*>(dst);
    p->offsets = const_cast<int64_t*>(offsets);
    p->status = c->d_status;
    p->in_bytes = src_bytes;
    if (launch_fields_unpack(*p, static_cast<cudaStream_t>(cuda_stream)) !=
        cudaSuccess)
      ret = KVTC_ECUDA;
  }
  delete p;
  return ret;
}

int kvtc_wait_selftest(const kvtc_calib* c, uint32_t limit_us,
                       void* cuda_stream) {
  if (!c || limit_us < 1 || limit_us > 2000000u) return KVTC_EINVAL;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  return launch_wait_selftest(c->d_status, 1000ull * limit_us,
                              static_cast<cudaStream_t>(cuda_stream)) ==
                 cudaSuccess
             ? KVTC_OK
             : KVTC_ECUDA;
}

int kvtc_device_status(const kvtc_calib* c, void* cuda_stream,
                       unsigned* flags) {
  if (!c || !flags) return KVTC_EINVAL;
  DeviceGuard guard(c->device);
  if (!guard.ok) return KVTC_ECUDA;
  cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
  unsigned v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess ||
      cudaMemcpy(&v, c->d_status, 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(c->d_status, 0, 4) != cudaSuccess)
    return KVTC_ECUDA;
  *flags = v;
  return KVTC_OK;
}

}  // extern "C"
