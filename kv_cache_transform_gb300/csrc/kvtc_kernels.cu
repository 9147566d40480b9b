// sm_103a kernels of the kvtc hot path.
//
//   compress   (kvtc page, technical summary 2B): c = V^T x - V^T mu on the
//              5th-generation tensor cores (bf16 x bf16 -> fp32 in TMEM), run
//              by CTA pairs (M = 256 over the pair) with x and V_enc staged
//              by 3-D TMA boxes of two K blocks, then a fused epilogue of 16
//              warps that quantises each 16-component group with its own
//              fp16 shift/scale (microscaling, 2A) and writes bit-plane
//              records with coalesced 16-byte stores.
//   decompress (2C): a fused prologue unpacks the bit-planes and dequantises
//              each group straight into an fp16 A operand held in TMEM; the
//              tensor cores (CTA pairs, M = 256, N up to 256) form
//              V c_hat + mu (the mean as one more K step) in fp32; the
//              epilogue rounds to bf16 and writes rows with TMA tensor
//              stores (contiguous) or 16-byte stores through the block table
//              (paged).
//   raw rows   (2A): attention-sink and recent-window rows are copied
//              verbatim in 16-byte chunks, by two warps inside the tensor-core
//              kernels (or a copy kernel when nothing is coded).
//
// Every mbarrier wait is bounded; a wait that runs out sets a sticky flag
// and the CTA drains its own copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <type_traits>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"
#include "ptx.cuh"

namespace kvtc {

// Optional per-role timing (compiled in only with -DKVTC_TRACE): each warp
// accumulates the SM cycles it spends in up to eight phases and lane 0
// stores the sums per CTA.  Timestamps only; no work is skipped.
#ifdef KVTC_TRACE
__device__ unsigned long long g_kvtc_trace[2][160][32][8];
#define KVTC_TR_DECL                              \
  unsigned long long tr_[8] = {0, 0, 0, 0, 0, 0, 0, 0}; \
  unsigned long long tr_t = clock64();
#define KVTC_TR(i)                                    \
  {                                                   \
    const unsigned long long tr_n = clock64();        \
    tr_[i] += tr_n - tr_t;                            \
    tr_t = tr_n;                                      \
  }
#define KVTC_TR_SAVE(k)                                  \
  if (lane == 0 && blockIdx.x < 160)                     \
    for (int i_ = 0; i_ < 8; ++i_)                       \
      g_kvtc_trace[k][blockIdx.x][warp][i_] = tr_[i_];
#else
#define KVTC_TR_DECL
#define KVTC_TR(i)
#define KVTC_TR_SAVE(k)
#endif

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  uint32_t s = smem_u32(p);
  uint32_t pad = (1024u - (s & 1023u)) & 1023u;
  return reinterpret_cast<uint8_t*>(a + pad);
}

__device__ __forceinline__ void raise_abort(volatile int* abort_flag,
                                            unsigned* status) {
  *abort_flag = 1;
  atomicOr(status, KVTC_FLAG_TIMEOUT);
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_v4(void* p, uint32_t a, uint32_t b,
                                      uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b,
                                       uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(a),
               "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"((uint16_t)v)
               : "memory");
}

// 4-bit field of w at bit `pos` (one bfe).
__device__ __forceinline__ uint32_t bfe4(uint32_t w, uint32_t pos) {
  uint32_t r;
  asm("bfe.u32 %0, %1, %2, 4;" : "=r"(r) : "r"(w), "r"(pos));
  return r;
}

// Codes of one group from its B bit-planes (16 bits each, at byte offset po
// of the staged record): w_n collects components 4n..4n+3, one code per
// byte.  Plane j's nibble is spread straight to bit j of each byte (the
// spread multiplier and mask shifted by j), so a nibble costs a bfe, a
// multiply and one and-or.  (n * 0x00204081) & 0x01010101 moves bit m of a
// nibble n to bit 8m: the four shifted copies 0, 7, 14, 21 never collide.
template <int B>
__device__ __forceinline__ void unpack_planes(const uint32_t* stg, int po,
                                              int lane, uint32_t& w0,
                                              uint32_t& w1, uint32_t& w2,
                                              uint32_t& w3) {
#pragma unroll
  for (int j = 0; j < B; ++j) {
    const int bo = po + 2 * j;
    const uint32_t word = stg[(bo >> 2) * 33 + lane];
    const uint32_t base = (uint32_t)(bo & 2) << 3;  // low or high half
    const uint32_t mul = 0x00204081u << j;
    const uint32_t mask = 0x01010101u << j;
    w0 |= (bfe4(word, base) * mul) & mask;
    w1 |= (bfe4(word, base + 4u) * mul) & mask;
    w2 |= (bfe4(word, base + 8u) * mul) & mask;
    w3 |= (bfe4(word, base + 12u) * mul) & mask;
  }
}

// Gather bit 0 of each byte of x (x & 0x01010101) into bits 0..3.
__device__ __forceinline__ uint32_t gather4(uint32_t x) {
  return (x * 0x10204080u) >> 28;
}

// Two codes (bytes selected by sel) -> half2 of shift + q * scale, one
// rounding to fp16 (fused multiply-add).
__device__ __forceinline__ uint32_t dequant_pair(uint32_t w, uint32_t sel,
                                                 __half2 sc2, __half2 sh2) {
  uint32_t hb = __byte_perm(w, 0x64646464u, sel);  // fp16 1024 + q
  __half2 h = *reinterpret_cast<__half2*>(&hb);
  h = __hsub2(h, __half2half2(__ushort_as_half((unsigned short)0x6400)));
  h = __hfma2(h, sc2, sh2);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Tensor store shared -> global of one box, tracked by the thread's bulk
// group.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t x,
                                             int32_t y, const void* ssrc) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], "
      "[%3];" ::"l"(tmap),
      "r"(x), "r"(y), "r"(smem_u32(ssrc))
      : "memory");
}

__device__ __forceinline__ void tma_store_3d(const void* tmap, int32_t x,
                                             int32_t y, int32_t z,
                                             const void* ssrc) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, "
      "%3}], [%4];" ::"l"(tmap),
      "r"(x), "r"(y), "r"(z), "r"(smem_u32(ssrc))
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Raw rows (sink and window, and zero padding) of a RawList, copied in
// 16-byte chunks by the `stride` threads of the raw-copy role across the
// grid (thread `tid` of them), four chunks in flight per thread.  Runs
// beside the tensor-core work of the same kernel.  kPk: segments may sit in
// packed streams (restore from packed input), read where the stream's
// offsets frame them; kHdr: and only when the stream's header holds the
// magic and T_c (in the restore kernel the prologue checks the header of
// every stream, as it has coded tokens, so the copy skips that read).
template <bool kPk = false, bool kHdr = false>
__device__ __forceinline__ void raw_list_copy(const RawList& r, int64_t tid,
                                              int64_t stride,
                                              unsigned* status) {
  int sg = 0;  // chunks visit increasing indices, so the segment only grows
  for (int64_t c0 = tid; c0 < r.total_chunks; c0 += 4 * stride) {
    uint4 v[4];
    char* d[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t c = c0 + u * stride;
      d[u] = nullptr;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (c < r.total_chunks) {
        while (sg + 1 < r.nseg && r.seg[sg + 1].chunk_begin <= c) ++sg;
        const RawListSeg& g = r.seg[sg];
        const int64_t cpr = g.row_bytes >> 4;
        const int64_t local = c - g.chunk_begin;
        const int64_t row = local / cpr;
        const int64_t col = local - row * cpr;
        const char* src = g.src;
        if (kPk && g.pk >= 0) {
          // rows of a packed stream: found through its offsets, and only
          // read when they lie inside the stream and the input
          const int64_t o0 = r.pk_offs[g.pk], o1 = r.pk_offs[g.pk + 1];
          const int64_t need = g.pk_off + (int64_t)g.rows * g.row_bytes;
          src = nullptr;
          if (o0 >= 0 && ((o0 | o1) & 15) == 0 && o1 >= o0 + need &&
              o1 <= r.pk_bytes) {
            const uint32_t* hd =
                reinterpret_cast<const uint32_t*>(r.pk_base + o0);
            if (!kHdr ||
                (__ldg(hd) == kFpMagic && (int32_t)__ldg(hd + 1) == g.pk_tc))
              src = reinterpret_cast<const char*>(r.pk_base) + o0 + g.pk_off;
          }
          if (!src) {
            if (col == 0 && row == 0) atomicOr(status, KVTC_FLAG_FORMAT);
            continue;
          }
        }
        if (src) v[u] = ld_nc_v4(src + row * g.src_ld + col * 16);
        d[u] = g.dst + row * g.dst_ld + col * 16;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (d[u]) *reinterpret_cast<uint4*>(d[u]) = v[u];
  }
}

// Raw rows of packed streams that have no coded token: the RawList copy on
// its own, every thread of the grid one copier.
__global__ void __launch_bounds__(256)
    raw_list_kernel(const __grid_constant__ RawList r, unsigned* status) {
  raw_list_copy<true, true>(r, (int64_t)blockIdx.x * 256 + threadIdx.x,
                            (int64_t)gridDim.x * 256, status);
}

// ======================================================================
//                               decompress
// ======================================================================
// 0 TMA, 1 MMA, 2-9 prologue, 10-25 epilogue, 26-27 raw rows
constexpr int kDecWarps = 28;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecMaxNC = 256;  // widest output chunk (one MMA's N)
constexpr int kDecMaxStages = 8;
// one B stage = this CTA's half of a chunk, up to four K blocks:
// [kbs][nc/2][64]; a chunk takes one stage (k + 16 <= 256) or two
constexpr int kDecMaxKbs = 4;
constexpr int kDecBStage = (kDecMaxNC / 2) * 128 * kDecMaxKbs;
constexpr int kDecStgWarp = 32 * 128;  // 32 rows x 64 bf16, SW128
constexpr int kDecBarBytes = 512;
// Shared memory: [B ring: nstages x 64 KB][staging: 16 warps x 4 KB]
// [records: 8 warps x rec_words x 33 u32][barriers][misc].  The ring is as
// deep as fits: two stages for records up to 128 bytes, one (the B load of
// the next chunk waits for the MMAs of this one) for longer records.
int decompress_smem_bytes(int nstages, int rec_words) {
  return nstages * kDecBStage + 16 * kDecStgWarp + 8 * rec_words * 33 * 4 +
         kDecBarBytes + 64 + 1024;
}
int decompress_stages(int rec_words) {
  int n = kDecMaxStages;
  while (n > 1 && decompress_smem_bytes(n, rec_words) > 232448) --n;
  return n;
}
// TMEM columns: accumulators in [0, 256) (256 / nc of them, nc columns
// each), A operands at 256 and 384.
constexpr uint32_t kDecTmemCols = 512;


struct DecTile {
  const uint8_t* rec;  // record of compressed token 0 of the stream
  char* dst;           // contiguous: output row of compressed token 0
  int64_t ld_bytes;
  char* cache;         // paged: pool of this stream
  int tc, tile, cs, s_, req;
  int seg;             // output tensor map: contiguous segment, or paged
                       // stream of the launch
};


__device__ __forceinline__ DecTile resolve(const DecParams& p, int item) {
  const int lo = item / p.tiles_per_seg;
  const DecSeg& g = p.seg[lo];
  DecTile t;
  t.rec = g.rec;
  t.dst = g.dst;
  t.ld_bytes = g.ld_bytes;
  t.cache = nullptr;
  t.tc = g.tc;
  t.tile = item - lo * p.tiles_per_seg;
  t.cs = g.cs;
  t.seg = lo;
  t.s_ = 0;
  t.req = 0;
  return t;
}

__device__ __forceinline__ DecTile resolve(const PagedParams& p, int item) {
  const int per = max(1, p.tile_begin[p.nreq]);  // tiles of one stream
  const int j = item / per;
  const int idx = item - j * per;
  int lo = 0, hi = p.nreq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.tile_begin[mid] <= idx) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  DecTile t;
  t.tile = idx - p.tile_begin[r];
  t.cs = p.cs[j];
  t.tc = p.tc[r];
  t.rec = p.src[r] + (int64_t)p.sidx[j] * p.sbytes[r] +
          (int64_t)p.raw_rows[r] * p.D * 2;
  t.dst = nullptr;
  t.ld_bytes = 0;
  t.cache = p.cache[j];
  t.s_ = p.s_[r];
  t.req = p.req_index[r];
  t.seg = j;
  return t;
}

// kLayout of a launch: 0 (narrow) when every stream has k <= 240: two
// 128-column A buffers, one B stage per chunk; 2 (wide) when a stream has
// k > 240: one 256-column A buffer and up to two B stages per chunk; 3 the
// narrow layout reading its records from packed streams (field packing
// holds at most 15 groups).  A template parameter, so that the narrow
// kernel carries none of the others' state.
template <class P, int kLayout>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kDecThreads, 1)
    decompress_kernel(const __grid_constant__ P p) {
  constexpr bool kWide = kLayout == 2;
  // kLayout 3: narrow, records read from packed streams
  constexpr bool kPacked = kLayout == 3;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nst = p.nstages;
  const int rec_words = p.rec_words;
  uint8_t* sB = smem;
  uint8_t* sStg = smem + nst * kDecBStage;
  uint32_t* sRec = reinterpret_cast<uint32_t*>(sStg + 16 * kDecStgWarp);
  uint64_t* bar = reinterpret_cast<uint64_t*>(
      reinterpret_cast<uint8_t*>(sRec) + 8 * rec_words * 33 * 4);
  uint64_t* full_b = bar;                       // [nst], leader's used
  uint64_t* empty_b = bar + kDecMaxStages;      // [nst]
  uint64_t* a_full = bar + 2 * kDecMaxStages;   // [2], leader's used
  uint64_t* a_empty = a_full + 2;               // [2]
  uint64_t* acc_full = a_full + 4;              // [4]
  uint64_t* acc_empty = a_full + 8;             // [4], leader's used
  uint64_t* mma_done = a_full + 12;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(
      reinterpret_cast<uint8_t*>(bar) + kDecBarBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The CTA pair (a cluster of two) restores 256-token super-tiles: CTA
  // `rank` owns rows [128 rank, 128 rank + 128) of each and the rank-th half
  // of every V_dec chunk; the leader (rank 0) issues the M = 256 MMAs.
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full_b[i], 1);
      mbar_init(&empty_b[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      // the prologue warps that fill a buffer, in each CTA: one set of 4,
      // or in a wide launch both sets (8), each with half of the groups
      mbar_init(&a_full[i], kWide ? 16 : 8);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&acc_full[i], 1);
      // the epilogue warps of both CTAs that read a chunk arrive with
      // counts adding up to 32 whatever the chunk width
      mbar_init(&acc_empty[i], 32);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kDecTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = p.total_tiles;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      KVTC_TR_DECL
      uint32_t it_b = 0, s = 0, ph = 0;
      bool ok = true;
      const uint32_t full_leader = mapa_shared(smem_u32(full_b), 0);
      for (int item = pair; item < total && ok; item += npairs) {
        const DecTile t = resolve(p, item);
        const DevStream* ds = p.streams + t.cs;
        const int nc = ds->nc, nch = ds->D / nc, half = nc >> 1;
        const int kbs = ds->kbs, nbs = kWide ? ds->nbs : 1;
        // both halves of the chunk, kbs K blocks (a box past the last K
        // block is filled with zeros and still counts its full bytes)
        const uint32_t bytes_pair = (uint32_t)nc * 128u * (uint32_t)kbs;
        if (item == pair) prefetch_tmap(&ds->tm_vdec);
        for (int ch = 0; ch < nch && ok; ++ch) {
          for (int h = 0; h < nbs; ++h) {
            KVTC_TR(0)
            if (!mbar_wait(&empty_b[s], ph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full_b[s], bytes_pair);
            KVTC_TR(1)
            tma_load_3d_pair(sB + s * kDecBStage, &ds->tm_vdec, 0,
                             ch * nc + (int)rank * half, h * kbs,
                             full_leader + s * 8u);
            ++it_b;
            if (++s == (uint32_t)nst) {
              s = 0;
              ph ^= 1u;
            }
            KVTC_TR(2)
          }
        }
      }
      KVTC_TR(0)
      KVTC_TR_SAVE(0)
      if (!ok) raise_abort(abort_flag, p.status);
      if (leader) {
        // the leader's full barriers count both CTAs' loads
        for (uint32_t s2 = 0; s2 < (uint32_t)nst; ++s2) {
          if (it_b > s2) {
            const uint32_t last = s2 + nst * ((it_b - 1 - s2) / nst);
            mbar_drain(&full_b[s2], (last / nst) & 1u);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (leader)
    if (lane == 0 && leader) {
      KVTC_TR_DECL
      uint32_t chunk = 0, it = 0, s = 0, ph = 0;
      bool ok = true;
      // the next chunk's accumulator and B stage, when already known ready
      bool acc_ready = false, b_ready = false;
      const uint64_t desc_b0 = sw128_desc(smem_u32(sB));
      // wide launch: the tile's first K-step slot of the cyclic A region
      uint32_t slot0 = 0;
      for (int item = pair; item < total && ok; item += npairs) {
        const DecTile t = resolve(p, item);
        KVTC_TR(7)
        const DevStream* ds = p.streams + t.cs;
        const int nc = ds->nc, nch = ds->D / nc;
        // 256 / nc accumulators of nc columns: log2 of their count
        const uint32_t lg = nc == 256 ? 0u : nc == 128 ? 1u : 2u;
        const uint32_t nbm = (1u << lg) - 1u;
        const int ksteps = ds->kp / kGroup;  // kept groups + the mean step
        const int kb_units = (ds->nc / 2) * 128 / 16;  // one K block, >> 4
        const int sstep = 4 * ds->kbs;       // K steps per B stage
        const int nbs = kWide ? ds->nbs : 1;
        const uint32_t idesc = make_idesc(256, (uint32_t)nc, 0);
        // A buffers: two of 128 columns, or (wide launch) a cyclic region
        // of 32 K-step slots of 8 columns where tiles take their ksteps
        // slots one after another; the barriers alternate by tile
        const uint32_t abuf = it & 1u;
        const uint32_t ause = it >> 1;
        KVTC_TR(0)
        if (!mbar_wait(&a_full[abuf], ause & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        KVTC_TR(1)
        const uint32_t a_col = tmem + 256u + abuf * 128u;
        for (int ch = 0; ch < nch && ok; ++ch) {
          const uint32_t accb = chunk & nbm;
          KVTC_TR(0)
          if (!acc_ready &&
              !mbar_wait(&acc_empty[accb], ((chunk >> lg) & 1u) ^ 1u,
                         abort_flag)) {
            ok = false;
            break;
          }
          KVTC_TR(2)
          const uint32_t d = tmem + accb * (uint32_t)nc;
          const uint32_t c_next = chunk + 1;
          for (int h = 0; h < nbs; ++h) {
            KVTC_TR(0)
            if (!b_ready && !mbar_wait(&full_b[s], ph, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            KVTC_TR(3)
            // K block kb of this stage lies at kb * half * 128 bytes; the
            // descriptor start address advances 32 bytes (2 units) per
            // K=16.  The tensor pipe queues almost nothing ahead, so a
            // stage's steps are one unrolled, branch-free run of predicated
            // MMAs whose operands are all simple offsets of two registers.
            const uint64_t bdesc =
                desc_b0 + (uint64_t)(s * (kDecBStage >> 4));
            const int step0 = h * sstep;
            const int nsteps = min(ksteps - step0, sstep);
            const uint32_t a_h = a_col + (uint32_t)step0 * 8u;
            const uint32_t sl_h = slot0 + (uint32_t)step0;
            // the next stage's and the next chunk's barriers are tested
            // (never waited on) right after the first MMA, so the test
            // overlaps the MMA run
            const uint32_t s_next = s + 1 == (uint32_t)nst ? 0u : s + 1;
            const uint32_t ph_next = s + 1 == (uint32_t)nst ? ph ^ 1u : ph;
#pragma unroll
            for (int step = 0; step < 4 * kDecMaxKbs; ++step) {
              mma_ts_pair_if(d,
                             kWide ? tmem + 256u +
                                         (((sl_h + (uint32_t)step) & 31u) << 3)
                                   : a_h + (uint32_t)step * 8u,
                             bdesc + (uint64_t)((step >> 2) * kb_units +
                                                (step & 3) * 2),
                             idesc, (h | step) > 0, step < nsteps);
              if (step == 0) {
                acc_ready = mbar_test_wait(&acc_empty[c_next & nbm],
                                           ((c_next >> lg) & 1u) ^ 1u);
                b_ready = mbar_test_wait(&full_b[s_next], ph_next);
              }
            }
            tc_commit_pair(&empty_b[s], 3);
            if (++s == (uint32_t)nst) {
              s = 0;
              ph ^= 1u;
            }
            KVTC_TR(4)
          }
          if (!ok) break;
          tc_commit_pair(&acc_full[accb], 3);
          KVTC_TR(5)
          ++chunk;
        }
        if (!ok) break;
        tc_commit_pair(&a_empty[abuf], 3);
        KVTC_TR(6)
        ++it;
        slot0 = (slot0 + (uint32_t)ksteps) & 31u;
      }
      KVTC_TR(0)
      KVTC_TR_SAVE(0)
      if (!ok) raise_abort(abort_flag, p.status);
      tc_commit_pair(mma_done, 3);
    }
    if (lane == 0) mbar_drain(mma_done, 0);
    __syncwarp();
  } else if (warp < 10) {
    // ------------------------------------ prologue: unpack + dequantise
    // Two sets of four warps (one per TMEM lane quadrant each): set 0 builds
    // the A operand of the even super-tiles (buffer 0), set 1 of the odd;
    // in a wide launch both sets build every tile's, half of its groups
    // each.
    const int q = warp & 3;
    const uint32_t set = (uint32_t)(warp - 2) >> 2;
    uint32_t* stg = sRec + (warp - 2) * (rec_words * 33);
    const uint32_t a_full_leader = mapa_shared(smem_u32(a_full), 0);
    uint32_t it = 0;
    bool ok = true;
    // Packed input: the offsets, header and slot table of the set's next
    // tile are loaded while this one is decoded (registers; an offset of -1
    // marks a stream whose offsets do not frame its header and table), so
    // each tile waits on memory once, for its records.
    int64_t nx_o0 = -1, nx_o1 = 0;
    uint32_t nx_hw = 0;
    // wide launch: the tile's first slot of the cyclic A region (32 K-step
    // slots of 8 columns, tiles taking Ga + 1 of them one after another)
    // and the slot count of the tile before
    uint32_t slot0 = 0;
    int n_prev = 0;
    const auto pk_fetch = [&](int itm) {
      nx_o0 = -1;
      nx_o1 = 0;
      nx_hw = 0;
      if constexpr (kPacked) {
      if (itm >= total) return;
      const int sg = itm / p.tiles_per_seg;
      const int gn = p.streams[p.seg[sg].cs].Ga;
      const int64_t a0 = p.raw.pk_offs[sg + p.pk_first];
      const int64_t a1 = p.raw.pk_offs[sg + p.pk_first + 1];
      if (a0 >= 0 && ((a0 | a1) & 15) == 0 && a1 >= a0 + fp_prefix_bytes(gn) &&
          a1 <= p.raw.pk_bytes) {
        nx_o0 = a0;
        nx_o1 = a1;
        // the 128-byte prefix (header, slot table) in one load, a word a
        // lane; the slot entries are unpacked when the tile starts
        nx_hw = __ldg(reinterpret_cast<const uint32_t*>(p.raw.pk_base + a0) +
                      lane);
      }
      }
    };
    if constexpr (kPacked) pk_fetch(pair + (int)set * npairs);
    KVTC_TR_DECL
    for (int item = pair; item < total; item += npairs, ++it) {
      // A buffers: two of 128 columns, each filled by its own set of warps
      // on alternate tiles; or (wide launch) a cyclic region of 256 columns
      // filled by both sets together tile after tile, each decoding half of
      // the groups.  Both sets see every tile there; a tile's slots are
      // released by its MMAs (barriers alternating by tile, as for the two
      // buffers), and a warp writes only after the release of the tile two
      // back (and, for the slots it shares with it, of the tile before),
      // so no wait is ever two phases ahead (where a parity wait cannot
      // tell the phase it wants from the one before)
      if (!kWide && (it & 1u) != set) continue;
      const uint32_t abuf = it & 1u;
      const uint32_t ause = it >> 1;
      const DecTile t = resolve(p, item);
      const DevStream* ds = p.streams + t.cs;
      const int R = ds->R, Ga = ds->Ga;
      // group widths and plane offsets: lane a holds group a's (Ga <= 31),
      // broadcast per group by shuffle
      const int my_b = lane < Ga ? (int)ds->bits[lane] : 0;
      const int my_po = lane < Ga ? (int)ds->poff[lane] : 0;
      const int row0 = t.tile * kPairM + (int)rank * kTileM + q * 32;
      // record index of the warp's first row: rows are tokens for paged
      // output (its tiles start at token 0), records otherwise; lanes
      // [lo, hi) have a record, the others decode zeros
      const int rec0 =
          std::is_same<P, PagedParams>::value ? row0 - t.s_ : row0;
      const int lo = max(-rec0, 0);
      const int hi = min(max(t.tc - rec0, 0), 32);
      const uint8_t* rbase = t.rec + (int64_t)rec0 * R;
      // Packed input: the stream's header and slot table (lane s = field
      // slot s: vmin, code bits d, bit position of its code), checked
      // against the calibration, T and the offsets before anything they
      // frame is read; its records are Rp bytes long.
      int pk_vmin = 0, pk_d = 0, pk_pos = 0, pk_hb2 = 0, pk_rp = 0;
      int pk_po = 0;
      uint32_t pk_grp = 0;
      bool pk_ok = false;
      if constexpr (kPacked) {
        const int ns = 2 * Ga;
        const int64_t o0 = nx_o0, o1 = nx_o1;   // fetched for this tile
        const uint32_t hw = nx_hw;              // prefix word `lane`
        // slot `lane`'s entry: halfword lane of the table (word 4 + lane/2)
        const uint32_t tw = __shfl_sync(0xFFFFFFFFu, hw, (4 + (lane >> 1)) & 31);
        const uint32_t te = lane < ns ? (tw >> ((lane & 1) << 4)) & 0xFFFFu : 0u;
        const int pre = fp_prefix_bytes(Ga);  // header + slot table
        const int64_t rawb = (int64_t)p.pk_raw_rows * ds->D * 2;
        const bool in = o0 >= 0;
        const uint8_t* sb = p.raw.pk_base + (in ? o0 : 0);
        pk_vmin = (int)(te & 0xFFu);
        pk_d = (int)(te >> 8);
        const int wbits = lane < ns ? pk_d + 2 : 0;
        int incl = wbits;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
          if (lane >= o) incl += v;
        }
        pk_pos = incl - wbits;
        pk_hb2 = (__shfl_sync(0xFFFFFFFFu, incl, 31) + 15) >> 4;
        const int used = __shfl_sync(0xFFFFFFFFu, my_po, Ga - 1) +
                         2 * __shfl_sync(0xFFFFFFFFu, my_b, Ga - 1);
        pk_rp = fp_record_bytes(Ga, pk_hb2, used);
        const uint32_t h0 = __shfl_sync(0xFFFFFFFFu, hw, 0);
        const uint32_t h1 = __shfl_sync(0xFFFFFFFFu, hw, 1);
        const uint32_t h2 = __shfl_sync(0xFFFFFFFFu, hw, 2);
        const bool slot_ok = lane >= ns || (pk_d <= 6 && pk_vmin <= 63);
        pk_ok = __all_sync(0xFFFFFFFFu, slot_ok) && in && h0 == kFpMagic &&
                (int)h1 == t.tc && (int)(h2 & 0xFFFFu) == pk_rp &&
                (int)(h2 >> 16) == ns &&
                o0 + pre + rawb + (int64_t)t.tc * pk_rp <= o1;
        if (!pk_ok) {
          // decoded as all-zero records: zero fields, codes and planes
          pk_vmin = pk_d = pk_pos = pk_hb2 = 0;
          if (lane == 0 && q == 0 && rank == 0)
            atomicOr(p.status, KVTC_FLAG_FORMAT);
        }
        rbase = sb + pre + rawb + (int64_t)row0 * pk_rp;
        // lane a (< Ga): group a's two slots in one word -- the bit where
        // slot 2a's code starts (the codes begin at halfword Ga), the two
        // code widths less 2 and the two 4 vmin
        const int v0 = __shfl_sync(0xFFFFFFFFu, pk_vmin, (2 * lane) & 31);
        const int v1 = __shfl_sync(0xFFFFFFFFu, pk_vmin, (2 * lane + 1) & 31);
        const int d0 = __shfl_sync(0xFFFFFFFFu, pk_d, (2 * lane) & 31);
        const int d1 = __shfl_sync(0xFFFFFFFFu, pk_d, (2 * lane + 1) & 31);
        const int bp = 16 * Ga + __shfl_sync(0xFFFFFFFFu, pk_pos,
                                             (2 * lane) & 31);
        pk_grp = (uint32_t)bp | ((uint32_t)d0 << 10) | ((uint32_t)d1 << 13) |
                 ((uint32_t)(v0 & 63) << 18) | ((uint32_t)(v1 & 63) << 26);
        pk_po = my_po - 2 * Ga + 2 * pk_hb2;  // planes follow the codes
      }
      if constexpr (kPacked) {
        // the warp's packed records are 32 Rp contiguous bytes (whole
        // 128-byte lines of the stream: Rp is a multiple of 4 and the
        // records start on a line); coalesced 16-byte loads, each word
        // stored at its token's place in the word-transposed staging
        const int nvalid = pk_ok ? min(max(t.tc - row0, 0), 32) : 0;
        // tokens without a record (past T_c, or all of an invalid stream)
        // decode from zeros, as in the codec layout
        if (nvalid < 32) {
          const int nz = 32 - nvalid;
          for (int i = lane; i < rec_words * nz; i += 32)
            stg[(i / nz) * 33 + nvalid + i % nz] = 0u;
        }
        const int wpr = pk_rp >> 2;
        const int nchunk = (nvalid * pk_rp + 15) >> 4;
        for (int c0 = 0; c0 < nchunk; c0 += 8 * 32) {
          uint4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            v[u] = c < nchunk ? ld_nc_v4(rbase + 16 * c)
                              : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c >= nchunk) continue;
            const uint32_t wv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            int tr = (4 * c) / wpr;
            int wd = 4 * c - tr * wpr;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (tr < nvalid) stg[wd * 33 + tr] = wv[j];
              if (++wd == wpr) {
                wd = 0;
                ++tr;
              }
            }
          }
        }
        pk_fetch(item + 2 * npairs);  // the set's next tile
      } else {
      // Coalesced 16-byte loads of the warp's 32 records (up to eight in
      // flight per lane), stored word-transposed ([word][token], row pitch
      // 33) in shared memory; done before waiting for the A buffer so the
      // memory latency overlaps the MMAs still reading it.
      const int nld = (32 * R) >> 9;  // 16-byte loads per lane
      for (int b0 = 0; b0 < nld; b0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int o = (b0 + u) * 512 + lane * 16;
          v[u] = make_uint4(0u, 0u, 0u, 0u);
          if (b0 + u < nld && o / R >= lo && o / R < hi)
            v[u] = ld_nc_v4(rbase + o);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          if (b0 + u >= nld) break;
          const int o = (b0 + u) * 512 + lane * 16;
          const int tr = o / R;
          const int wd = (o - tr * R) >> 2;
          stg[(wd + 0) * 33 + tr] = v[u].x;
          stg[(wd + 1) * 33 + tr] = v[u].y;
          stg[(wd + 2) * 33 + tr] = v[u].z;
          stg[(wd + 3) * 33 + tr] = v[u].w;
        }
      }
      }
      KVTC_TR(2)
      if (!mbar_wait(&a_empty[abuf], (ause & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      KVTC_TR(1)
      __syncwarp();
      KVTC_TR(2)
      const uint32_t a_tmem = tmem + ((uint32_t)(q * 32) << 16) + 256u +
                              (kWide ? 0u : abuf * 128u);
      // groups [g0, g1) of this warp, and whether it writes the mean step
      const int gh = (Ga + 1) >> 1;
      const int g0 = kWide && set ? gh : 0, g1 = kWide && !set ? gh : Ga;
      // Wide launch: K step a of this tile lives in slot slot0 + a (mod 32).
      // The wait above released the slots of the tile two back; the first
      // 32 - n_prev steps miss the slots of the tile before, so they are
      // written while its MMAs still run, and the others after its release.
      const int conflict_from = it == 0u ? 32 : 32 - n_prev;
      bool prev_free = false;
      const auto a_col = [&](int a) -> uint32_t {
        return kWide ? ((slot0 + (uint32_t)a) & 31u) << 3 : (uint32_t)a * 8u;
      };
      const auto claim = [&](int a) -> bool {
        if (!kWide || prev_free || a < conflict_from) return true;
        if (!mbar_wait(&a_empty[abuf ^ 1u], ((it - 1u) >> 1) & 1u,
                       abort_flag))
          return false;
        tc_fence_after();
        __syncwarp();
        prev_free = true;
        return true;
      };
      for (int a = g0; a < g1; ++a) {
        if (!claim(a)) {
          ok = false;
          break;
        }
        const int b = __shfl_sync(0xFFFFFFFFu, my_b, a);
        int po;
        uint32_t f;
        if constexpr (kPacked) {
          // packed record: the low bytes of the 2 Ga fields, the codes of
          // their high bytes (per slot, high byte - 4 vmin in d + 2 bits),
          // the bit-planes
          po = __shfl_sync(0xFFFFFFFFu, pk_po, a);
          const uint32_t e = __shfl_sync(0xFFFFFFFFu, pk_grp, a);
          const uint32_t wi = min((e & 1023u) >> 5, (uint32_t)rec_words - 2u);
          const uint32_t bits = __funnelshift_r(
              stg[wi * 33 + lane], stg[(wi + 1) * 33 + lane], e & 31u);
          // code = high byte - 4 vmin, in d + 2 bits
          const uint32_t d0 = (e >> 10) & 7u, d1 = (e >> 13) & 7u;
          const uint32_t c0 = bits & ((4u << d0) - 1u);
          const uint32_t c1 = (bits >> (d0 + 2u)) & ((4u << d1) - 1u);
          const uint32_t h0 = (c0 + ((e >> 16) & 0xFCu)) & 0xFFu;
          const uint32_t h1 = (c1 + ((e >> 24) & 0xFCu)) & 0xFFu;
          const uint32_t lo16 = stg[(a >> 1) * 33 + lane] >> ((a & 1) << 4);
          // shift = lo byte 0 | h0 << 8, scale = lo byte 1 | h1 << 8
          f = __byte_perm(lo16, h0 | (h1 << 8), 0x5140);
        } else {
          po = __shfl_sync(0xFFFFFFFFu, my_po, a);
          f = stg[a * 33 + lane];
        }
        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
        switch (b) {  // uniform over the warp
          case 1: unpack_planes<1>(stg, po, lane, w0, w1, w2, w3); break;
          case 2: unpack_planes<2>(stg, po, lane, w0, w1, w2, w3); break;
          case 3: unpack_planes<3>(stg, po, lane, w0, w1, w2, w3); break;
          case 4: unpack_planes<4>(stg, po, lane, w0, w1, w2, w3); break;
          case 5: unpack_planes<5>(stg, po, lane, w0, w1, w2, w3); break;
          case 6: unpack_planes<6>(stg, po, lane, w0, w1, w2, w3); break;
          case 7: unpack_planes<7>(stg, po, lane, w0, w1, w2, w3); break;
          default: unpack_planes<8>(stg, po, lane, w0, w1, w2, w3); break;
        }
        const __half2 sh2 =
            __half2half2(__ushort_as_half((unsigned short)(f & 0xFFFFu)));
        const __half2 sc2 =
            __half2half2(__ushort_as_half((unsigned short)(f >> 16)));
        uint32_t out[8];
        out[0] = dequant_pair(w0, 0x4140u, sc2, sh2);
        out[1] = dequant_pair(w0, 0x4342u, sc2, sh2);
        out[2] = dequant_pair(w1, 0x4140u, sc2, sh2);
        out[3] = dequant_pair(w1, 0x4342u, sc2, sh2);
        out[4] = dequant_pair(w2, 0x4140u, sc2, sh2);
        out[5] = dequant_pair(w2, 0x4342u, sc2, sh2);
        out[6] = dequant_pair(w3, 0x4140u, sc2, sh2);
        out[7] = dequant_pair(w3, 0x4342u, sc2, sh2);
        tmem_st8(a_tmem + a_col(a), out);
      }
      if (!ok) break;
      if (!kWide || set) {
        // the mean step: A = (1, 1, 0, ..., 0) against (mu_hi, mu_lo, 0...)
        if (!claim(Ga)) {
          ok = false;
          break;
        }
        const uint32_t ones[8] = {0x3C003C00u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        tmem_st8(a_tmem + a_col(Ga), ones);
      }
      KVTC_TR(3)
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(a_full_leader + abuf * 8u);
      KVTC_TR(4)
      if constexpr (kWide) {
        slot0 = (slot0 + (uint32_t)(Ga + 1)) & 31u;
        n_prev = Ga + 1;
      }
    }
    KVTC_TR(0)
    KVTC_TR_SAVE(0)
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  } else if (warp >= 26) {
    // ------------------------------- raw rows (sink and window) back
    if constexpr (std::is_same<P, DecParams>::value)
      raw_list_copy<kPacked>(
          p.raw, (int64_t)blockIdx.x * 64 + (warp - 26) * 32 + lane,
          (int64_t)gridDim.x * 64, p.status);
  } else {
    // -------------- epilogue: bf16 rows (the mean came in the MMA)
    // Sixteen warps.  With 256 / nc accumulators, 16 nc / 256 warps read
    // each chunk (group g takes the chunks in accumulator g); within a
    // group, sets of four warps (one per TMEM lane quadrant each) split the
    // chunk's columns 64 apiece, so an accumulator is released after one
    // TMEM round trip of every warp of its group.  A warp stages its 32
    // rows x 64 columns as one 128-byte-swizzled box and writes it with a
    // TMA tensor store (contiguous output) or with coalesced 16-byte
    // stores through the block table (paged).
    constexpr bool kPaged = std::is_same<P, PagedParams>::value;
    const int e = warp - 10;
    const int q = warp & 3;
    uint8_t* stg_w = sStg + e * kDecStgWarp;
    const uint32_t sw = (uint32_t)(lane & 7);
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
    uint32_t chunk = 0;
    bool ok = true;
    KVTC_TR_DECL
    for (int item = pair; item < total && ok; item += npairs) {
      const DecTile t = resolve(p, item);
      const DevStream* ds = p.streams + t.cs;
      const int D = ds->D, nc = ds->nc, nch = D / nc;
      const uint32_t lg = nc == 256 ? 0u : nc == 128 ? 1u : 2u;
      const uint32_t nbm = (1u << lg) - 1u;
      // warps per chunk 16 >> lg; this warp's group and 64-column set
      const uint32_t grp = (uint32_t)e >> (4 - lg);
      const int col0 = ((e & ((16 >> lg) - 1)) >> 2) * 64;
      const int wrow0 = t.tile * kPairM + (int)rank * kTileM + q * 32;
      // Paged: rows are tokens, and the warp's 32 are the 16-token blocks
      // wrow0 / 16 and the one after.  A block whose 16 tokens all have
      // records goes out as one TMA tensor store (full0 / full1); the
      // rows of a block that also holds sink, window or no tokens go out
      // one by one (rowp non-null for this lane's row).
      int blk0 = -1, blk1 = -1;
      bool full0 = false, full1 = false, any_rows = false;
      char* rowp = nullptr;
      if constexpr (kPaged) {
        const int c_lo = t.s_, c_hi = t.s_ + t.tc;  // tokens with records
        int id = -1;
        if (lane < 2) {
          const int bi = wrow0 / 16 + lane;
          if (bi * 16 + 16 > c_lo && bi * 16 < c_hi) {  // holds coded rows
            id = bi < p.max_blocks
                     ? __ldg(p.block_table + (int64_t)t.req * p.max_blocks + bi)
                     : -1;
            if (id < 0 || (int64_t)id >= p.num_blocks) {
              atomicOr(p.status, KVTC_FLAG_BLOCK);
              id = -1;
            }
          }
        }
        blk0 = __shfl_sync(0xFFFFFFFFu, id, 0);
        blk1 = __shfl_sync(0xFFFFFFFFu, id, 1);
        full0 = blk0 >= 0 && wrow0 >= c_lo && wrow0 + 16 <= c_hi;
        full1 = blk1 >= 0 && wrow0 + 16 >= c_lo && wrow0 + 32 <= c_hi;
        const int tok = wrow0 + lane;
        const int myblk = lane < 16 ? blk0 : blk1;
        const bool myfull = lane < 16 ? full0 : full1;
        if (!myfull && myblk >= 0 && tok >= c_lo && tok < c_hi)
          rowp = t.cache + ((int64_t)myblk * 16 + (tok & 15)) * D * 2;
        any_rows = __any_sync(0xFFFFFFFFu, rowp != nullptr);
      }
      for (int ch = 0; ch < nch; ++ch, ++chunk) {
        const uint32_t accb = chunk & nbm;
        if (accb != grp) continue;
        KVTC_TR(0)
        if (!mbar_wait(&acc_full[accb], (chunk >> lg) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        KVTC_TR(1)
        // 64 columns as 32 bf16 pairs, packed 32 columns at a time
        uint32_t pk[32];
        {
          const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) +
                                 accb * (uint32_t)nc + (uint32_t)col0;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)hh * 32u, v);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              pk[16 * hh + i] = pack_bf16(v[2 * i], v[2 * i + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
          mbar_arrive_cluster_n(acc_empty_leader + accb * 8u, 1u << lg);
        KVTC_TR(4)
        if (lane == 0) bulk_wait_read<0>();  // the last store read stg_w
        __syncwarp();
        KVTC_TR(5)
        const uint32_t srow = smem_u32(stg_w) + lane * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          sts_v4(srow + (((uint32_t)i ^ sw) << 4), pk[4 * i], pk[4 * i + 1],
                 pk[4 * i + 2], pk[4 * i + 3]);
        KVTC_TR(2)
        if constexpr (!kPaged) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (wrow0 < t.tc)
              tma_store_2d(&p.tm_out[t.seg], ch * nc + col0, wrow0, stg_w);
            bulk_commit();
          }
        } else {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // whole blocks: rows 0-15 and 16-31 of the box are the two
            // blocks (the 128-byte swizzle repeats every 8 rows)
            if (full0)
              tma_store_3d(&p.tm_cache[t.seg], ch * nc + col0, 0, blk0, stg_w);
            if (full1)
              tma_store_3d(&p.tm_cache[t.seg], ch * nc + col0, 0, blk1,
                           stg_w + 16 * 128);
            bulk_commit();
          }
          if (any_rows) {
            // the other coded rows: 8 lanes per 128-byte row, four rows
            // per store instruction (unrolled by two only: fully unrolled,
            // its live values push the kernel past its register cap)
#pragma unroll 2
            for (int r0 = 0; r0 < 32; r0 += 4) {
              const int r = r0 + (lane >> 3);
              const int sub = lane & 7;
              char* rp = reinterpret_cast<char*>(__shfl_sync(
                  0xFFFFFFFFu, reinterpret_cast<uintptr_t>(rowp), r));
              const uint4 val = *reinterpret_cast<const uint4*>(
                  stg_w + r * 128 + ((sub ^ (r & 7)) << 4));
              if (rp)
                *reinterpret_cast<uint4*>(rp + (int64_t)(ch * nc + col0) * 2 +
                                          sub * 16) = val;
            }
          }
          __syncwarp();
        }
        KVTC_TR(3)
      }
    }
    if (lane == 0) bulk_wait<0>();
    KVTC_TR(0)
    KVTC_TR_SAVE(0)
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  }

  // No CTA of the pair may leave while the other can still reach its
  // barriers, shared memory or TMEM.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kDecTmemCols);
  }
  cluster_sync();
}
// ======================================================================
//                                compress
// ======================================================================
// 0 TMA, 1 MMA, 2-17 epilogue (four sets), 18-19 raw rows
constexpr int kCompWarps = 20;
constexpr int kCompThreads = kCompWarps * 32;
constexpr int kCompMaxStages = 6;
constexpr int kCompAStage = kTileM * 128;          // [128 rows][64 bf16]
constexpr uint32_t kCompTmemCols = 512;            // accumulators at 0, 256

int compress_smem_bytes(int nstages, int stage_bytes, int rec_stg_words) {
  return nstages * stage_bytes + 8 * rec_stg_words * 33 * 4 + 256 + 64 + 1024;
}

__device__ __forceinline__ int find_comp_seg(const CompParams& p, int item) {
  return item / p.tiles_per_seg;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kCompThreads, 1)
    compress_kernel(const __grid_constant__ CompParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nst = p.nstages;
  const int stage_bytes = p.stage_bytes;
  uint32_t* sRec = reinterpret_cast<uint32_t*>(smem + nst * stage_bytes);
  const int rec_words = p.rec_stg_words;
  uint64_t* bar =
      reinterpret_cast<uint64_t*>(smem + nst * stage_bytes + 8 * rec_words * 33 * 4);
  uint64_t* full = bar;
  uint64_t* empty = bar + kCompMaxStages;
  uint64_t* acc_full = bar + 2 * kCompMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_full + 4;
  uint64_t* rec_full = acc_full + 5;  // [2 buffers][4 quadrants]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 33);
  // tokens whose fields left the fp16 range, per lane quadrant: three tile
  // slots in rotation [3][4]
  uint32_t* range_mask = reinterpret_cast<uint32_t*>(bar + 34);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The CTA pair (a cluster of two) codes 256-token super-tiles: CTA `rank`
  // loads rows [128 rank, 128 rank + 128) and the rank-th half of V_enc's
  // components; the leader (rank 0) issues the M = 256 MMAs.
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 32);  // 16 epilogue warps in each CTA
    }
    for (int i = 0; i < 8; ++i) mbar_init(&rec_full[i], 4);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    for (int i = 0; i < 12; ++i) range_mask[i] = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kCompTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = p.total_tiles;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      KVTC_TR_DECL
      uint32_t it_b = 0, s = 0, ph = 0;
      bool ok = true;
      const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
      for (int item = pair; item < total && ok; item += npairs) {
        const int sg = find_comp_seg(p, item);
        const CompSeg& g = p.seg[sg];
        const int tile = item - sg * p.tiles_per_seg;
        const DevStream* ds = p.streams + g.cs;
        const int nkb = ds->D / kAtomK;
        const int half = ds->k >> 1;
        // a stage is kps K blocks; both CTAs' x tiles and V_enc halves land
        // on the leader's barrier (a box past the last K block is filled
        // with zeros and still counts its full bytes)
        const int kps = p.kps;
        const uint32_t bytes_pair =
            2u * (uint32_t)kps * ((uint32_t)kCompAStage + (uint32_t)half * 128u);
        for (int kb = 0; kb < nkb; kb += kps) {
          KVTC_TR(0)
          if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          KVTC_TR(1)
          uint8_t* st = smem + s * stage_bytes;
          if (leader) mbar_arrive_expect_tx(&full[s], bytes_pair);
          tma_load_3d_pair(st, &g.tm_x, 0,
                           g.row0 + tile * kPairM + (int)rank * kTileM, kb,
                           full_leader + s * 8u);
          tma_load_3d_pair(st + kps * kCompAStage,
                           kps == 2 ? &ds->tm_venc : &ds->tm_venc1, 0,
                           (int)rank * half, kb, full_leader + s * 8u);
          ++it_b;
          if (++s == (uint32_t)nst) {
            s = 0;
            ph ^= 1u;
          }
          KVTC_TR(2)
        }
      }
      KVTC_TR(0)
      KVTC_TR_SAVE(1)
      if (!ok) raise_abort(abort_flag, p.status);
      if (leader) {
        // the leader's full barriers count both CTAs' loads
        for (uint32_t s = 0; s < (uint32_t)nst; ++s) {
          if (it_b > s) {
            const uint32_t last = s + nst * ((it_b - 1 - s) / nst);
            mbar_drain(&full[s], (last / nst) & 1u);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------- MMA issuer (leader)
    if (lane == 0 && leader) {
      KVTC_TR_DECL
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      const uint64_t desc_s0 = sw128_desc(smem_u32(smem));
      const uint64_t stage_units = (uint64_t)(stage_bytes >> 4);
      const int kps = p.kps;
      const uint64_t b_units = (uint64_t)((kps * kCompAStage) >> 4);
      const uint64_t a_kb_units = (uint64_t)(kCompAStage >> 4);
      for (int item = pair; item < total && ok; item += npairs) {
        const CompSeg& g = p.seg[find_comp_seg(p, item)];
        const DevStream* ds = p.streams + g.cs;
        const int nkb = ds->D / kAtomK;
        // N = k as one MMA per K step, or for k > 256 two: N = 256 into
        // accumulator columns [0, 256) from rows [0, 128) of each CTA's
        // V_enc half, and N = k - 256 into [256, k) from the rows after
        // (the rows are stored so that column j is component j)
        const uint32_t n1 = ds->k > 256 ? 256u : (uint32_t)ds->k;
        const uint32_t n2 = ds->k > 256 ? (uint32_t)ds->k - 256u : 0u;
        const uint32_t idesc = make_idesc(256, n1, 1);
        const uint32_t idesc2 = make_idesc(256, n2 ? n2 : 16u, 1);
        // one K block of this CTA's V_enc half, in 16-byte units
        const uint64_t b_kb_units = (uint64_t)((ds->k >> 1) * 128 / 16);
        // double-buffered accumulators, or one of k columns (wide launch)
        const uint32_t accb = p.wide ? 0u : it & 1u;
        const uint32_t ause = p.wide ? it : it >> 1;
        KVTC_TR(0)
        if (!mbar_wait(&acc_empty[accb], (ause & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        KVTC_TR(1)
        const uint32_t d = tmem + accb * 256u;
        for (int kb = 0; kb < nkb; kb += kps) {
          KVTC_TR(0)
          if (!mbar_wait(&full[s], ph, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          KVTC_TR(2)
          // kps K blocks, four K=16 steps each: one unrolled run (a second
          // block predicated off past the last K block, or in one-block
          // stages)
          const uint64_t ad = desc_s0 + s * stage_units;
          const uint64_t bd = ad + b_units;
          const uint32_t two = kps == 2 && kb + 1 < nkb;
          // (the tensor pipe queues almost nothing ahead, so a tile with
          // one MMA per K step runs without the second, predicated-off
          // instruction between its MMAs)
          if (n2 == 0) {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int st = 0; st < 4; ++st)
                mma_ss_pair_if(d, ad + (uint64_t)j * a_kb_units + 2u * st,
                               bd + (uint64_t)j * b_kb_units + 2u * st, idesc,
                               (kb | j | st) != 0, j == 0 || two);
          } else {
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int st = 0; st < 4; ++st) {
                mma_ss_pair_if(d, ad + (uint64_t)j * a_kb_units + 2u * st,
                               bd + (uint64_t)j * b_kb_units + 2u * st, idesc,
                               (kb | j | st) != 0, j == 0 || two);
                // rows [128, k/2) of the half: 128 rows x 128 B further
                mma_ss_pair_if(
                    d + 256u, ad + (uint64_t)j * a_kb_units + 2u * st,
                    bd + (uint64_t)j * b_kb_units + 2u * st + 1024u, idesc2,
                    (kb | j | st) != 0, j == 0 || two);
              }
          }
          tc_commit_pair(&empty[s], 3);
          if (++s == (uint32_t)nst) {
            s = 0;
            ph ^= 1u;
          }
          KVTC_TR(3)
        }
        if (!ok) break;
        tc_commit_pair(&acc_full[accb], 3);
        ++it;
      }
      KVTC_TR(0)
      KVTC_TR_SAVE(1)
      if (!ok) raise_abort(abort_flag, p.status);
      tc_commit_pair(mma_done, 3);
    }
    if (lane == 0) mbar_drain(mma_done, 0);
    __syncwarp();
  } else if (warp >= 18) {
    // ---------------------------- raw rows (sink, window) and padding
    raw_list_copy(p.raw, (int64_t)blockIdx.x * 64 + (warp - 18) * 32 + lane,
                  (int64_t)gridDim.x * 64, p.status);
  } else {
    // ------------------------- epilogue: quantise + bit-plane records
    // Four sets of four warps (one per TMEM lane quadrant each) share every
    // tile: set s codes the s-th quarter of the kept groups (in pairs), so
    // an accumulator is released after a quarter of a tile's work and four
    // warps per scheduler hide each other's latency.  The four warps of a
    // quadrant build their 32 tokens' records in one staging buffer (two
    // buffers alternate between tiles), meet on an mbarrier, and each
    // writes a quarter of the records out.
    const int q = warp & 3;
    const uint32_t set = (uint32_t)(warp - 2) >> 2;
    const uint32_t acc_empty_leader = mapa_shared(smem_u32(acc_empty), 0);
    uint32_t it = 0;
    bool ok = true;
    KVTC_TR_DECL
    for (int item = pair; item < total; item += npairs, ++it) {
      // accumulator (double-buffered, or one of k columns in a wide
      // launch) and record staging buffer (always two, alternating)
      const uint32_t accb = p.wide ? 0u : it & 1u;
      const uint32_t ause = p.wide ? it : it >> 1;
      const uint32_t sb = it & 1u;
      uint32_t* stg = sRec + (sb * 4u + (uint32_t)q) * (rec_words * 33);
      const uint32_t stg_addr = smem_u32(stg);
      const int sg = find_comp_seg(p, item);
      const CompSeg& g = p.seg[sg];
      const int tile = item - sg * p.tiles_per_seg;
      const DevStream* ds = p.streams + g.cs;
      const int R = ds->R, Ga = ds->Ga;
      // set s: groups [s gq, s gq + gq) within [0, Ga); gq even (pairs of
      // groups per TMEM load)
      const int gq = ((Ga + 7) >> 3) << 1;
      const int a_begin = min(Ga, (int)set * gq);
      const int a_end = min(Ga, (int)set * gq + gq);
      KVTC_TR(0)
      if (!mbar_wait(&acc_full[accb], ause & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      KVTC_TR(1)
      const int row0 = tile * kPairM + (int)rank * kTileM + q * 32;
      const int nvalid = min(max(g.tc - row0, 0), 32);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + accb * 256u;
      // Range masks rotate over three slots.  Set 0 clears the slot of tile
      // it + 1 here: that slot last held tile it - 2, whose records every set
      // has written before arriving for tile it - 1 (which set 0 has waited
      // for), and no set can mark tile it + 1 before passing tile it's
      // barrier, which waits for this warp.
      const uint32_t mslot = it % 3u;
      if (set == 0 && lane == 0)
        range_mask[((it + 1u) % 3u) * 4u + (uint32_t)q] = 0u;
      if ((int)set == (Ga ? (Ga - 1) / gq : 0)) {
        // the warp coding the last group zeroes the record's padding:
        // fields and planes cover bytes [0, used) exactly
        const int used = Ga ? ds->poff[Ga - 1] + 2 * ds->bits[Ga - 1] : 0;
        if (used & 2)
          sts_u16(stg_addr + (uint32_t)(((used >> 2) * 33 + lane) * 4 + 2),
                  0u);
        for (int w = (used + 3) >> 2; w < (R >> 2); ++w) stg[w * 33 + lane] = 0u;
      }
      if (a_begin >= a_end) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_leader + accb * 8u);
      }
      bool range_err = false;
      for (int a0 = a_begin; a0 < a_end; a0 += 2) {
        // two groups per TMEM round trip (the second may lie past k when Ga
        // is odd; it is inside the allocation and left unused)
        float v2[32];
        tmem_ld32(taddr + (uint32_t)a0 * 16u, v2);
        tmem_wait_ld();
        if (a0 + 2 >= a_end) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_leader + accb * 8u);
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int a = a0 + h;
          if (a >= a_end) break;
          float* v = v2 + 16 * h;
          const float4* m4 = reinterpret_cast<const float4*>(ds->m + a * 16);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 mm = __ldg(m4 + i);
            v[4 * i] -= mm.x;
            v[4 * i + 1] -= mm.y;
            v[4 * i + 2] -= mm.z;
            v[4 * i + 3] -= mm.w;
          }
          float lo = v[0], hi = v[0];
#pragma unroll
          for (int i = 1; i < 16; ++i) {
            lo = fminf(lo, v[i]);
            hi = fmaxf(hi, v[i]);
          }
          const int b = ds->bits[a];
          const int po = ds->poff[a];
          const float lev = (float)((1 << b) - 1);
          const __half sh = __float2half_rd(lo);
          const float shf = __half2float(sh);
          // scale = the least fp16 s with s * lev >= hi - shift: an upper
          // bound of the quotient rounded up to fp16 lands on s or on the
          // fp16 value after it; the product of the value before with lev
          // (at most 11 + 8 significant bits) is exact in fp32, so one
          // comparison settles which
          const float dif = __fsub_ru(hi, shf);
          __half sc = __float2half_ru(__fmul_ru(dif, __frcp_ru(lev)));
          {
            const unsigned short sb = __half_as_ushort(sc);
            if (sb > 0u && sb < 0x7C00u) {
              const __half below = __ushort_as_half((unsigned short)(sb - 1u));
              if (__half2float(below) * lev >= dif) sc = below;
            }
          }
          const float scf = __half2float(sc);
          range_err |= __hisinf(sh) != 0 || __hisinf(sc) != 0 ||
                       __hisnan(sh) || __hisnan(sc);
          const float inv = scf > 0.f ? __frcp_rn(scf) : 0.f;
          uint32_t cb[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float u = fmaf(v[i] - shf, inv, 0.5f);
            u = fminf(fmaxf(u, 0.f), lev);
            cb[i] = __float_as_uint(__fadd_rd(u, 8388608.f));  // low byte = q
          }
          uint32_t w[4];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            w[kk] = __byte_perm(__byte_perm(cb[4 * kk], cb[4 * kk + 1], 0x0040u),
                                __byte_perm(cb[4 * kk + 2], cb[4 * kk + 3],
                                            0x0040u),
                                0x5410u);
          stg[a * 33 + lane] = (uint32_t)__half_as_ushort(sh) |
                               ((uint32_t)__half_as_ushort(sc) << 16);
          for (int j = 0; j < b; ++j) {
            uint32_t plane = 0;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              plane |= gather4((w[kk] >> j) & 0x01010101u) << (4 * kk);
            const int bo = po + 2 * j;
            sts_u16(
                stg_addr + (uint32_t)(((bo >> 2) * 33 + lane) * 4 + (bo & 2)),
                plane);
          }
        }
      }
      // a token whose fields left the fp16 range raises the sticky flag and
      // its record is not written
      const uint32_t bad = __ballot_sync(0xFFFFFFFFu, range_err && lane < nvalid);
      if (bad && lane == 0) {
        atomicOr(p.status, KVTC_FLAG_RANGE);
        atomicOr(&range_mask[mslot * 4u + (uint32_t)q], bad);
      }
      __syncwarp();
      KVTC_TR(2)
      // all four warps of the quadrant have staged their groups
      if (lane == 0) mbar_arrive(&rec_full[sb * 4u + (uint32_t)q]);
      if (!mbar_wait(&rec_full[sb * 4u + (uint32_t)q], (it >> 1) & 1u,
                     abort_flag)) {
        ok = false;
        break;
      }
      const uint32_t skip =
          *reinterpret_cast<volatile uint32_t*>(&range_mask[mslot * 4u + (uint32_t)q]);
      // set s writes tokens [8 s, 8 s + 8) of the quadrant
      uint8_t* rbase = g.rec + (int64_t)row0 * R;
      const int o_end = (int)(set + 1) * 8 * R;
      for (int o = (int)set * 8 * R + lane * 16; o < o_end; o += 512) {
        const int tr = o / R;
        const int wd = (o - tr * R) >> 2;
        if (tr < nvalid && !((skip >> tr) & 1u))
          st_v4(rbase + o, stg[wd * 33 + tr], stg[(wd + 1) * 33 + tr],
                stg[(wd + 2) * 33 + tr], stg[(wd + 3) * 33 + tr]);
      }
      __syncwarp();
      KVTC_TR(3)
    }
    KVTC_TR(0)
    KVTC_TR_SAVE(1)
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  }

  // No CTA of the pair may leave while the other can still reach its
  // barriers, shared memory or TMEM.
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kCompTmemCols);
  }
  cluster_sync();
}

// ======================================================================
//                                raw rows
// ======================================================================
// Self-test of the bounded wait every kernel above relies on: one thread
// waits on an mbarrier that nothing will ever arrive at, with a short limit;
// when the limit runs out it raises the same sticky flag the kernels raise
// and returns, leaving the context usable.
__global__ void __launch_bounds__(32) wait_selftest_kernel(unsigned* status,
                                                           uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 &&
      !mbar_wait_for(&bar, 0u, &abort_flag, limit_ns))
    atomicOr(status, KVTC_FLAG_TIMEOUT);
}

__global__ void __launch_bounds__(256) raw_copy_kernel(
    const __grid_constant__ RawParams p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       c < p.total_chunks; c += stride) {
    int lo = 0, hi = p.nseg - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (p.seg[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
    }
    const RawSeg& g = p.seg[lo];
    const int cpr = g.row_bytes >> 4;
    const int64_t local = c - g.chunk_begin;
    const int64_t row = local / cpr;
    const int col = (int)(local - row * cpr);
    const uint4 v = ld_nc_v4(g.src + row * g.src_ld + col * 16);
    *reinterpret_cast<uint4*>(g.dst + row * g.dst_ld + col * 16) = v;
  }
}

__global__ void __launch_bounds__(256) paged_raw_kernel(
    const __grid_constant__ PagedParams p) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int row_bytes = p.D * 2;
  const int cpr = row_bytes >> 4;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
       c < p.total_raw_chunks; c += stride) {
    int lo = 0, hi = p.nreq - 1;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (p.raw_begin[mid] <= c) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int64_t per_stream = (int64_t)p.raw_rows[r] * cpr;
    const int64_t local = c - p.raw_begin[r];
    const int j = (int)(local / per_stream);
    const int64_t rem = local - j * per_stream;
    const int rr = (int)(rem / cpr);
    const int col = (int)(rem - (int64_t)rr * cpr);
    const int s_ = p.s_[r];
    const int tok = rr < s_ ? rr : s_ + p.tc[r] + (rr - s_);
    const int bi = tok / p.block_size;
    if (bi >= p.max_blocks) {
      atomicOr(p.status, KVTC_FLAG_BLOCK);
      continue;
    }
    const int blk = p.block_table[(int64_t)p.req_index[r] * p.max_blocks + bi];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
      atomicOr(p.status, KVTC_FLAG_BLOCK);
      continue;
    }
    const uint4 v = ld_nc_v4(p.src[r] + (int64_t)p.sidx[j] * p.sbytes[r] +
                             (int64_t)rr * row_bytes + col * 16);
    char* dst = p.cache[j] +
                ((int64_t)blk * p.block_size + tok % p.block_size) * row_bytes +
                col * 16;
    *reinterpret_cast<uint4*>(dst) = v;
  }
}

// ======================================================================
//                                launchers
// ======================================================================
#ifdef KVTC_TRACE
}  // namespace kvtc
extern "C" int kvtc_trace_read(void* host, size_t bytes) {
  if (bytes < sizeof(kvtc::g_kvtc_trace)) return KVTC_ESIZE;
  return cudaMemcpyFromSymbol(host, kvtc::g_kvtc_trace,
                              sizeof(kvtc::g_kvtc_trace)) == cudaSuccess
             ? KVTC_OK
             : KVTC_ECUDA;
}
namespace kvtc {
#endif

static int max_pairs(const void* func, int threads, int smem) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cfg.gridDim = dim3(2 * (sms / 2), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, func, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return sms / 2;
  }
  return n;
}

static void allow_smem(const void* func, int bytes) {
  cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       bytes);
}

int max_pairs_compress(int smem_bytes) {
  allow_smem((const void*)compress_kernel, 232448);
  return max_pairs((const void*)compress_kernel, kCompThreads, smem_bytes);
}

int max_pairs_decompress(int smem_bytes) {
  allow_smem((const void*)decompress_kernel<DecParams, 0>, 232448);
  return max_pairs((const void*)decompress_kernel<DecParams, 0>, kDecThreads,
                   smem_bytes);
}

cudaError_t launch_compress(const CompParams& p, int pairs, cudaStream_t st) {
  const int smem = compress_smem_bytes(p.nstages, p.stage_bytes, p.rec_stg_words);
  allow_smem((const void*)compress_kernel, 232448);
  compress_kernel<<<2 * pairs, kCompThreads, smem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

template <class P, int kLayout>
static cudaError_t launch_dec_as(const P& p, int pairs, cudaStream_t st) {
  allow_smem((const void*)decompress_kernel<P, kLayout>, 232448);
  decompress_kernel<P, kLayout>
      <<<2 * pairs, kDecThreads, decompress_smem_bytes(p.nstages, p.rec_words),
         st>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_raw_list(const RawList& r, unsigned* status,
                            cudaStream_t st) {
  if (r.total_chunks <= 0) return cudaSuccess;
  const int64_t b = (r.total_chunks + 1023) / 1024;
  raw_list_kernel<<<(int)std::min<int64_t>(b, 4 * 152), 256, 0, st>>>(r,
                                                                     status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_decompress(const DecParams& p, int pairs, cudaStream_t st) {
  return p.packed ? launch_dec_as<DecParams, 3>(p, pairs, st)
         : p.wide ? launch_dec_as<DecParams, 2>(p, pairs, st)
                  : launch_dec_as<DecParams, 0>(p, pairs, st);
}

cudaError_t launch_decompress_paged(const PagedParams& p, int pairs,
                                    cudaStream_t st) {
  return p.wide ? launch_dec_as<PagedParams, 2>(p, pairs, st)
                : launch_dec_as<PagedParams, 0>(p, pairs, st);
}

cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns,
                                 cudaStream_t st) {
  count_launch();
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_raw_copy(const RawParams& p, cudaStream_t st) {
  if (p.total_chunks == 0) return cudaSuccess;
  int64_t blocks = (p.total_chunks + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  raw_copy_kernel<<<(int)blocks, 256, 0, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_paged_raw(const PagedParams& p, cudaStream_t st) {
  if (p.total_raw_chunks == 0) return cudaSuccess;
  int64_t blocks = (p.total_raw_chunks + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  paged_raw_kernel<<<(int)blocks, 256, 0, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvtc
