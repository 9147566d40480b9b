// sm_103a kernels of the kvtc hot path.
//
//   compress   (kvtc page, technical summary 2B): c = V^T x - V^T mu on the
//              5th-generation tensor cores (bf16 x bf16 -> fp32 in TMEM, both
//              operands staged by TMA with the 128-byte swizzle), then a fused
//              epilogue that quantises each 16-component group with its own
//              fp16 shift/scale (microscaling, 2A) and writes bit-plane
//              records with coalesced 16-byte stores.
//   decompress (2C): a fused prologue unpacks the bit-planes and dequantises
//              each group straight into an fp16 A operand held in TMEM; the
//              tensor cores form V c_hat (fp16 x fp16 -> fp32) in 128-column
//              chunks; the epilogue adds mu, rounds to bf16 and writes rows
//              with bulk copies (contiguous or block-paged).
//   raw rows   (2A): attention-sink and recent-window rows are copied
//              verbatim in 16-byte chunks.
//
// Every mbarrier wait is bounded; a wait that runs out sets a sticky flag
// and the CTA drains its own copies and MMAs, frees TMEM and returns.
#include <type_traits>

#include "../../include/kvtc.h"
#include "kvtc_internal.cuh"
#include "ptx.cuh"

namespace kvtc {

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

// Spread the 4 bits of n into bit 0 of each byte: bit m -> bit 8m.
__device__ __forceinline__ uint32_t spread4(uint32_t n) {
  return (n * 0x00204081u) & 0x01010101u;
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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ======================================================================
//                               decompress
// ======================================================================
constexpr int kDecWarps = 10;  // 0 TMA, 1 MMA, 2-5 prologue, 6-9 epilogue
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecNC = 128;
constexpr int kDecStages = 4;
constexpr int kDecBStage = kDecNC * 128;           // [128 rows][64 fp16]
constexpr int kDecStgRow = kDecNC * 2 + 16;        // padded staging row
constexpr int kDecStgWarp = 32 * kDecStgRow;
constexpr int kRecWords = kMaxRecord / 4;
constexpr int kRecStgWarp = kRecWords * 33 * 4;    // [words][33] u32
constexpr int kDecOffStg = kDecStages * kDecBStage;
constexpr int kDecOffRec = kDecOffStg + 4 * 2 * kDecStgWarp;
constexpr int kDecOffBar = kDecOffRec + 4 * kRecStgWarp;
constexpr int kDecOffMisc = kDecOffBar + 256;
constexpr int kDecSmem = kDecOffMisc + 64 + 1024;
// TMEM columns: accumulators at 0 and 128, A operands at 256 and 384.
constexpr uint32_t kDecTmemCols = 512;

int decompress_smem_bytes() { return kDecSmem; }

struct DecTile {
  const uint8_t* rec;  // record of compressed token 0 of the stream
  char* dst;           // contiguous: output row of compressed token 0
  int64_t ld_bytes;
  char* cache;         // paged: pool of this stream
  int tc, tile, cs, s_, req;
};

__device__ __forceinline__ DecTile resolve(const DecParams& p, int item) {
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.seg[mid].tile_begin <= item) lo = mid; else hi = mid - 1;
  }
  const DecSeg& g = p.seg[lo];
  DecTile t;
  t.rec = g.rec;
  t.dst = g.dst;
  t.ld_bytes = g.ld_bytes;
  t.cache = nullptr;
  t.tc = g.tc;
  t.tile = item - g.tile_begin;
  t.cs = g.cs;
  t.s_ = 0;
  t.req = 0;
  return t;
}

__device__ __forceinline__ DecTile resolve(const PagedParams& p, int item) {
  int lo = 0, hi = p.nreq - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.tile_begin[mid] <= item) lo = mid; else hi = mid - 1;
  }
  const int r = lo;
  const int tiles = max(1, (p.tc[r] + kTileM - 1) / kTileM);
  const int idx = item - p.tile_begin[r];
  const int j = idx / tiles;
  DecTile t;
  t.tile = idx - j * tiles;
  t.cs = p.cs[j];
  t.tc = p.tc[r];
  t.rec = p.src[r] + (int64_t)j * p.sbytes[r] +
          (int64_t)p.raw_rows[r] * p.D * 2;
  t.dst = nullptr;
  t.ld_bytes = 0;
  t.cache = p.cache[j];
  t.s_ = p.s_[r];
  t.req = p.req_index[r];
  return t;
}

template <class P>
__device__ __forceinline__ char* dec_row_ptr(const P& p, const DecTile& t,
                                             int row, int D) {
  if constexpr (std::is_same<P, PagedParams>::value) {
    const int tok = t.s_ + row;
    const int bi = tok / p.block_size;
    if (bi >= p.max_blocks) {
      atomicOr(p.status, KVTC_FLAG_BLOCK);
      return nullptr;
    }
    const int blk = p.block_table[(int64_t)t.req * p.max_blocks + bi];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
      atomicOr(p.status, KVTC_FLAG_BLOCK);
      return nullptr;
    }
    return t.cache +
           ((int64_t)blk * p.block_size + tok % p.block_size) * D * 2;
  } else {
    return t.dst + (int64_t)row * t.ld_bytes;
  }
}

template <class P>
__global__ void __launch_bounds__(kDecThreads, 1)
    decompress_kernel(const __grid_constant__ P p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sB = smem;
  uint8_t* sStg = smem + kDecOffStg;
  uint32_t* sRec = reinterpret_cast<uint32_t*>(smem + kDecOffRec);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kDecOffBar);
  uint64_t* full_b = bar;
  uint64_t* empty_b = bar + 4;
  uint64_t* a_full = bar + 8;
  uint64_t* a_empty = bar + 10;
  uint64_t* acc_full = bar + 12;
  uint64_t* acc_empty = bar + 14;
  uint64_t* mma_done = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kDecOffMisc);
  volatile int* abort_flag =
      reinterpret_cast<volatile int*>(smem + kDecOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(&full_b[i], 1);
      mbar_init(&empty_b[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kDecTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = p.total_tiles;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it_b = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const DecTile t = resolve(p, item);
        const DevStream* ds = p.streams + t.cs;
        const int nc = ds->nc, nch = ds->D / nc;
        const int nkb = (ds->k + kAtomK - 1) / kAtomK;
        const uint32_t bytes = (uint32_t)nc * 128u;
        if (item == (int)blockIdx.x) prefetch_tmap(&ds->tm_vdec);
        for (int ch = 0; ch < nch && ok; ++ch) {
          for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t s = it_b % kDecStages;
            const uint32_t ph = (it_b / kDecStages) & 1u;
            if (!mbar_wait(&empty_b[s], ph ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_b[s], bytes);
            tma_load_2d(sB + s * kDecBStage, &ds->tm_vdec, kb * kAtomK,
                        ch * nc, &full_b[s]);
            ++it_b;
          }
        }
      }
      if (!ok) raise_abort(abort_flag, p.status);
      for (uint32_t s = 0; s < kDecStages; ++s) {
        if (it_b > s) {
          const uint32_t last = s + kDecStages * ((it_b - 1 - s) / kDecStages);
          mbar_drain(&full_b[s], (last / kDecStages) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it_b = 0, chunk = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const DecTile t = resolve(p, item);
        const DevStream* ds = p.streams + t.cs;
        const int nc = ds->nc, nch = ds->D / nc;
        const int nkb = (ds->k + kAtomK - 1) / kAtomK;
        const int ksteps = ds->k / kGroup;
        const uint32_t idesc = make_idesc(128, (uint32_t)nc, 0);
        const uint32_t abuf = it & 1u;
        if (!mbar_wait(&a_full[abuf], (it >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_col = tmem + 256u + abuf * 128u;
        for (int ch = 0; ch < nch && ok; ++ch) {
          const uint32_t accb = chunk & 1u;
          if (!mbar_wait(&acc_empty[accb], ((chunk >> 1) & 1u) ^ 1u,
                         abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + accb * 128u;
          for (int kb = 0; kb < nkb; ++kb) {
            const uint32_t s = it_b % kDecStages;
            if (!mbar_wait(&full_b[s], (it_b / kDecStages) & 1u,
                           abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t base = smem_u32(sB + s * kDecBStage);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const int step = kb * 4 + ks;
              if (step < ksteps)
                mma_ts(d, a_col + (uint32_t)step * 8u,
                       sw128_desc(base + ks * 32), idesc, step > 0);
            }
            tc_commit(&empty_b[s]);
            ++it_b;
          }
          if (!ok) break;
          tc_commit(&acc_full[accb]);
          ++chunk;
        }
        if (!ok) break;
        tc_commit(&a_empty[abuf]);
        ++it;
      }
      if (!ok) raise_abort(abort_flag, p.status);
      tc_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------ prologue: unpack + dequantise
    const int q = warp & 3;
    uint32_t* stg = sRec + (warp - 2) * (kRecWords * 33);
    uint32_t it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const DecTile t = resolve(p, item);
      const DevStream* ds = p.streams + t.cs;
      const int R = ds->R, Ga = ds->Ga;
      const uint32_t abuf = it & 1u;
      if (!mbar_wait(&a_empty[abuf], ((it >> 1) & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int row0 = t.tile * kTileM + q * 32;
      const int nvalid = min(max(t.tc - row0, 0), 32);
      const uint8_t* rbase = t.rec + (int64_t)row0 * R;
      // Coalesced 16-byte loads of the warp's 32 records, stored
      // word-transposed ([word][token], row pitch 33) in shared memory.
      for (int o = lane * 16; o < 32 * R; o += 512) {
        const int tr = o / R;
        const int wd = (o - tr * R) >> 2;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (tr < nvalid) v = ld_nc_v4(rbase + o);
        stg[(wd + 0) * 33 + tr] = v.x;
        stg[(wd + 1) * 33 + tr] = v.y;
        stg[(wd + 2) * 33 + tr] = v.z;
        stg[(wd + 3) * 33 + tr] = v.w;
      }
      __syncwarp();
      const uint32_t a_tmem =
          tmem + ((uint32_t)(q * 32) << 16) + 256u + abuf * 128u;
      for (int a = 0; a < Ga; ++a) {
        const int b = ds->bits[a];
        const int po = ds->poff[a];
        const uint32_t f = stg[a * 33 + lane];
        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
        for (int j = 0; j < b; ++j) {
          const int bo = po + 2 * j;
          const uint32_t word = stg[(bo >> 2) * 33 + lane];
          const uint32_t pl = (bo & 2) ? (word >> 16) : (word & 0xFFFFu);
          w0 |= spread4(pl & 0xFu) << j;
          w1 |= spread4((pl >> 4) & 0xFu) << j;
          w2 |= spread4((pl >> 8) & 0xFu) << j;
          w3 |= spread4((pl >> 12) & 0xFu) << j;
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
        tmem_st8(a_tmem + (uint32_t)a * 8u, out);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[abuf]);
      ++it;
    }
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  } else {
    // ------------------------------- epilogue: + mu, bf16, bulk stores
    const int q = warp & 3;
    uint8_t* stg_base = sStg + (warp - 6) * 2 * kDecStgWarp;
    uint32_t chunk = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
      const DecTile t = resolve(p, item);
      const DevStream* ds = p.streams + t.cs;
      const int D = ds->D, nc = ds->nc, nch = D / nc;
      const int row = t.tile * kTileM + q * 32 + lane;
      const bool valid = row < t.tc;
      char* rowp = valid ? dec_row_ptr(p, t, row, D) : nullptr;
      const float* mu = ds->mu;
      for (int ch = 0; ch < nch; ++ch) {
        const uint32_t accb = chunk & 1u;
        if (!mbar_wait(&acc_full[accb], (chunk >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint8_t* stg = stg_base + (chunk & 1u) * kDecStgWarp + lane * kDecStgRow;
        const uint32_t stg_addr = smem_u32(stg);
        bulk_wait_read<1>();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + accb * 128u;
        const int npc = nc / 32;
        for (int pc = 0; pc < npc; ++pc) {
          float v[32];
          tmem_ld32(taddr + (uint32_t)pc * 32u, v);
          tmem_wait_ld();
          if (pc == npc - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[accb]);
          }
          const float4* m4 =
              reinterpret_cast<const float4*>(mu + ch * nc + pc * 32);
          uint32_t o[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 mm = __ldg(m4 + i);
            o[2 * i] = pack_bf16(v[4 * i] + mm.x, v[4 * i + 1] + mm.y);
            o[2 * i + 1] = pack_bf16(v[4 * i + 2] + mm.z, v[4 * i + 3] + mm.w);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
            sts_v4(stg_addr + pc * 64 + i * 16, o[4 * i], o[4 * i + 1],
                   o[4 * i + 2], o[4 * i + 3]);
        }
        fence_proxy_async_smem();
        if (rowp) bulk_s2g(rowp + (int64_t)ch * nc * 2, stg, (uint32_t)nc * 2u);
        bulk_commit();
        ++chunk;
      }
    }
    bulk_wait<0>();
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kDecTmemCols);
  }
}

// ======================================================================
//                                compress
// ======================================================================
constexpr int kCompWarps = 6;  // 0 TMA, 1 MMA, 2-5 epilogue
constexpr int kCompThreads = kCompWarps * 32;
constexpr int kCompMaxStages = 6;
constexpr int kCompAStage = kTileM * 128;          // [128 rows][64 bf16]
constexpr uint32_t kCompTmemCols = 512;            // accumulators at 0, 256

int compress_smem_bytes(int nstages, int stage_bytes, int rec_stg_words) {
  return nstages * stage_bytes + 4 * rec_stg_words * 33 * 4 + 256 + 64 + 1024;
}

__device__ __forceinline__ int find_comp_seg(const CompParams& p, int item) {
  int lo = 0, hi = p.nseg - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (p.seg[mid].tile_begin <= item) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kCompThreads, 1)
    compress_kernel(const __grid_constant__ CompParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int nst = p.nstages;
  const int stage_bytes = p.stage_bytes;
  uint32_t* sRec = reinterpret_cast<uint32_t*>(smem + nst * stage_bytes);
  const int rec_words = p.rec_stg_words;
  uint64_t* bar =
      reinterpret_cast<uint64_t*>(smem + nst * stage_bytes + 4 * rec_words * 33 * 4);
  uint64_t* full = bar;
  uint64_t* empty = bar + kCompMaxStages;
  uint64_t* acc_full = bar + 2 * kCompMaxStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* mma_done = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 32);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bar + 33);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCompTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = p.total_tiles;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it_b = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const CompSeg& g = p.seg[find_comp_seg(p, item)];
        const int tile = item - g.tile_begin;
        const DevStream* ds = p.streams + g.cs;
        const int nkb = ds->D / kAtomK;
        const uint32_t bytes = (uint32_t)kCompAStage + (uint32_t)ds->k * 128u;
        for (int kb = 0; kb < nkb; ++kb) {
          const uint32_t s = it_b % nst;
          if (!mbar_wait(&empty[s], ((it_b / nst) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + s * stage_bytes;
          mbar_arrive_expect_tx(&full[s], bytes);
          tma_load_2d(st, &g.tm_x, kb * kAtomK, g.row0 + tile * kTileM,
                      &full[s]);
          tma_load_2d(st + kCompAStage, &ds->tm_venc, kb * kAtomK, 0, &full[s]);
          ++it_b;
        }
      }
      if (!ok) raise_abort(abort_flag, p.status);
      for (uint32_t s = 0; s < (uint32_t)nst; ++s) {
        if (it_b > s) {
          const uint32_t last = s + nst * ((it_b - 1 - s) / nst);
          mbar_drain(&full[s], (last / nst) & 1u);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it_b = 0, it = 0;
      bool ok = true;
      for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
        const CompSeg& g = p.seg[find_comp_seg(p, item)];
        const DevStream* ds = p.streams + g.cs;
        const int nkb = ds->D / kAtomK;
        const uint32_t idesc = make_idesc(128, (uint32_t)ds->k, 1);
        const uint32_t accb = it & 1u;
        if (!mbar_wait(&acc_empty[accb], ((it >> 1) & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + accb * 256u;
        for (int kb = 0; kb < nkb; ++kb) {
          const uint32_t s = it_b % nst;
          if (!mbar_wait(&full[s], (it_b / nst) & 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = smem_u32(smem + s * stage_bytes);
          const uint32_t b = a + kCompAStage;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_ss(d, sw128_desc(a + ks * 32), sw128_desc(b + ks * 32), idesc,
                   (kb | ks) != 0);
          tc_commit(&empty[s]);
          ++it_b;
        }
        if (!ok) break;
        tc_commit(&acc_full[accb]);
        ++it;
      }
      if (!ok) raise_abort(abort_flag, p.status);
      tc_commit(mma_done);
      mbar_drain(mma_done, 0);
    }
    __syncwarp();
  } else {
    // ------------------------- epilogue: quantise + bit-plane records
    const int q = warp & 3;
    uint32_t* stg = sRec + (warp - 2) * (rec_words * 33);
    const uint32_t stg_addr = smem_u32(stg);
    uint32_t it = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const CompSeg& g = p.seg[find_comp_seg(p, item)];
      const int tile = item - g.tile_begin;
      const DevStream* ds = p.streams + g.cs;
      const int R = ds->R, Ga = ds->Ga;
      const uint32_t accb = it & 1u;
      if (!mbar_wait(&acc_full[accb], (it >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int row0 = tile * kTileM + q * 32;
      const int nvalid = min(max(g.tc - row0, 0), 32);
      for (int w = 0; w < (R >> 2); ++w) stg[w * 33 + lane] = 0u;
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + accb * 256u;
      bool range_err = false;
      for (int a = 0; a < Ga; ++a) {
        float v[16];
        tmem_ld16(taddr + (uint32_t)a * 16u, v);
        tmem_wait_ld();
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
        const __half sc = __float2half_ru(__fdiv_ru(__fsub_ru(hi, shf), lev));
        const float scf = __half2float(sc);
        range_err |= __hisinf(sh) != 0 || __hisinf(sc) != 0 ||
                     __hisnan(sh) || __hisnan(sc);
        const float inv = scf > 0.f ? __frcp_rn(scf) : 0.f;
        uint32_t code[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float u = fmaf(v[i] - shf, inv, 0.5f);
          u = fminf(fmaxf(u, 0.f), lev);
          code[i] = __float_as_uint(__fadd_rd(u, 8388608.f)) & 0xFFu;
        }
        uint32_t w[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          w[kk] = code[4 * kk] | (code[4 * kk + 1] << 8) |
                  (code[4 * kk + 2] << 16) | (code[4 * kk + 3] << 24);
        stg[a * 33 + lane] = (uint32_t)__half_as_ushort(sh) |
                             ((uint32_t)__half_as_ushort(sc) << 16);
        for (int j = 0; j < b; ++j) {
          uint32_t plane = 0;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            plane |= gather4((w[kk] >> j) & 0x01010101u) << (4 * kk);
          const int bo = po + 2 * j;
          sts_u16(stg_addr + (uint32_t)(((bo >> 2) * 33 + lane) * 4 + (bo & 2)),
                  plane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[accb]);
      if (range_err && lane < nvalid) atomicOr(p.status, KVTC_FLAG_RANGE);
      uint8_t* rbase = g.rec + (int64_t)row0 * R;
      for (int o = lane * 16; o < 32 * R; o += 512) {
        const int tr = o / R;
        const int wd = (o - tr * R) >> 2;
        if (tr < nvalid)
          st_v4(rbase + o, stg[wd * 33 + tr], stg[(wd + 1) * 33 + tr],
                stg[(wd + 2) * 33 + tr], stg[(wd + 3) * 33 + tr]);
      }
      __syncwarp();
      ++it;
    }
    if (!ok && lane == 0) raise_abort(abort_flag, p.status);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCompTmemCols);
  }
}

// ======================================================================
//                                raw rows
// ======================================================================
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
    const uint4 v = ld_nc_v4(p.src[r] + (int64_t)j * p.sbytes[r] +
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
cudaError_t launch_compress(const CompParams& p, int grid, cudaStream_t st) {
  const int smem = compress_smem_bytes(p.nstages, p.stage_bytes, p.rec_stg_words);
  static int configured = 0;
  if (configured < smem) {
    cudaError_t e = cudaFuncSetAttribute(
        compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    configured = 232448;
  }
  compress_kernel<<<grid, kCompThreads, smem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

template <class P>
static cudaError_t launch_dec(const P& p, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(
        decompress_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
        kDecSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  decompress_kernel<P><<<grid, kDecThreads, kDecSmem, st>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_decompress(const DecParams& p, int grid, cudaStream_t st) {
  return launch_dec(p, grid, st);
}

cudaError_t launch_decompress_paged(const PagedParams& p, int grid,
                                    cudaStream_t st) {
  return launch_dec(p, grid, st);
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
