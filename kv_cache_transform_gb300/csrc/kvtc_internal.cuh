// Internal definitions shared by the host side and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace kvtc {

constexpr int kGroup = 16;         // components per microscaling group
constexpr int kTileM = 128;        // tokens per CTA tile (TMEM lanes)
constexpr int kPairM = 256;        // tokens per CTA-pair super-tile (MMA M)
constexpr int kAtomK = 64;         // 16-bit elements per 128-byte swizzle row
constexpr int kMaxK = 496;         // kept components supported (TMEM: the
                                   // decompress A operand, k + 16 fp16
                                   // columns, in 256 TMEM columns)
constexpr int kNarrowK = 240;      // up to here both kernels double-buffer
                                   // (compress: k <= 256 accumulators of
                                   // 256 columns; decompress: A buffers of
                                   // 128 columns hold k + 16 <= 256)
constexpr int kMaxRecord = 256;    // record bytes supported by the kernels
constexpr int kMaxD = 8192;

// Device-resident description of one calibrated (layer, K|V) stream; built
// once by kvtc_calib_load and read by every kernel launch.
struct DevStream {
  CUtensorMap tm_vdec;      // fp16 [kb][D][64]: V_kept, then mu_hi, mu_lo,
                            // zeros (kp = k + 16 columns, padded to 64s),
                            // box {64, nc/2, kb}
  CUtensorMap tm_venc;      // bf16 V_kept, K-block major [D/64][k][64],
                            // box {64, k/2, 2}
  CUtensorMap tm_venc1;     // the same, box {64, k/2, 1} (one K block)
  const float* mu;          // [D]   fp32 mean
  const float* m;           // [k]   fp32 projection of the mean
  const uint8_t* bits;      // [Ga]  width of each active group
  const uint16_t* poff;     // [Ga]  byte offset of the group's first plane
  int32_t D, k, Ga, R;      // R = record bytes
  int32_t nc;               // reconstruction N chunk: 256, 128 or 64
  int32_t kp;               // reconstruction K: k + 16 (the mean step)
  int32_t kbs;              // reconstruction: K blocks per B ring stage
  int32_t nbs;              // reconstruction: B ring stages per chunk
};

// Raw rows (sink and window) copied by two warps of a tensor-core kernel
// while it runs: up to kRawListMax row segments; a segment whose src is
// null writes zeros (stream padding).
constexpr int kRawListMax = 192;
struct RawListSeg {
  const char* src;          // source row base, or null for zeros
  char* dst;                // destination row base
  int64_t src_ld, dst_ld;   // row strides in bytes
  int32_t rows;             // rows to copy
  int32_t row_bytes;        // bytes per row (multiple of 16)
  int64_t chunk_begin;      // first 16-byte chunk index of this segment
  int32_t pk;               // >= 0: the rows sit in packed stream pk, at
                            // pk_off bytes from its start (src unused)
  int32_t pk_tc;            // the T_c its header must hold
  int64_t pk_off;
};
struct RawList {
  RawListSeg seg[kRawListMax];
  int32_t nseg;
  int32_t pad;
  int64_t total_chunks;
  // packed input (kvtc_decompress_packed): stream i spans
  // [pk_offs[i], pk_offs[i + 1]) of pk_base, pk_bytes in all
  const uint8_t* pk_base;
  const int64_t* pk_offs;
  int64_t pk_bytes;
};

// ---------------------------------------------------------------- compress
constexpr int kCompMaxSeg = 64;
struct CompSeg {
  CUtensorMap tm_x;         // bf16 rows [s'+T_c][D] of the source viewed as
                            // {64, rows, D/64}, box {64, 128, 2}
  uint8_t* rec;             // first record of the stream (device)
  int32_t tc;               // compressed tokens
  int32_t row0;             // s' (first compressed source row)
  int32_t cs;               // calibration stream index
  int32_t pad;
};
struct CompParams {
  CompSeg seg[kCompMaxSeg];
  const DevStream* streams;
  unsigned* status;
  int32_t nseg;
  int32_t total_tiles;
  int32_t tiles_per_seg;    // every stream of a call has the same T
  int32_t nstages;
  int32_t stage_bytes;      // A + B bytes of one stage (two K blocks)
  int32_t b_bytes_max;      // B bytes reserved per stage
  int32_t rec_stg_words;    // record staging words per thread
  int32_t wide;             // a stream keeps k > 256: one k-column
                            // accumulator, two MMAs (N = 256, k - 256) per
                            // K step
  int32_t kps;              // K blocks per ring stage: 2, or 1 where two
                            // stages of two do not fit
  RawList raw;              // sink/window rows and padding of these streams
};

// -------------------------------------------------------------- decompress
constexpr int kDecMaxSeg = 96;
struct DecSeg {
  const uint8_t* rec;       // first record
  char* dst;                // output row of the first compressed token
  int64_t ld_bytes;         // output row stride
  int32_t tc;
  int32_t cs;
};
struct DecParams {
  CUtensorMap tm_out[kDecMaxSeg];  // bf16 [T_c rows][D] from dst, box {64,32}
  DecSeg seg[kDecMaxSeg];
  const DevStream* streams;
  unsigned* status;
  int32_t nseg;
  int32_t total_tiles;
  int32_t tiles_per_seg;    // every stream of a call has the same T
  int32_t nstages;          // B ring depth (shared-memory stages)
  int32_t rec_words;        // record staging words per thread (max R / 4)
  int32_t wide;             // a stream has k + 16 > 256: one A buffer
  int32_t packed;           // records come from packed streams (below)
  int32_t pk_first;         // packed stream index of segment 0
  int32_t pk_raw_rows;      // s' + w' (every stream of a call has one T)
  RawList raw;              // sink/window rows of these streams; for packed
                            // input also pk_base, pk_offs and pk_bytes
};
// every stream's sink, window and padding segments fit one launch's list
static_assert(3 * kCompMaxSeg <= kRawListMax, "raw list too short");
static_assert(2 * kDecMaxSeg <= kRawListMax, "raw list too short");

// Paged restore: work items are (stream, request, tile), stream-major, so
// that the CTA pairs running side by side share one stream's basis.  A
// request's tiles cover its tokens from token 0 (not from the first coded
// token), so that each epilogue warp's 32 rows are two whole 16-token
// blocks; rows without a record (sink, window, past the coded range) are
// decoded as zeros and never stored.
constexpr int kPagedMaxReq = 256;
constexpr int kPagedMaxStream = 64;      // streams per launch
// Super-tiles of one (request, stream): its tokens from 0 to the last one
// with a record, 256 at a time (none when no token is coded).
__host__ __device__ __forceinline__ int paged_tiles(int s_, int tc) {
  return tc > 0 ? (s_ + tc + kPairM - 1) / kPairM : 0;
}
struct PagedParams {
  CUtensorMap tm_cache[kPagedMaxStream]; // pool of stream j as {D, 16,
                                         // num_blocks}, box {64, 16, 1}
  const uint8_t* src[kPagedMaxReq];      // request's concatenated streams
  int64_t sbytes[kPagedMaxReq];          // bytes of one stream of request r
  int32_t tc[kPagedMaxReq];              // compressed tokens of request r
  int32_t s_[kPagedMaxReq];              // sink rows kept of request r
  int32_t raw_rows[kPagedMaxReq];        // s' + w' of request r
  int32_t tile_begin[kPagedMaxReq + 1];  // request r's first tile in a stream
  int64_t raw_begin[kPagedMaxReq + 1];   // first raw 16-byte chunk of request r
  int32_t req_index[kPagedMaxReq];       // absolute request id (block table row)
  char* cache[kPagedMaxStream];          // pool of stream j
  int32_t cs[kPagedMaxStream];           // calibration stream of stream j
  int32_t sidx[kPagedMaxStream];         // stream j's place in a request's
                                         // concatenated streams
  const DevStream* streams;
  unsigned* status;
  const int32_t* block_table;
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t block_size;
  int32_t nreq;
  int32_t nstream;
  int32_t total_tiles;
  int32_t D;
  int64_t total_raw_chunks;
  int32_t nstages;          // B ring depth (shared-memory stages)
  int32_t rec_words;        // record staging words per thread (max R / 4)
  int32_t wide;             // a stream has k + 16 > 256: one A buffer
};

// ---------------------------------------------------------------- raw rows
constexpr int kRawMaxSeg = 256;
struct RawSeg {
  const char* src;          // source row base
  char* dst;                // destination row base
  int64_t src_ld, dst_ld;   // row strides in bytes
  int32_t rows;             // rows to copy
  int32_t row_bytes;        // bytes per row (multiple of 16)
  int64_t chunk_begin;      // first 16-byte chunk index of this segment
};
struct RawParams {
  RawSeg seg[kRawMaxSeg];
  int32_t nseg;
  int64_t total_chunks;
};

// ----------------------------------------------------------- field packing
// Lossless packing of codec streams (kvtc_fieldpack.cu).  Work of one launch
// group: up to kFpMaxStream streams; items are per stream its raw-row
// chunks then its record tiles.
constexpr int kFpMaxStream = 256;
constexpr int kFpChunks = 8;          // min/max partial results per stream
constexpr int kFpWorkWords = 32;      // u32 words per (stream, chunk)
constexpr int kFpRawChunk = 32768;    // raw-row bytes per copy item; a
                                      // record tile is at most this long
constexpr int kFpHeader = 16;         // packed stream header bytes
constexpr uint32_t kFpMagic = 0x5046564Bu;  // "KVFP", little-endian
// Bytes of a packed stream's header and slot table: a multiple of 128, so
// that its records start on a 128-byte line of the stream.
__host__ __device__ __forceinline__ int fp_prefix_bytes(int ga) {
  return (kFpHeader + 4 * ga + 127) & ~127;
}
// Packed record bytes: 2 G_a low bytes, 2 hb2 code bytes, the bit-planes
// (used - 4 G_a bytes), zero-padded to a multiple of 4.
__host__ __device__ __forceinline__ int fp_record_bytes(int ga, int hb2,
                                                        int used) {
  return (2 * hb2 + used - 2 * ga + 3) & ~3;
}
struct FpStream {
  int64_t in_off;       // pack: codec stream offset in the input
  int64_t out_off;      // unpack: codec stream offset in the output
  int64_t raw_bytes;    // (s' + w') * D * 2
  int32_t tc;           // compressed tokens
  int32_t item_begin;   // first work item of this stream
  int32_t ntiles;       // ceil(tc / tile)
  int32_t nraw;         // ceil(raw_bytes / kFpRawChunk)
  int16_t ga;           // active groups
  int16_t used;         // used bytes of a codec record
  int16_t R;            // codec record bytes
  int16_t tile;         // tokens per record tile: (kFpRawChunk / R) & ~15
};
struct FpParams {
  FpStream s[kFpMaxStream];
  const uint8_t* in;
  uint8_t* out;
  int64_t* offsets;     // packed stream offsets [all streams + 1]
  uint32_t* work;       // pack: min/max partials [n][kFpChunks][32]
  unsigned* status;
  int64_t in_bytes;     // unpack: bytes of the packed input
  int32_t n;            // streams of this launch group
  int32_t first;        // index of its first stream in offsets
  int32_t total_items;
  int32_t pad;
};

// Launchers (kvtc_kernels.cu).  Return a cudaError_t.
// `pairs`: CTA pairs to launch (each kernel runs as clusters of two).
cudaError_t launch_compress(const CompParams& p, int pairs, cudaStream_t st);
cudaError_t launch_decompress(const DecParams& p, int pairs, cudaStream_t st);
cudaError_t launch_decompress_paged(const PagedParams& p, int pairs,
                                    cudaStream_t st);
// CTA pairs of each kernel that can be resident at once on this device.
int max_pairs_compress(int smem_bytes);
int max_pairs_decompress(int smem_bytes);
cudaError_t launch_raw_copy(const RawParams& p, cudaStream_t st);
cudaError_t launch_wait_selftest(unsigned* status, uint64_t limit_ns,
                                 cudaStream_t st);
cudaError_t launch_paged_raw(const PagedParams& p, cudaStream_t st);
// Raw rows of packed streams with no coded token (a RawList on its own).
cudaError_t launch_raw_list(const RawList& r, unsigned* status,
                            cudaStream_t st);
// Field packing (kvtc_fieldpack.cu): the three pack launches, and unpack.
cudaError_t launch_fields_pack(const FpParams& p, cudaStream_t st);
cudaError_t launch_fields_unpack(const FpParams& p, cudaStream_t st);
// Kernel launches issued by this library (all devices, all threads).
void count_launch();
// CRC-32 of IEEE 802.3 (as zlib): reflected 0xEDB88320, init/final ~0.
uint32_t crc32_ieee(const uint8_t* p, size_t n);
int compress_smem_bytes(int nstages, int stage_bytes, int rec_stg_words);
// Decompress shared memory for a ring of `nstages` and records of up to
// 4 * rec_words bytes; decompress_stages picks the deepest ring that fits.
int decompress_smem_bytes(int nstages, int rec_words);
int decompress_stages(int rec_words);

}  // namespace kvtc
