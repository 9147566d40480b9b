/*
 * kvtc.h -- C ABI of the GB300 (sm_103a) KV-cache transform codec.
 *
 * The method is KV-cache transform coding ("KV Cache Transform Coding for
 * Compact Storage in LLM Inference", technical summary section 2):
 *   compress    (2B)  c = V^T (x - mu), keep the principal components whose
 *                     group the DP allocation gave a nonzero width, quantise
 *                     each 16-component group with an fp16 shift and scale
 *                     of its own (microscaling, 2A), pack the codes;
 *   decompress  (2C)  unpack, dequantise, x_hat = V c_hat + mu, bf16;
 *   sinks/window (2A) the first s and the last w tokens are stored raw.
 * The DEFLATE stage the page runs after packing (2B) is not part of this
 * library; an optional lossless field-packing stage of its own is
 * (kvtc_fields_pack / kvtc_fields_unpack).
 *
 * Conventions for every entry point:
 *   - All device pointers are caller-owned CUDA device memory on the device
 *     the calibration was loaded on.  The library allocates device memory
 *     only in kvtc_calib_load (and frees it in kvtc_calib_free); the codec
 *     calls allocate nothing.
 *   - Work is enqueued on the caller's stream (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  KVTC_OK means "validated
 *     and enqueued", not "finished".
 *   - Arguments are validated on the host before any launch; on error
 *     nothing is enqueued and a negative status is returned.
 *   - Faults detected by the kernels (fp16 field overflow, a block id out
 *     of range, a bounded wait that ran out) never trap: the kernel skips
 *     the affected write and ORs a flag into a sticky per-calibration status
 *     word, read and cleared with kvtc_device_status.
 *   - Pointers that the kernels reach with 16-byte vector or bulk copies
 *     must be 16-byte aligned, and row strides (ld) multiples of 8 elements.
 *   - The calls are thread-safe on the host, and a launch's parameters
 *     travel with the launch (nothing is staged in library-owned memory).
 *     A loaded calibration is read-only on the device, so codec calls that
 *     use it may run at the same time on several streams; their kernel
 *     flags all land in its one status word.  The one exception is
 *     kvtc_calib_mean_static (below).
 *
 * Formats (all little-endian):
 *
 *   Token record (R = 16 * ceil(budget_bits / 128) bytes): for each active
 *   group g in ascending order a u16 fp16 shift then a u16 fp16 scale; then
 *   for each active group in ascending order its b_g bit-planes, one u16
 *   each, bit i of plane j = bit j of the code of the group's i-th
 *   component; zero padding to R.  Code q of coefficient c:
 *     shift = fp16 round-down of the group minimum,
 *     scale = fp16 round-up of (max - shift) / (2^b - 1),
 *     q = clamp(floor((c - shift) / scale + 1/2), 0, 2^b - 1)  (0 if scale 0),
 *     c_hat = shift + q * scale.
 *
 *   Stream of one (request, layer, K|V) with T tokens, s' = min(s, T),
 *   w' = min(w, T - s'), T_c = T - s' - w':  s' sink rows (bf16 [s'][D]),
 *   w' window rows (bf16 [w'][D]), T_c records in token order; the stream
 *   is padded to a multiple of 256 bytes.  Several streams are concatenated
 *   in (layer, K, V) order.
 *
 *   Calibration blob, version 1: "KVTC", u32 version, n_streams, group (16),
 *   bmax (8), sink, window, budget_bits; per stream u32 layer, kv (0 = K,
 *   1 = V), D, k, u8 widths[D/16] zero-padded to a multiple of 8 bytes, f64
 *   mu[D], f64 V_kept[k][D] (row a = a-th kept principal vector, ascending
 *   component order), f64 eigenvalues[D]; trailer u32 CRC-32 (IEEE 802.3) of
 *   all preceding bytes, u32 0.
 */
#ifndef KVTC_H
#define KVTC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum kvtc_status {
  KVTC_OK = 0,
  KVTC_EINVAL = -1,   /* null/invalid argument, layer or kv not in blob */
  KVTC_EFORMAT = -2,  /* blob magic/version/checksum/structure */
  KVTC_ESIZE = -3,    /* buffer too small, sizes inconsistent */
  KVTC_ENOMEM = -4,   /* device allocation in kvtc_calib_load failed */
  KVTC_ECUDA = -5,    /* a CUDA runtime/driver call failed */
  KVTC_ERANGE = -6,   /* device flag: fp16 field overflow in compress */
  KVTC_EDEVICE = -7,  /* device flag: bounded wait ran out / bad block id */
  KVTC_EALIGN = -8,   /* pointer or stride misaligned */
  KVTC_ENOTSUP = -9   /* shape outside what the kernels support */
};

/* Sticky device flags reported by kvtc_device_status (bit mask). */
#define KVTC_FLAG_RANGE 1u     /* a shift/scale left the fp16 range */
#define KVTC_FLAG_TIMEOUT 2u   /* a bounded mbarrier wait ran out */
#define KVTC_FLAG_BLOCK 4u     /* block-table id outside [0, num_blocks) */
#define KVTC_FLAG_FORMAT 8u    /* packed stream inconsistent (field packing) */

typedef struct kvtc_calib kvtc_calib;

/*
 * kvtc_calib_load -- parse a calibration blob and build the device operands.
 * Reading of technical summary 2A: mu, the basis V and the per-group widths
 * come from a one-time calibration and are shared by every request.
 *   blob, blob_bytes : host memory, read only during the call.
 *   cuda_device      : device ordinal that will run the codec.
 *   out              : receives an opaque handle (owned by the caller, free
 *                      with kvtc_calib_free).
 * Derived on load: bf16 V_kept (projection), fp16 V_kept (reconstruction),
 * fp32 mu and fp32 m = bf16(V_kept) mu, group layout tables, TMA
 * descriptors.  Requirements: D % 64 == 0, D <= 8192, 16 <= k <= 496 (the
 * reconstruction holds k plus one mean step of 16 fp16 columns in 256
 * tensor-memory columns) and record bytes <= 256; otherwise ENOTSUP.  Up
 * to k = 240 both kernels double-buffer their tensor-memory operands;
 * above, a launch that holds such a stream single-buffers them (the
 * projection above k = 256, the reconstruction's A operand above k = 240).
 * The projection's shared-memory ring holds two or more stages while
 * 2 (32768 + 128 k) + 264 R + 1344 <= 232448 bytes (k <= 382 at R = 256),
 * one stage beyond.
 * Errors: EINVAL, EFORMAT, ENOMEM, ECUDA, ENOTSUP.
 */
int kvtc_calib_load(const void* blob, size_t blob_bytes, int cuda_device,
                    kvtc_calib** out);
void kvtc_calib_free(kvtc_calib* calib);

/* Shape of stream (layer, kv): D, kept components k, sink s, window w,
 * record bytes R.  Any output pointer may be NULL.  EINVAL if absent. */
int kvtc_calib_query(const kvtc_calib* calib, int layer, int kv, int* D,
                     int* k, int* s, int* w, int* record_bytes);

/* Bytes of one stream of T tokens (multiple of 256); < 0 on error. */
int64_t kvtc_stream_bytes(const kvtc_calib* calib, int layer, int kv,
                          int64_t T);

/*
 * kvtc_compress -- technical summary 2B (and 2A for sinks/window).
 *   layer0, nlayers : layers [layer0, layer0 + nlayers).
 *   kv_mask         : 1 = K, 2 = V, 3 = both.
 *   src             : HOST array of 2*nlayers device pointers, entry
 *                     2*(l - layer0) + kv = bf16 [T][ld] rows of that stream
 *                     (entries of kinds not in kv_mask are ignored).
 *   ld              : row stride of src in elements (>= D, % 8 == 0).
 *   T               : tokens (>= 0).
 *   dst, dst_bytes  : device output; streams concatenated in (layer, K, V)
 *                     order, each kvtc_stream_bytes long.
 * Errors: EINVAL, ESIZE, EALIGN, ECUDA, ENOTSUP.
 */
int kvtc_compress(const kvtc_calib* calib, int layer0, int nlayers,
                  int kv_mask, const void* const* src, int64_t ld, int64_t T,
                  void* dst, int64_t dst_bytes, void* cuda_stream);

/*
 * kvtc_decompress -- technical summary 2C.
 *   src, src_bytes  : input written by kvtc_compress (same layers, kv_mask
 *                     and T), in device memory or in pinned host memory
 *                     (cudaHostAlloc / cudaHostRegister).  Pinned host
 *                     memory is read by the kernels themselves over the
 *                     host link (on GB300, NVLink-C2C), with no staging
 *                     copy.  Pageable host memory: EINVAL.
 *   dst             : HOST array of 2*nlayers device pointers (as src of
 *                     kvtc_compress), each bf16 [T][ld].
 *   layer_events    : NULL, or a HOST array of nlayers cudaEvent_t (as
 *                     void*).  When given, layers are restored one launch
 *                     per layer in order and event l is recorded once layer
 *                     layer0 + l is complete, so a consumer can start on
 *                     early layers (layer-wise decompression, 2C).
 * Errors: EINVAL, ESIZE, EALIGN, ECUDA, ENOTSUP.
 */
int kvtc_decompress(const kvtc_calib* calib, int layer0, int nlayers,
                    int kv_mask, const void* src, int64_t src_bytes,
                    int64_t T, void* const* dst, int64_t ld,
                    void* cuda_stream, void* const* layer_events);

/*
 * kvtc_decompress_paged -- restore R requests into a paged KV pool (the
 * block-paged prefix cache of technical summary section 1).
 *   src          : HOST array [R] of pointers; src[r] holds request r's
 *                  streams as kvtc_compress wrote them, in device memory or
 *                  pinned host memory (as for kvtc_decompress).
 *   T            : HOST array [R] of token counts.
 *   block_table  : DEVICE int32 [R][max_blocks]; token t of request r goes
 *                  to block block_table[r*max_blocks + t/block_size], row
 *                  t % block_size.  Ids outside [0, num_blocks) are skipped
 *                  and flag KVTC_FLAG_BLOCK.
 *   block_size   : tokens per block; 16 (other sizes return ENOTSUP).
 *   max_blocks   : columns of block_table; every request needs
 *                  ceil(T[r] / block_size) of them (ESIZE otherwise).
 *   cache        : HOST array of 2*nlayers device pointers, each bf16
 *                  [num_blocks][block_size][D] (entries of kinds not in
 *                  kv_mask ignored).
 * All selected streams must share one D.  R <= 4096 (split larger sets).
 * Errors: EINVAL, ESIZE, EALIGN, ECUDA, ENOTSUP.
 */
int kvtc_decompress_paged(const kvtc_calib* calib, int layer0, int nlayers,
                          int kv_mask, const void* const* src,
                          const int64_t* T, int R, const int32_t* block_table,
                          int max_blocks, int block_size, void* const* cache,
                          int64_t num_blocks, void* cuda_stream);

/*
 * Field packing -- a lossless stage after bit-packing.  The page runs DEFLATE
 * there (technical summary 2B); this library runs a format of its own that
 * targets the one redundant part of a record, the high byte of each fp16
 * field.  Per stream and field slot (slot 2a = shift of active group a,
 * 2a + 1 = its scale), v = high byte h >> 2 (sign and exponent) spans
 * [vmin, vmin + 2^dbits) over the stream's records (dbits <= 6), so h is
 * stored as h - 4 vmin in dbits + 2 bits; the other bits are kept, and the
 * record's zero padding is dropped.
 *
 *   Packed stream (little-endian): header "KVFP", u32 T_c, u16 Rp (packed
 *   record bytes), u16 nslot (= 2 G_a), u32 0; slot table nslot x (u8 vmin,
 *   u8 dbits) zero-padded so that header and table fill 128 bytes (a
 *   multiple of 128 above 56 slots); the s' + w' raw rows as in the codec
 *   stream; T_c packed records of Rp bytes; zeros to a 256-byte multiple.
 *   Packed record: the low bytes of the 2 G_a fields in slot order; the
 *   codes, per slot h - 4 vmin in dbits + 2 bits, least significant bit
 *   first, in 2 ceil(bits / 16) bytes; the bit-planes of the codec record
 *   unchanged; zeros to a multiple of 4 bytes.  Rp <= R, so a packed
 *   stream is never longer than the codec stream plus its 128-byte prefix.
 *   The records of a stream start on a 128-byte line and 32 of them fill
 *   whole lines, which the restore from packed input reads line by line.
 *   Streams are concatenated in (layer, K, V) order.
 */

/* Field packing holds one field slot per lane of a warp: every selected
 * stream must keep at most 15 groups (k <= 240), else the three calls below
 * return ENOTSUP. */

/* Upper bound on the packed bytes of the selected streams at T tokens
 * (< 0 on error). */
int64_t kvtc_fields_bound(const kvtc_calib* calib, int layer0, int nlayers,
                          int kv_mask, int64_t T);

/* Device workspace bytes kvtc_fields_pack needs (< 0 on error). */
int64_t kvtc_fields_workspace_bytes(const kvtc_calib* calib, int layer0,
                                    int nlayers, int kv_mask);

/*
 * kvtc_fields_pack -- pack codec streams.
 *   src, src_bytes   : device codec streams as kvtc_compress wrote them
 *                      (same layers, kv_mask and T).
 *   dst, dst_capacity: device output, at least kvtc_fields_bound bytes; the
 *                      packed streams are written back to back.
 *   offsets          : device int64 [n + 1] (n = selected streams), written:
 *                      packed stream i occupies [offsets[i], offsets[i+1])
 *                      of dst; offsets[n] is the packed size.
 *   workspace        : device scratch of kvtc_fields_workspace_bytes bytes,
 *                      used only while the call's work runs on cuda_stream.
 * Three kernel launches per 256 streams (a min/max pass, a layout pass that
 * writes headers, tables and offsets, and the pack pass); no host
 * synchronisation.  src, dst and workspace 16-byte aligned, offsets 8.
 * Errors: EINVAL, ESIZE, EALIGN, ENOMEM, ECUDA.
 */
int kvtc_fields_pack(const kvtc_calib* calib, int layer0, int nlayers,
                     int kv_mask, const void* src, int64_t src_bytes,
                     int64_t T, void* dst, int64_t dst_capacity,
                     int64_t* offsets, void* workspace,
                     int64_t workspace_bytes, void* cuda_stream);

/*
 * kvtc_fields_unpack -- restore the codec streams that kvtc_fields_pack
 * packed, byte for byte.
 *   src, src_bytes : device packed streams.
 *   offsets        : device int64 [n + 1] as kvtc_fields_pack wrote them.
 *   dst, dst_bytes : device output, the codec streams (kvtc_stream_bytes
 *                    each, concatenated as kvtc_compress writes them).
 * Each stream's header and table are checked against its calibration, T
 * and offsets on the GPU; a stream that does not match is skipped and flags
 * KVTC_FLAG_FORMAT.  One kernel launch per 256 streams.
 * Errors: EINVAL, ESIZE, EALIGN, ENOMEM, ECUDA.
 */
int kvtc_fields_unpack(const kvtc_calib* calib, int layer0, int nlayers,
                       int kv_mask, const void* src, int64_t src_bytes,
                       const int64_t* offsets, int64_t T, void* dst,
                       int64_t dst_bytes, void* cuda_stream);

/*
 * kvtc_decompress_packed -- the restore of kvtc_decompress (the mapping of
 * technical summary 2A inverted: dequantise, project back with V_kept^T, add
 * mu) read straight from the packed streams that kvtc_fields_pack wrote: the
 * restore kernel unpacks each record's fields as it loads it, so the packed
 * bytes are the only compressed bytes read and no codec stream is written.
 * The output is bit-identical to kvtc_fields_unpack followed by
 * kvtc_decompress.
 *   src, src_bytes : the packed streams, in device memory or pinned host
 *                    memory (read by the kernels over the host link, zero
 *                    copy); pageable host memory is refused (EINVAL).
 *   offsets        : int64 [n + 1] as kvtc_fields_pack wrote them (n =
 *                    selected streams), device or pinned host memory.
 *   T, dst, ld, cuda_stream, layer_events : as for kvtc_decompress.
 * Each stream's header, slot table and length are checked against its
 * calibration, T, the offsets and src_bytes on the GPU before anything they
 * frame is read; a stream that does not match restores its coded tokens as
 * from all-zero records and flags KVTC_FLAG_FORMAT.  Its raw rows are copied
 * whenever its extent frames them (both offsets on the 16-byte grid, inside
 * src_bytes), and, in a call with no coded token, only when its magic and
 * T_c check out too; an out-of-frame stream flags KVTC_FLAG_FORMAT.
 * Kernel launches as for kvtc_decompress (the raw rows of a call with no
 * coded token take one copy launch per 96 streams).  Streams must keep at
 * most 15 groups, else ENOTSUP.  src 16-byte aligned, offsets 8.
 * Errors: EINVAL, ESIZE, EALIGN, ENOTSUP, ENOMEM, ECUDA.
 */
int kvtc_decompress_packed(const kvtc_calib* calib, int layer0, int nlayers,
                           int kv_mask, const void* src, int64_t src_bytes,
                           const int64_t* offsets, int64_t T,
                           void* const* dst, int64_t ld, void* cuda_stream,
                           void* const* layer_events);

/*
 * kvtc_calibrate -- the one-time calibration of technical summary 2A, on
 * the GPU, writing a version-1 blob (format above).  Per stream: mu = mean of
 * the calibration rows; V = eigenvectors of their covariance, sorted by
 * eigenvalue descending, each signed so that its largest-magnitude entry is
 * positive; E[g][b] = summed squared coefficient error of group g at width
 * b (b = 0: the group's energy) measured with the codec's quantiser; widths
 * = the DP allocation minimising sum E[g][b_g] with sum (32 + 16 b_g) over
 * groups with b_g > 0 at most budget_bits (ties keep the smaller width).
 *   tokens      : HOST array [n] of device pointers, stream i's calibration
 *                 rows, bf16 [N][ld]; layers, kvs: HOST arrays [n].
 *   blob        : HOST output of capacity bytes (kvtc_blob_max_bytes is an
 *                 upper bound); *blob_bytes receives the size (also when
 *                 the capacity is too small: ESIZE).
 * Unlike the codec calls it allocates temporary device memory (freed before
 * returning) and synchronises cuda_stream.  fp64 arithmetic on the device:
 * mean, covariance, eigenvector order and signs, coefficient products,
 * distortion table and DP are this library's kernels; the symmetric
 * eigensolver is cuSOLVER's (syevd).
 * Errors: EINVAL, ENOMEM, ECUDA, ESIZE.
 */
int kvtc_calibrate(int cuda_device, int n, const int* layers, const int* kvs,
                   const void* const* tokens, int64_t N, int64_t ld, int D,
                   int sink, int window, int budget_bits, void* blob,
                   size_t capacity, size_t* blob_bytes, void* cuda_stream);

/* Upper bound on the blob size of n streams of width D (< 0 on error). */
int64_t kvtc_blob_max_bytes(int n, int D);

/* Synchronise cuda_stream, then return the sticky device flags in *flags
 * (KVTC_FLAG_*) and clear them.  Returns KVTC_OK or ECUDA. */
int kvtc_device_status(const kvtc_calib* calib, void* cuda_stream,
                       unsigned* flags);

/*
 * kvtc_wait_selftest -- exercise the bounded wait that every kernel of this
 * library uses on its mbarriers (the pages have no counterpart: this is a
 * failure-detection check).  One thread waits, for at most limit_us
 * microseconds, on a barrier that nothing ever arrives at; when the limit
 * runs out it sets KVTC_FLAG_TIMEOUT in the handle's sticky flag word, the
 * same way a kernel reports a wait that ran out, and returns.  Read the
 * flag with kvtc_device_status; the context stays usable.
 *   limit_us    : 1 .. 2000000.
 *   cuda_stream : the launch is enqueued on it.
 * Errors: EINVAL, ECUDA.
 */
int kvtc_wait_selftest(const kvtc_calib* calib, uint32_t limit_us,
                       void* cuda_stream);

/*
 * kvtc_calib_mean_static -- the per-channel mean of calibration rows (the
 * mean that kvtc_calibrate stores for a stream), computed without
 * allocating any device memory.  The paper has no counterpart: this entry
 * point exists for callers that cannot call cudaMalloc, such as serving
 * engines that give nearly all device memory to their own KV-cache pool at
 * start-up, or latency-sensitive paths that cannot take the device-wide
 * synchronisation of cudaMalloc / cudaFree.
 *   tokens : device bf16 rows [N][ld] (N >= 1, ld >= D).
 *   mu_out : device fp64 [D], written.
 *   D      : at most 4096; wider rows return KVTC_ESIZE.
 * Scratch comes from a fixed 1 MiB array inside the library.  CUDA loads
 * modules lazily by default, so the array comes into being on a device at
 * the first call there, which loads this code and looks up the array's
 * device address (a one-time set-up), and it is then held until the process
 * exits.  That first call can therefore fail with ECUDA when the device has
 * no free memory left: make it before reserving the device's memory for a
 * KV pool (or run with CUDA_MODULE_LOADING=EAGER, which creates the array
 * with the context), and before any stream capture.  All calls on a device
 * share the array: each call writes every entry it reads, but calls that
 * overlap on the GPU race with each other, so serialise them.  No
 * cudaMalloc, cudaFree or allocating library routine is called.  Enqueued
 * on cuda_stream.
 * Errors: EINVAL, ESIZE, ECUDA.
 */
int kvtc_calib_mean_static(int cuda_device, const void* tokens, int64_t N,
                           int64_t ld, int D, double* mu_out,
                           void* cuda_stream);

/* Number of kernels this library has launched since it was loaded (all
 * devices and threads); a cheap way for callers to count launches. */
uint64_t kvtc_launch_count(void);

/* Static description of a status code. */
const char* kvtc_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* KVTC_H */
