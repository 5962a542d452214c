/*
 * nwc.h -- C ABI of the GB300 (sm_103a) library for batch-1 (and small-batch) matrix-vector
 * products over losslessly entropy-coded BF16 (and fp8 e4m3) weight matrices.
 *
 * What the calls compute is defined by two pages:
 *   "NWC -- Neural Weight Compression" (PyPI project page, v0.9.0), section "How it works":
 *     a BF16 weight splits into a raw part and an entropy-coded exponent; the exponent is ranked
 *     by frequency and written as a unary rank code plus a raw sign bit, with an escape for rare
 *     values; a peek into a shared-memory table yields up to two complete codes; lanes decode
 *     their own bit streams over blocks of 8 rows x 512 columns inside the matrix-vector kernel;
 *     dequantization and the embedding lookup run on the same decoder; any shape works (fillers
 *     cost a short code and no mantissa).
 *     In this format (version 4) the sign sits beside the 7 raw mantissa bits (a byte per
 *     element), the coded stream holds only the unary rank codes, written by row pairs so that
 *     one 13-bit peek always holds a pair (a pair longer than that keeps its first code and a
 *     tail of ones, and its second element is listed), and an escape code is n_ranked ones whose
 *     raw exponent sits in the block's escape list.
 *   "Qwen3-4B-NWC-fp8" (model card): weight-only e4m3 with a symmetric per-output-channel
 *     scale, fp8 bytes coded losslessly, the scale applied at the end of the matvec.
 *
 * Conventions
 *   - Every call returns nwc_status; no exception or abort crosses this boundary.
 *   - Host pointers are read (or written) only during the call. Device pointers stay owned
 *     by the caller; the library allocates no device or pinned memory, ever.
 *   - GPU calls are asynchronous on the given stream (NULL = the legacy default stream).
 *     A launch failure returns NWC_ERR_CUDA. Data errors found on the device (a lane
 *     stream that runs past its words, an escape list that does not match the stream's
 *     escape codes, a gather id out of range) do not fault: every read stays inside the
 *     block's staged region (or the lane's own words), the outputs of a malformed block are
 *     unspecified (a bad gather id writes a zero row), and the kernel raises the device
 *     error word, which nwc_check() reads and clears.
 *   - Matrices are row-major: element (n, k) of an N x K matrix is at index n*ld + k.
 *     N = output features (rows), K = input features (columns), ld >= K.
 *   - BF16 values are passed as their 16-bit patterns (uint16_t); x is BF16, y is FP32.
 *   - Any call may come from any host thread. Calls that share a workspace (or the one
 *     scratch array of nwc_gemv_noalloc) must not overlap on the GPU; order them on one
 *     stream or with events. The device error word is per device, shared by all streams.
 *   - Every device the process uses gets its own kernel configuration on its first call
 *     there (made with that device current).
 */
#ifndef NWC_H
#define NWC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without the CUDA headers; pass a cudaStream_t (or torch's raw stream). */
typedef struct CUstream_st *nwc_stream;

typedef enum nwc_status {
    NWC_OK = 0,
    NWC_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad enum, misaligned buffer      */
    NWC_ERR_FORMAT = 2,      /* blob fails validation (header, tables, region sizes)     */
    NWC_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed              */
    NWC_ERR_TIMEOUT = 4,     /* a bounded device wait ran out (reported by nwc_check)    */
    NWC_ERR_DEVICE_FLAG = 5, /* a kernel raised the device error word (see nwc_check)    */
    NWC_ERR_UNSUPPORTED = 6, /* valid request this build does not implement              */
    NWC_ERR_IO = 7           /* a blob file could not be opened, read or written         */
} nwc_status;

enum { NWC_ELEM_BF16 = 0, NWC_ELEM_FP8_E4M3 = 1 };

/* Geometry of the format (fixed by the pages: blocks of 8 rows x 512 columns, 32 lanes of
 * 16 columns x 8 rows). */
enum { NWC_BLOCK_ROWS = 8, NWC_BLOCK_COLS = 512, NWC_LANES = 32, NWC_MAX_RANKED = 12 };

/* Entries and bytes of a matrix's decode table (see nwc_decode_table). */
enum { NWC_TABLE_ENTRIES = 8192, NWC_TABLE_BYTES = 32768 };

/*
 * A bound, validated matrix: plain data, safe to copy by value. Built by nwc_bind from the
 * blob's host copy (parsed once) and the address of its device copy. All pointers are device
 * pointers into that device copy; the caller keeps it alive while the struct is used.
 */
typedef struct nwc_matrix {
    int32_t elem;            /* NWC_ELEM_BF16 or NWC_ELEM_FP8_E4M3                          */
    int32_t n_ranked;        /* exponents with a unary code (1..12)                         */
    int64_t n, k;            /* rows (output features), columns (input features)           */
    int64_t row_blocks;      /* ceil(n / 8)                                                 */
    int64_t col_blocks;      /* ceil(k / 512)                                               */
    uint8_t rank_exp[16];    /* exponent value of rank 0..n_ranked-1                        */
    const uint32_t *block_tab; /* u32[row_blocks*col_blocks + 1], 16-byte units from data  */
    const uint8_t *data;     /* start of the block regions                                  */
    const float *scales;     /* fp32[n] per-row scales (fp8), NULL for BF16                 */
    uint64_t blob_bytes;     /* size of the whole blob                                      */
    uint64_t max_block_bytes;/* largest block region                                        */
    uint64_t data_bytes;     /* bytes of all block regions                                  */
    const uint32_t *table;   /* device copy of the decode table (nwc_decode_table), or NULL:   */
                             /* set by the caller after nwc_bind; NULL makes every kernel      */
                             /* build the table in shared memory itself (slower prologue)      */
} nwc_matrix;

/* Human-readable name of a status code (static string). */
const char *nwc_status_str(nwc_status s);

/* Library version string, e.g. "nwc 4 (format 4, sm_103a)". */
const char *nwc_version(void);

/*
 * nwc_encode -- host encoder ("How it works": byte planes, prefix code, per-lane bit streams).
 *   w       host, N x K BF16 bit patterns, row stride ld (elements).
 *   elem    NWC_ELEM_BF16 codes w as is. NWC_ELEM_FP8_E4M3 first quantizes each row n to
 *           e4m3 with scale s_n = absmax_n / 448 (FP32, s_n = 1 for an all-zero row), q =
 *           nearest e4m3 to fp32(w)/s_n (ties to even, saturating), then codes the bytes
 *           ("Qwen3-4B-NWC-fp8": symmetric per-output-channel scale). Non-finite weights
 *           are rejected for fp8 (NWC_ERR_INVALID_ARG).
 *   threads host worker threads (<= 0: all hardware threads). Output bytes do not depend on it.
 *   blob    host output buffer or NULL. Two-call pattern: with blob == NULL only *blob_bytes
 *           is set (the exact size); otherwise *blob_bytes holds the capacity on entry and
 *           the written size on return (NWC_ERR_INVALID_ARG if too small).
 */
nwc_status nwc_encode(const uint16_t *w, int64_t n, int64_t k, int64_t ld, int elem, int threads,
                      void *blob, size_t *blob_bytes);

/*
 * nwc_encode_fp8 -- codes already-quantized e4m3 bytes q (N x K, stride ld) with their row
 * scales (fp32[N], stored as given). Same two-call pattern and threads as nwc_encode.
 */
nwc_status nwc_encode_fp8(const uint8_t *q, const float *scales, int64_t n, int64_t k, int64_t ld,
                          int threads, void *blob, size_t *blob_bytes);

/*
 * nwc_quantize_fp8 -- the quantization step of nwc_encode(elem = FP8) alone, on the host:
 * q (N x K, stride ldq) and scales (fp32[N]) as defined there.
 */
nwc_status nwc_quantize_fp8(const uint16_t *w, int64_t n, int64_t k, int64_t ld, uint8_t *q,
                            int64_t ldq, float *scales);

/*
 * nwc_validate -- host check of a blob: header, rank table, block table, every block
 * region's size against its lane word counts (at most 26 each) and its raw section, and every
 * escape list (entries name real elements, carry an exponent field of the element's width,
 * come in lane-then-t order, then at most three padding words). NWC_ERR_FORMAT if any check
 * fails. Stream contents are checked by the kernels while decoding.
 */
nwc_status nwc_validate(const void *blob_host, size_t bytes);

/*
 * nwc_bind -- validates the host copy of a blob (as nwc_validate) and fills *out with its
 * geometry and the device pointers of the same blob copied to blob_dev (16-byte aligned,
 * caller-owned). out->table is NULL. No device call is made.
 */
nwc_status nwc_bind(const void *blob_host, size_t bytes, const void *blob_dev, nwc_matrix *out);

/*
 * nwc_decode_table -- the matrix's decode table on the host (the NWC page, "How it works": a
 * shared-memory table indexed by the next bits of a lane's stream): NWC_TABLE_ENTRIES u32
 * entries into table_host, entry p for the 13-bit peek p (first stream bit = bit 12): the row
 * pair it holds, bits 0..4 its length in bits, bits 7..14 and 23..30 the two elements'
 * exponent fields in BF16 position (fp8: v + 120, 0 for 0; an escape or the tail of a cut pair:
 * 0), bits 16..17 how many of them the escape list holds. Copy it to device memory (16-byte
 * aligned, kept alive and unchanged while in use) and set m->table to that copy: every kernel
 * then loads it with one bulk copy instead of building it in shared memory. Host only.
 */
nwc_status nwc_decode_table(const nwc_matrix *m, uint32_t *table_host);

/*
 * nwc_decode -- dequantization to the stored elements, bit-exact (the NWC page, "How it
 * works": decoding is lossless): BF16 blobs write uint16 out[n*ld_out + k]; fp8 blobs write the e4m3 bytes
 * (uint8) to out and the row scales to scales_out (fp32[N], may be NULL). ld_out >= K.
 * Rows are written 16 columns at a time with the widest store of 16, 8 or 4 bytes to which both
 * out and the row stride in bytes (ld_out x element size) are aligned; any other out or ld_out
 * is written element by element (correct, slower).
 */
nwc_status nwc_decode(const nwc_matrix *m, void *out, int64_t ld_out, float *scales_out,
                      nwc_stream stream);

/*
 * nwc_dequantize_fp8 -- BF16 weights for prefill from fp8 rows (the "Qwen3-4B-NWC-fp8" model
 * card: prefill dequantizes the weights to BF16 and calls cuBLAS): out[n*ld_out + k] = the BF16
 * nearest (ties to even) to the FP32 product e4m3(q[n*ld_q + k]) * scales[n]; a NaN code (or
 * product) gives 0x7FC0. q and scales are what nwc_decode writes for an fp8 blob. Device
 * pointers, N x K, ld_q >= K, ld_out >= K; 8-byte loads and 16-byte stores when q, out and the
 * strides keep that alignment, else element by element. Asynchronous on the stream; N or K = 0
 * is a no-op.
 */
nwc_status nwc_dequantize_fp8(const uint8_t *q, int64_t ld_q, const float *scales, int64_t n, int64_t k,
                              uint16_t *out, int64_t ld_out, nwc_stream stream);

/*
 * nwc_gemv_workspace_bytes -- device scratch nwc_gemv needs for m (at least 16 bytes): FP32
 * partial-sum slots per (row, 512-column block) and one counter per 8-row block (both only when
 * K > 512).
 */
size_t nwc_gemv_workspace_bytes(const nwc_matrix *m);

/*
 * nwc_gemv_prepare -- readies a workspace for m: every partial-sum slot to the empty marker
 * (all bits set) and every counter to zero (asynchronously on the stream). Call once per
 * workspace before its first nwc_gemv; every nwc_gemv leaves the workspace in that state
 * again, so it serves repeated calls and CUDA-graph replays. ws is 16-byte aligned, ws_bytes >=
 * nwc_gemv_workspace_bytes(m). Calls sharing one workspace must not overlap on the GPU.
 */
nwc_status nwc_gemv_prepare(const nwc_matrix *m, void *ws, size_t ws_bytes, nwc_stream stream);

/*
 * nwc_gemv -- batch-1 y = W x with W decoded in registers (the NWC page, "How it works",
 * fused kernel): x is BF16[K] (16-byte
 * aligned), y is FP32[N], y_n = sum_k w[n,k] x[k] accumulated in FP32 (fp8: y_n = s_n * sum_k q x).
 * Finite inputs give |y_n - exact| <= 2^-10 * sum_k |w x| + 1e-6. ws/ws_bytes: a workspace
 * prepared by nwc_gemv_prepare for this matrix. Whatever the kernel (nwc_gemv_route), the
 * column blocks' sums are added in one fixed order, so results are bitwise repeatable and equal
 * to nwc_gemv_list's.
 */
nwc_status nwc_gemv(const nwc_matrix *m, const uint16_t *x, float *y, void *ws, size_t ws_bytes,
                    nwc_stream stream);

/* Kernels nwc_gemv launches (nwc_gemv_route). */
#define NWC_ROUTE_GEMV 0 /* one CTA per SM, blocks dealt round-robin; sums over column blocks
                            through the workspace (partial sums and a ticket)                 */
#define NWC_ROUTE_LIST 2 /* the nwc_gemv_list kernel with one item (a tall matrix with a
                            device decode table)                                              */

/*
 * nwc_gemv_route -- the kernel nwc_gemv launches for m on the current device: NWC_ROUTE_LIST
 * when m has more than one column block, m->table is set and every SM's share of the blocks
 * holds at least 32 whole row blocks (row blocks >= 33 x the SM count); else NWC_ROUTE_GEMV.
 * *route receives the value; NWC_ERR_CUDA when the device's SM count cannot be read.
 */
nwc_status nwc_gemv_route(const nwc_matrix *m, int *route);

/*
 * nwc_gemv_next -- nwc_gemv on m, which also brings the block regions, block table and decode
 * table of `next` (the matrix the caller multiplies after this one; NULL: none) into L2 while
 * this call decodes: each warp issues bulk L2 prefetches for its share once its own first
 * regions have landed, so the next call's weights are read from HBM during this call's decode
 * phase instead of at the start of its own. The result is nwc_gemv's, bit for bit. Worth it
 * when next's blob is a small part of the 129 MB L2 (the prefetched lines are evicted before
 * use otherwise). The pages run a whole decoding step as one CUDA graph ("Run a model"); this
 * is the overlap such a fixed sequence of products allows.
 */
nwc_status nwc_gemv_next(const nwc_matrix *m, const uint16_t *x, float *y, void *ws, size_t ws_bytes,
                         const nwc_matrix *next, nwc_stream stream);

/*
 * nwc_gemv_noalloc -- nwc_gemv for callers that cannot allocate device memory: no workspace
 * argument, and no call to cudaMalloc, cudaFree or any allocating routine. The pages have no
 * counterpart; it exists for hosts where device memory belongs to someone else (for example a
 * plugin inside an inference server whose allocator owns the whole device, or a real-time loop
 * where an allocation's implicit device synchronization is not acceptable).
 * The scratch (partial sums, counters) is a file-scope 4 MiB device array inside
 * this library, held by every GPU that loads it until the process exits. A matrix whose
 * nwc_gemv_workspace_bytes exceeds 4 MiB (about 1M rows x 512-column blocks) is rejected with
 * NWC_ERR_INVALID_ARG. Every call zeroes the counters there, then runs
 * the GEMV on the stream; results equal nwc_gemv's. All calls share the one array, so calls that
 * overlap on the GPU (different streams, or different host threads without ordering) race.
 * The first call on a device resolves the array's device address with cudaGetSymbolAddress
 * (on the device current at that moment) and keeps it for later calls on that device.
 */
nwc_status nwc_gemv_noalloc(const nwc_matrix *m, const uint16_t *x, float *y, nwc_stream stream);

/* Largest item count of one nwc_gemv_list call. */
#define NWC_GEMV_LIST_MAX 256

/* One product of an nwc_gemv_list call. */
typedef struct nwc_gemv_item {
    const nwc_matrix *m; /* bound matrix whose device decode table is set (m->table)          */
    const uint16_t *x;   /* BF16[K], 16-byte aligned                                          */
    float *y;            /* FP32[N]                                                           */
    void *ws;            /* a workspace prepared by nwc_gemv_prepare for m, 16-byte aligned   */
    size_t ws_bytes;     /* >= nwc_gemv_workspace_bytes(m)                                    */
} nwc_gemv_item;

/*
 * nwc_gemv_list -- y_i = W_i x_i for `count` independent products (1..NWC_GEMV_LIST_MAX) in one
 * launch. The pages run a whole decoding step, with fused projections, as one CUDA graph ("Run a
 * model": graph_decode with --fusion); this call puts many of that step's matrix-vector products
 * into one persistent kernel instead of one kernel each: every SM takes a contiguous share of all
 * items' blocks, so the per-launch start-up (decode table, first copies) is paid about once per
 * SM instead of once per matrix, and one item's final sums overlap the next item's decoding.
 * Each y_i equals nwc_gemv's result for its item bit for bit. Requirements: every item's x is
 * ready when the call starts (no item reads another item's y: dependent products go in separate
 * calls, in stream order); the y_i overlap neither one another nor any x or workspace; the items'
 * workspaces do not overlap (checked: NWC_ERR_INVALID_ARG); all items have the same element type
 * (NWC_ERR_INVALID_ARG otherwise). The items array is read during the call only. Asynchronous on
 * the stream; a workspace is left in its prepared state, as by nwc_gemv.
 */
nwc_status nwc_gemv_list(const nwc_gemv_item *items, int count, nwc_stream stream);

/* Largest vector count of one nwc_gemv_batch call. */
#define NWC_GEMV_BATCH_MAX 16

/*
 * nwc_gemv_batch_workspace_bytes -- device scratch nwc_gemv_batch needs for m and nb vectors
 * (1 <= nb <= NWC_GEMV_BATCH_MAX; 0 for any other nb): one counter per 8-row block and FP32
 * partial sums per (vector, row, 512-column block), both only when K > 512; at least 16 bytes.
 */
size_t nwc_gemv_batch_workspace_bytes(const nwc_matrix *m, int nb);

/*
 * nwc_gemv_batch_prepare -- as nwc_gemv_prepare, for a batch workspace sized for nb vectors: zeroes
 * its counters on the stream. A workspace prepared for nb serves every call with nb or fewer
 * vectors, repeated calls and graph replays included; calls sharing it must not overlap on the GPU.
 */
nwc_status nwc_gemv_batch_prepare(const nwc_matrix *m, int nb, void *ws, size_t ws_bytes,
                                  nwc_stream stream);

/*
 * nwc_gemv_batch -- Y = W X for nb activation vectors at once: nwc_gemv's decoder, with the
 * products of each decoded 8 x 512 block and all nb vectors done on the tensor cores (BF16
 * operands, FP32 accumulation; fp8 weights widened exactly to BF16). The pages run only batch 1
 * fused (the NWC page, "How it works") and send batch > 1 through a decode to BF16 and cuBLAS;
 * this call covers the small batches in between (a few tokens per step). Every weight is decoded
 * once per call, so the matrix bytes are read, and the codes decoded, once for the whole batch,
 * and any nb up to 16 costs about the same. x: BF16 [nb][ld_x], vector v at x + v*ld_x, x
 * 16-byte aligned, ld_x >= K and a multiple of 8. y: FP32 [nb][ld_y], ld_y >= N. Each y[v]
 * meets nwc_gemv's bound for its own vector (the sum order differs from nwc_gemv's). ws/ws_bytes:
 * a workspace prepared by nwc_gemv_batch_prepare for this matrix and at least nb vectors. nb
 * outside [1, NWC_GEMV_BATCH_MAX] is NWC_ERR_INVALID_ARG. nb == 1 runs nwc_gemv's kernel (on
 * this workspace), with nwc_gemv's result bit for bit; nb == 2 runs it with a second accumulator
 * set (FMAs per vector), which is faster than the tensor-core path for two vectors.
 */
nwc_status nwc_gemv_batch(const nwc_matrix *m, const uint16_t *x, int64_t ld_x, int nb, float *y,
                          int64_t ld_y, void *ws, size_t ws_bytes, nwc_stream stream);

/*
 * nwc_gather -- embedding lookup on the same decoder (the NWC page, "How it works": the
 * embedding lookup of a tied lm_head shares the GEMV's decoder): out row i = row ids[i] of the stored matrix,
 * bit-exact (uint16 BF16 or uint8 e4m3), out[i*ld_out + k]. An id outside [0, N) writes a
 * zero row and raises the device error word. Every id decodes its whole 8-row block row (the
 * format's unit), so a gather costs about 8x the bytes of the rows it returns. Store alignment
 * as for nwc_decode. n_ids x ceil(K / 512) must stay below 2^31 (NWC_ERR_INVALID_ARG otherwise;
 * the output of such a call would not fit in device memory anyway).
 */
nwc_status nwc_gather(const nwc_matrix *m, const int32_t *ids, int64_t n_ids, void *out,
                      int64_t ld_out, nwc_stream stream);

/*
 * nwc_check -- synchronizes the stream, then reads and clears the device error word of the
 * current device. NWC_OK if clear; NWC_ERR_DEVICE_FLAG (format/bounds) or NWC_ERR_TIMEOUT
 * (a bounded wait ran out) otherwise; *flags (if not NULL) receives the raw bits.
 */
nwc_status nwc_check(nwc_stream stream, uint32_t *flags);

/*
 * Blob files -- compressed checkpoints (the NWC page's usage block: a compressed model is
 * saved once and later loaded straight onto the GPU, without the BF16 originals). A file holds
 * named blobs: "NWCF", u32 entry count, then per entry u32 name length, the UTF-8 name (1..4096
 * bytes, unique, no NUL), u64 blob length, zero bytes to the next 16-byte file offset, the blob;
 * the file ends with the last blob. Host calls only, except the copy nwc_file_load enqueues.
 * A file that cannot be opened, read or written is NWC_ERR_IO; a file whose index does not hold
 * together (lengths past its end, duplicate names, trailing bytes) or one of whose blobs fails
 * nwc_validate is NWC_ERR_FORMAT; an index outside [0, count) is NWC_ERR_INVALID_ARG.
 */

/* nwc_file_save -- writes count named blobs (blobs[i], bytes[i] bytes, names[i] a NUL-terminated
 * string) to path, replacing it. Every blob is validated first; on any error nothing at path
 * changes (the file is written beside it and renamed over it). */
nwc_status nwc_file_save(const char *path, int count, const char *const *names, const void *const *blobs,
                         const size_t *bytes);

/* nwc_file_count -- number of entries in the file (its whole index is checked). */
nwc_status nwc_file_count(const char *path, int *count);

/* nwc_file_entry -- name (copied with its NUL into name, name_cap bytes; NULL to skip) and blob
 * length (*bytes; NULL to skip) of entry index. A name longer than name_cap - 1 bytes is
 * NWC_ERR_INVALID_ARG, with *bytes still set. */
nwc_status nwc_file_entry(const char *path, int index, char *name, size_t name_cap, size_t *bytes);

/* nwc_file_find -- index of the entry called name (NWC_ERR_INVALID_ARG if none is). */
nwc_status nwc_file_find(const char *path, const char *name, int *index);

/* nwc_file_read -- entry index's blob into blob_host (cap bytes) and validated; *bytes (if not
 * NULL) receives its length, also when cap is too small (then NWC_ERR_INVALID_ARG). */
nwc_status nwc_file_read(const char *path, int index, void *blob_host, size_t cap, size_t *bytes);

/*
 * nwc_file_load -- entry index read into blob_host (host_cap bytes; page-locked memory makes the
 * copy asynchronous), validated and bound to blob_dev (dev_cap bytes, 16-byte aligned,
 * caller-owned) as nwc_bind does, then copied to blob_dev with one cudaMemcpyAsync on the
 * stream. *out is set only on success; out->table is NULL. blob_host must stay unchanged until
 * the stream has passed the copy; kernels using *out go on the same stream (or wait for it).
 * The blob's length comes from nwc_file_entry.
 */
nwc_status nwc_file_load(const char *path, int index, void *blob_host, size_t host_cap, void *blob_dev,
                         size_t dev_cap, nwc_matrix *out, nwc_stream stream);

/* Streaming multiprocessors of the current device (queried, never assumed). */
int nwc_sm_count(void);

#ifdef __cplusplus
}
#endif

#endif /* NWC_H */
