/*
 * splitzip.h — C ABI of the GB300 (sm_103a) SplitZip lossless KV-cache codec.
 *
 * Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
 * Serving" (gist.science summary page), section "Method: SplitZip".  A BF16,
 * FP8-E5M2 or FP16 tensor is split into
 *   - a 4-bit code per element: the exponent mapped through an offline
 *     calibrated Top-16 codebook, two codes per byte ("Encoding strategy:
 *     Fixed-length coding");
 *   - the sign and mantissa bits, stored raw ("Sign/mantissa preservation";
 *     FP8-E5M2 per Contributions 4; FP16, one of the other formats the page's
 *     Significance section points to, is this library's extension);
 *   - a sparse escape stream of (16-bit in-chunk position, 8-bit exponent)
 *     for exponents outside the codebook ("Escape stream").
 * Decoding maps every code back through a 16-entry table and then overwrites
 * the escaped exponents ("Decoding strategy: Parallelism, Correction"), so the
 * output is bit-identical to the input.
 *
 * Conventions for every entry point:
 *   - The caller owns every buffer.  d_ pointers are CUDA device pointers on
 *     the current device, h_ pointers are host pointers.  The library keeps no
 *     reference to any buffer after the call returns.
 *   - Device work is enqueued on `stream` and is asynchronous: the return value
 *     reports only errors detectable on the host before launch (bad arguments,
 *     too-small buffers, CUDA launch failures).  Data-dependent errors found by
 *     the GPU are written to *d_status (a device int) in stream order.
 *   - Device pointers must be 16-byte aligned (SPLITZIP_ERR_INVALID_ARG
 *     otherwise).
 *   - Elements are raw bits: BF16 and FP16 as 16-bit little-endian words,
 *     FP8-E5M2 as bytes.  No value is special: NaN, inf, signed zeros and subnormals round
 *     trip bit for bit.
 *   - On any error the contents of output buffers are unspecified, but no
 *     access is made outside the buffers at the sizes passed in.
 *
 * Container format v1 (little-endian; every section starts on a 16-byte
 * boundary; all padding bytes are zero).  The page gives no byte format; this
 * layout is this library's own:
 *   off 0   u32 magic 0x50495A53 ("SZIP")   off 4  u16 version = 1
 *   off 6   u8  dtype (splitzip_dtype_t)     off 7  u8  reserved = 0
 *   off 8   u64 n (elements)                 off 16 u32 chunk_elems
 *   off 20  u32 n_chunks C = ceil(n / chunk_elems)
 *   off 24  u64 E = total escapes            off 32 u8  codebook[16]
 *   off 48  16 reserved bytes = 0
 *   off 64  u64 esc_offset[C]: exclusive prefix sum of esc_count
 *           u32 esc_count[C]:  escapes in chunk c
 *   A16     nibble stream, ceil(n/2) bytes: element 2k in the low nibble of
 *           byte k, element 2k+1 in the high nibble; an escaped element's
 *           nibble is 0
 *   A16     sign|mantissa stream: BF16 one byte per element,
 *           (sign << 7) | mantissa7; FP8-E5M2 3 bits per element,
 *           (sign << 2) | mantissa2, LSB-first bitstream, element i at bits
 *           [3i, 3i+3), padded with zero bits to 3*ceil(n/8) bytes; FP16 11
 *           bits per element, (sign << 10) | mantissa10, the same way at bits
 *           [11i, 11i+11), 11*ceil(n/8) bytes
 *   A16     escape records, 3 bytes each: the in-chunk position (u16,
 *           little-endian) then the original exponent (u8; E5M2 and FP16:
 *           the 5-bit exponent zero-extended); chunk by chunk, ascending
 *           position within a chunk; the container ends after the last record.
 * Size = A16(64 + 12C) + A16(ceil(n/2)) + A16(S) + 3E, A16 = round up to 16,
 * S = n (BF16), 3*ceil(n/8) (FP8-E5M2) or 11*ceil(n/8) (FP16).
 * chunk_elems is a power of two in [64, 65536] (the 16-bit position field of
 * the escape records bounds it; the page uses 65,536-element chunks).
 */
#ifndef SPLITZIP_H
#define SPLITZIP_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SPLITZIP_BF16 = 0,      /* bfloat16: 1 sign, 8 exponent, 7 mantissa bits */
    SPLITZIP_FP8_E5M2 = 1,  /* FP8-E5M2: 1 sign, 5 exponent, 2 mantissa bits */
    SPLITZIP_FP16 = 2       /* IEEE half: 1 sign, 5 exponent, 10 mantissa bits */
} splitzip_dtype_t;

typedef enum {
    SPLITZIP_OK = 0,
    SPLITZIP_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad dtype, chunk size, codebook */
    SPLITZIP_ERR_CAPACITY = 2,    /* output or workspace smaller than required */
    SPLITZIP_ERR_CORRUPT = 3,     /* container inconsistent (header, index, escapes, size) */
    SPLITZIP_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    SPLITZIP_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (never expected) */
    SPLITZIP_ERR_UNSUPPORTED = 6  /* no sm_103a device, or a size beyond the limits */
} splitzip_status_t;

#define SPLITZIP_DEFAULT_CHUNK_ELEMS 65536u
#define SPLITZIP_HEADER_BYTES 64u

/* Top-16 codebook: code i stands for exponent exps[i].  The 16 values must be
 * distinct and below 256 (BF16) or 32 (FP8-E5M2, FP16). */
typedef struct {
    uint8_t dtype;    /* splitzip_dtype_t */
    uint8_t exps[16];
} splitzip_codebook_t;

/* Parsed header plus the derived section offsets (bytes from blob start). */
typedef struct {
    uint64_t n_elems;
    uint64_t total_escapes;
    uint64_t size;          /* total container bytes */
    uint64_t index_off, counts_off, nibble_off, signmant_off, escrec_off;
    uint32_t chunk_elems;
    uint32_t n_chunks;
    uint8_t dtype;
    uint8_t codebook[16];
} splitzip_header_t;

/* Human-readable name of a splitzip_status_t value (static storage). */
const char* splitzip_status_string(int status);

/* Exponent histogram of n elements (Results, "Ablations: Calibration": the
 * codebook is calibrated offline from exponent statistics).
 * d_x: n elements of `dtype`; d_hist256: 256 u64 counts, overwritten (bins
 * 32..255 stay 0 for FP8-E5M2 and FP16).  Enqueued on `stream`. */
int splitzip_exponent_histogram(const void* d_x, uint64_t n, int dtype, uint64_t* d_hist256,
                                cudaStream_t stream);

/* Top-16 codebook from a 256-bin exponent histogram (Method, "Fixed-length
 * coding": the 16 most frequent exponents get the 4-bit codes).  Ties go to
 * the smaller exponent; unseen exponents fill the remaining codes in
 * ascending order; code 0 is the most frequent exponent.
 * hist256: host array, or device array on the current device when
 * hist_is_device != 0: the call then blocks in cudaDeviceSynchronize() until
 * all work queued on every stream of the device has finished (so a histogram
 * that splitzip_exponent_histogram enqueued on any stream, non-blocking
 * streams included, is complete) and copies the 256 counts to the host.
 * FP8-E5M2 and FP16 histograms with counts in bins >= 32 are rejected. */
int splitzip_calibrate(const uint64_t* hist256, int hist_is_device, int dtype,
                       splitzip_codebook_t* out_cb);

/* Container size for n elements with exactly `total_escapes` escapes. */
int splitzip_compressed_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t total_escapes,
                             uint64_t* out_bytes);

/* Worst-case container size (every element escapes): the capacity that
 * splitzip_encode requires of d_out. */
int splitzip_max_compressed_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t* out_bytes);

/* Device scratch bytes splitzip_encode needs for n elements: about 4 bytes
 * per element (each tile of 16 KB of input -- 8,192 BF16 / FP16 or 16,384
 * E5M2 elements -- or each chunk when chunks are smaller, has a staging slot big
 * enough for all of its elements to escape) plus 40 bytes per tile and 4 per
 * 256 tiles. */
int splitzip_encode_workspace_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t* out_bytes);

/* Encode n elements (Method, "Encoding strategy").  Four kernels, no waits
 * between blocks: a streaming pass that writes the nibble and sign|mantissa
 * streams and stages each tile's escape records in element order, a pass
 * that totals the escapes of every 256 tiles, a pass that computes the index
 * (per-chunk offsets and counts), and a pass that moves the records into the
 * escape stream.  The input is read through a
 * tensor map (cuTensorMapEncodeTiled, fetched from the runtime with
 * cudaGetDriverEntryPointByVersion); SPLITZIP_ERR_CUDA if that fails.
 * d_in: n elements; cb: host codebook of the same dtype; d_out: container,
 * out_capacity >= splitzip_max_compressed_size; d_ws: ws_bytes >=
 * splitzip_encode_workspace_size, contents need not be initialised; d_out_size: device u64 that receives the
 * container size; d_status: device int, cleared by the call; it becomes
 * SPLITZIP_ERR_TIMEOUT only if a bounded wait on a bulk copy ran out (not
 * expected).  n = 0 is valid and gives a 64-byte container.  Calls that share
 * d_ws must not overlap on the GPU. */
int splitzip_encode(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                    uint32_t chunk_elems, void* d_out, uint64_t out_capacity, void* d_ws,
                    uint64_t ws_bytes, uint64_t* d_out_size, int* d_status, cudaStream_t stream);

/* Online calibration, all on the device and stream-ordered (no host
 * synchronisation): the exponent histogram of d_x into d_hist256 (as
 * splitzip_exponent_histogram), then its Top-16 codebook (Method, "Top-16
 * exponent coding"; count descending, exponent ascending on ties, as
 * splitzip_calibrate) into the device struct *d_cb.  The page calibrates
 * offline to avoid exactly this pass (section "Method: SplitZip", and Results,
 * "Ablations: Calibration"); this entry point measures what it costs.
 * d_hist256: device, 256 u64, 16-byte aligned; d_cb: device splitzip_codebook_t. */
int splitzip_calibrate_device(const void* d_x, uint64_t n, int dtype, uint64_t* d_hist256,
                              splitzip_codebook_t* d_cb, cudaStream_t stream);

/* splitzip_encode with the codebook in device memory (d_cb, e.g. written by
 * splitzip_calibrate_device), so that calibrate and encode can follow each
 * other on a stream without the host.  The GPU checks the codebook (its
 * dtype field, exponents in range and distinct) and writes
 * SPLITZIP_ERR_INVALID_ARG to *d_status for a bad one (output unspecified).
 * Everything else as splitzip_encode; the output is byte-identical to
 * splitzip_encode's with the same codebook on the host. */
int splitzip_encode_device_codebook(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* d_cb,
                                    uint32_t chunk_elems, void* d_out, uint64_t out_capacity, void* d_ws,
                                    uint64_t ws_bytes, uint64_t* d_out_size, int* d_status, cudaStream_t stream);

/* Size of the device array that splitzip_encode_noalloc uses as scratch. */
#define SPLITZIP_NOALLOC_SCRATCH_BYTES (32ull << 20)

/* splitzip_encode without a caller-provided workspace.  The SplitZip page has
 * no counterpart to this entry point; it exists for callers that cannot
 * allocate device memory at encode time: a serving engine whose KV pool and
 * allocator already own nearly all of the GPU's memory, or a path that must
 * not call cudaMalloc/cudaFree because they can synchronise the device.
 * Its scratch is a fixed device array of SPLITZIP_NOALLOC_SCRATCH_BYTES
 * (32 MiB) held by every GPU that loads this library until the process
 * exits.  Limits: n must satisfy splitzip_encode_workspace_size(n, dtype,
 * chunk_elems) <= SPLITZIP_NOALLOC_SCRATCH_BYTES (8,372,224 elements at the
 * default chunk size, for either dtype); larger n returns SPLITZIP_ERR_CAPACITY before any GPU
 * work.  The call allocates nothing: the caller still passes input, output,
 * d_out_size and d_status exactly as for splitzip_encode, and the output is
 * byte-identical to splitzip_encode's.  Every call looks up the array's
 * device address on the current device (cudaGetSymbolAddress), so an address
 * from before a device reset is never reused; the first call on a device also
 * loads the library's device code there, so make that first call before any
 * stream capture.  Every call on a device
 * shares the array, so calls whose GPU work overlaps (other streams or host
 * threads) race and must be serialised by the caller.  The encode writes
 * every word of its workspace before reading it, so whatever an earlier call
 * left in the array does no harm. */
int splitzip_encode_noalloc(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                            uint32_t chunk_elems, void* d_out, uint64_t out_capacity,
                            uint64_t* d_out_size, int* d_status, cudaStream_t stream);

/* Decode a container into n elements (Method, "Decoding strategy").
 * d_in: in_bytes bytes of container (in_bytes >= its size); d_out: n
 * elements.  The GPU checks the header (magic, version, dtype and n equal to
 * the arguments, chunk size, sizes against in_bytes), the index (offsets are
 * the prefix of the counts, counts fit their chunks) and every escape
 * (position inside its chunk and ascending, exponent in range); on a
 * mismatch it writes SPLITZIP_ERR_CORRUPT to *d_status, else SPLITZIP_OK. */
int splitzip_decode(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n, int dtype,
                    int* d_status, cudaStream_t stream);

/* Paged KV cache (serving engines keep a cache in fixed-size pages of a pool,
 * listed per request in a page table; a transfer gathers them on the sending
 * side and scatters them on the receiving one).  d_pool holds pool_pages
 * pages of page_elems elements each (page_elems a power of two); d_pages
 * (device int32, n_pages entries) lists the pages of the tensor in order.
 * splitzip_encode_paged encodes the n_pages * page_elems elements of those
 * pages, gathered by the encoder's tensor-map copies straight from the pool:
 * the container is byte-identical to splitzip_encode of the gathered tensor.
 * page_elems must be a multiple of the encoder's tile (8,192 BF16 / FP16 or
 * 16,384 E5M2 elements, or chunk_elems when that is smaller).  The workspace and
 * output sizes are those of n = n_pages * page_elems elements.  A page index
 * outside [0, pool_pages) is reported in *d_status as
 * SPLITZIP_ERR_INVALID_ARG (and never read). */
int splitzip_encode_paged(const void* d_pool, uint64_t pool_pages, const int32_t* d_pages, uint64_t n_pages,
                          uint64_t page_elems, int dtype, const splitzip_codebook_t* cb, uint32_t chunk_elems,
                          void* d_out, uint64_t out_capacity, void* d_ws, uint64_t ws_bytes, uint64_t* d_out_size,
                          int* d_status, cudaStream_t stream);

/* Decode a container of n_pages * page_elems elements into the pages listed
 * in d_pages of the pool d_pool (element g goes to element g mod page_elems
 * of page d_pages[g / page_elems]); every other byte of the pool is left as
 * it is.  page_elems: a power of two >= 16.  Checks as splitzip_decode; a
 * page index outside the pool is reported (SPLITZIP_ERR_INVALID_ARG in
 * *d_status) and never written. */
int splitzip_decode_paged(const void* d_in, uint64_t in_bytes, void* d_pool, uint64_t pool_pages,
                          const int32_t* d_pages, uint64_t n_pages, uint64_t page_elems, int dtype, int* d_status,
                          cudaStream_t stream);

/* The page's ablation formats (section "Results", "Ablation Studies"):
 * variant 1 = Top-8 (8 coded exponents, 3-bit codes packed LSB-first, 3 bytes
 * per 8 elements; escapes as 3-byte (position, exponent) records), variant 2 =
 * Top-15 + sentinel (15 coded exponents; code 15 marks an escape; the escape
 * stream holds one exponent byte per escape, positions found from the
 * sentinels), variant 0 = Top-16 (the main format, byte-identical to
 * splitzip_encode's container).  Header, index and sign|mantissa stream as the
 * main format; header byte 7 = the variant.  These entry points run one plain
 * kernel family for all three (the production Top-16 kernels are
 * splitzip_encode / splitzip_decode), so their measured speeds differ by the
 * formats alone.  The codebook holds the variant's k = 16, 8 or 15 exponents
 * (the first k of the Top-16 order), distinct and in range, then zeros.
 * splitzip_ablation_max_size: the container size with every element
 * escaping.  Encode: no workspace (the counts go to the container's index);
 * three kernels.  Decode: the header, index and escapes are checked like
 * splitzip_decode's; errors go to *d_status. */
int splitzip_ablation_max_size(uint64_t n, int dtype, uint32_t chunk_elems, int variant, uint64_t* out_bytes);
int splitzip_ablation_encode(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                             uint32_t chunk_elems, int variant, void* d_out, uint64_t out_capacity,
                             uint64_t* d_out_size, int* d_status, cudaStream_t stream);
int splitzip_ablation_decode(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n, int dtype, int variant,
                             int* d_status, cudaStream_t stream);

/* Parse and check a container header held in host memory (bytes >= 64).
 * Returns SPLITZIP_ERR_CORRUPT for a malformed header or a size larger than
 * `bytes`. */
int splitzip_parse_header(const void* h_blob, uint64_t bytes, splitzip_header_t* out);

/* Scratch that splitzip_transfer needs: device bytes (with compress = 1: a
 * ring of 4 send and 4 receive slots, each one piece's maximum container
 * size, one encode workspace and 16 bytes per piece; 0 with compress = 0) and
 * pinned host bytes (a ring of 4 staging slots, each a maximum container or,
 * with compress = 0, a raw piece, plus 16 bytes per piece when compressing).
 * Slots are rounded up to A = 2 MiB (64 KiB when a slot is under 2 MiB) and
 * each area has A - 16 bytes more, so that a 16-byte-aligned base can be
 * moved up to the next multiple of A.  SPLITZIP_ERR_INVALID_ARG unless n > 0
 * and piece_elems is a positive multiple of chunk_elems. */
int splitzip_transfer_scratch_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t piece_elems,
                                   int compress, uint64_t* out_device_bytes, uint64_t* out_host_bytes);

/* Move n elements from d_src to d_dst (both on the current GPU) across the
 * GPU <-> host link, the transfer that the page speeds up (section
 * "Results": prefill-to-decode KV transfer in disaggregated serving).  The
 * tensor is cut into pieces of piece_elems elements (whole chunks; the last
 * piece may be shorter).  compress = 1: each piece is encoded into its own
 * container, exactly the container's bytes are copied device -> h_stage and
 * back, and the received container is decoded into d_dst; compress = 0: the
 * raw piece is copied the same way (the baseline).  Encode, the two copies
 * and decode of different pieces overlap on four internal streams; the host
 * reads each container's size, which a one-thread kernel behind its encode
 * stores into h_stage through the device's mapping of it (a 12-byte copy
 * where h_stage has no device mapping), while the next piece encodes.  The call starts after the work already on `stream`,
 * makes `stream` wait for its end, and blocks until d_dst is complete.
 * d_scratch / h_stage: at least splitzip_transfer_scratch_size's bytes,
 * 16-byte aligned, h_stage page-locked host memory (cudaHostAlloc or
 * cudaHostRegister; SPLITZIP_ERR_INVALID_ARG otherwise).  out_link_bytes
 * (optional): the bytes that crossed the link in each direction;
 * out_ms (optional): GPU time from the first to the last operation.  An
 * encode or decode error of any piece is returned (the first one found). */
int splitzip_transfer(const void* d_src, void* d_dst, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                      uint32_t chunk_elems, uint64_t piece_elems, int compress, void* d_scratch,
                      uint64_t d_scratch_bytes, void* h_stage, uint64_t h_stage_bytes, uint64_t* out_link_bytes,
                      float* out_ms, cudaStream_t stream);

/* Batches: several tensors, each into (or from) its own container, in one
 * launch sequence.  The page's transfers are per request and per layer
 * (section "Results": the gains vary with sequence length and batch size), so
 * a serving engine moves many pieces of a few megabytes; at that size a call
 * costs its launches, not HBM time, and a batch pays them once.
 * splitzip_encode and splitzip_decode take the same path on their own for
 * small tensors (encode: up to 8,192 tiles -- 67,108,864 BF16 / FP16 or
 * 134,217,728 E5M2 elements at the default chunk, as one cooperative kernel
 * when the tiles fit the GPU at once; decode: up to 2^21 elements), so a
 * single small call gains the same way.
 * Limits: 1..SPLITZIP_MAX_BATCH items, each of at most
 * SPLITZIP_MAX_BATCH_ITEM_ELEMS elements (SPLITZIP_ERR_UNSUPPORTED beyond);
 * all items share dtype, chunk size and codebook; one status word for the
 * whole batch (the first error of any item).  The item arrays are host memory
 * read during the call only; every pointer in them follows the rules of the
 * single-tensor calls (device, 16-byte aligned; d_out_size 8-byte aligned). */
#define SPLITZIP_MAX_BATCH 256u
#define SPLITZIP_MAX_BATCH_ITEM_ELEMS (1ull << 26)

typedef struct {
    const void* d_in;      /* n elements */
    uint64_t n;
    void* d_out;           /* the item's container, out_capacity >= splitzip_max_compressed_size */
    uint64_t out_capacity;
    uint64_t* d_out_size;  /* device u64: the container's size */
} splitzip_encode_item_t;

typedef struct {
    const void* d_in;      /* in_bytes bytes of container (>= its size) */
    uint64_t in_bytes;
    void* d_out;           /* n elements */
    uint64_t n;
} splitzip_decode_item_t;

/* Workspace bytes for splitzip_encode_batch: each item's
 * splitzip_encode_workspace_size rounded up to 256 bytes, summed; h_n: the
 * items' element counts (host). */
int splitzip_encode_batch_workspace_size(const uint64_t* h_n, uint32_t count, int dtype, uint32_t chunk_elems,
                                         uint64_t* out_bytes);

/* Encode every item into its own container (byte-identical to splitzip_encode
 * of that item).  Three kernels for the whole batch, chained with
 * programmatic dependent launch: one CTA per 16 KB tile of every item, the
 * index of every item, the escape records of every tile.  d_ws: at least
 * splitzip_encode_batch_workspace_size bytes, contents need not be
 * initialised; d_status: device int, set by the call (SPLITZIP_OK or the
 * first error).  Calls that share d_ws must not overlap on the GPU. */
int splitzip_encode_batch(const splitzip_encode_item_t* h_items, uint32_t count, int dtype,
                          const splitzip_codebook_t* cb, uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes,
                          int* d_status, cudaStream_t stream);

/* Decode every item's container into its elements (each bit-identical to
 * splitzip_decode of it), checked as splitzip_decode checks; errors of any
 * item go to *d_status.  A one-thread kernel clears the status word, then one
 * CTA per 16,384 elements of every item decodes, patches and checks. */
int splitzip_decode_batch(const splitzip_decode_item_t* h_items, uint32_t count, int dtype, int* d_status,
                          cudaStream_t stream);

/* Join the containers of consecutive pieces of one tensor into the container
 * of the whole tensor, byte-identical to encoding it in one call.  Chunks are
 * independent (Method, "Escape stream": positions are 16-bit offsets within a
 * chunk), so a tensor can be encoded in pieces of whole chunks -- one piece
 * per GPU when the work is spread over several, or one per layer -- and
 * joined afterwards; the escape offsets of piece i move by the escapes of
 * pieces 0..i-1 (an exclusive scan of the per-piece totals).  Host memory
 * only: h_parts[i] holds part_bytes[i] bytes of piece i's container (pieces
 * in tensor order).  Every piece must have the same dtype, chunk size and
 * codebook, and every piece but the last a whole number of chunks
 * (SPLITZIP_ERR_INVALID_ARG otherwise); a malformed header or index gives
 * SPLITZIP_ERR_CORRUPT.  *out_bytes receives the merged size; with h_out ==
 * NULL nothing else happens (a size query), else out_capacity must cover
 * that size (SPLITZIP_ERR_CAPACITY) and h_out receives the container. */
int splitzip_merge(const void* const* h_parts, const uint64_t* part_bytes, uint32_t count, void* h_out,
                   uint64_t out_capacity, uint64_t* out_bytes);

/* Self-test of the bounded device wait.  Every wait of the encode and
 * decode kernels on a bulk-copy barrier gives up after a bounded number of SM
 * cycles (about one second), records SPLITZIP_ERR_TIMEOUT in the status word
 * and lets the kernel finish, so that a failed copy cannot hang the GPU; in a
 * healthy run that path never executes.  This call runs it on purpose with no
 * copy in flight: one warp waits, limit_cycles SM cycles at most, on an
 * mbarrier that nothing arrives on, then reports exactly as the streaming
 * kernels do.  The page has no counterpart (the codec never waits on data).
 * limit_cycles: 1 .. 2e9.  d_status: device int, cleared by the call, then
 * SPLITZIP_ERR_TIMEOUT (the expected outcome; a control wait on a completed
 * barrier must also succeed, else the status is the same and d_cycles[1] is
 * -1).  d_cycles (optional, device, 2 x int64): cycles the giving-up wait
 * took, and cycles the control wait took. */
int splitzip_selftest_bounded_wait(uint64_t limit_cycles, int* d_status, long long* d_cycles,
                                   cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPLITZIP_H */
