// Host side of the SplitZip C ABI declared in include/splitzip.h: argument
// checks, container geometry, codebook calibration, and the stream-ordered
// launch sequence of the encode / decode / histogram kernels.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "splitzip_internal.cuh"

using namespace splitzip;

namespace {

constexpr uint64_t kMaxElems = uint64_t(1) << 48;  // keeps every size below 2^52
// Up to these sizes a single call takes the small-tensor kernels of batch.cu
// (the persistent kernels' grids would not fill the GPU, and launches and
// dependent memory round trips dominate): encode by one cooperative kernel
// when every tile gets its own resident CTA, else by the two-kernel batch
// path up to kSmallEncodeTiles; decode by the batch decoder up to
// kSmallDecodeElems.
constexpr uint64_t kSmallEncodeTiles = 8192;
constexpr uint64_t kSmallDecodeElems = uint64_t(1) << 21;
constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready;
    int status;
    int sms;
    int encode_bpsm[3], decode_bpsm[3], hist_bpsm[3];  // per dtype
    int coop_encode_bpsm[3];
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];

// Per-device facts, computed once: SM count and resident CTAs per SM of
// every kernel (grids are sized as a multiple of the SM count).
int device_state(DeviceState* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SPLITZIP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SPLITZIP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        d.status = SPLITZIP_OK;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return SPLITZIP_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            d.status = SPLITZIP_ERR_UNSUPPORTED;  // the kernels are built for sm_103a only
        } else {
            for (int t = 0; t < 3; ++t) {
                if (occupancy_encode(&d.encode_bpsm[t], t) != cudaSuccess ||
                    occupancy_decode(&d.decode_bpsm[t], t) != cudaSuccess ||
                    occupancy_histogram(&d.hist_bpsm[t], t) != cudaSuccess ||
                    occupancy_coop(&d.coop_encode_bpsm[t], t) != cudaSuccess) {
                    cudaGetLastError();
                    return SPLITZIP_ERR_CUDA;
                }
            }
        }
        d.ready = true;
    }
    *out = d;
    return d.status;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool valid_dtype(int dtype) { return dtype == SPLITZIP_BF16 || dtype == SPLITZIP_FP8_E5M2 || dtype == SPLITZIP_FP16; }
bool valid_chunk(uint32_t c) { return c >= kMinChunk && c <= kMaxChunk && (c & (c - 1u)) == 0u; }
uint32_t exponent_bins(int dtype) { return dtype == SPLITZIP_BF16 ? 256u : 32u; }

int check_geometry(uint64_t n, int dtype, uint32_t chunk) {
    if (!valid_dtype(dtype) || !valid_chunk(chunk)) return SPLITZIP_ERR_INVALID_ARG;
    if (n > kMaxElems || (n + chunk - 1u) / chunk > 0xFFFFFFFFull) return SPLITZIP_ERR_UNSUPPORTED;
    return SPLITZIP_OK;
}

int check_codebook(const splitzip_codebook_t* cb, int dtype) {
    if (!cb || cb->dtype != dtype) return SPLITZIP_ERR_INVALID_ARG;
    bool seen[256] = {false};
    for (int i = 0; i < 16; ++i) {
        const uint8_t e = cb->exps[i];
        if (e >= exponent_bins(dtype) || seen[e]) return SPLITZIP_ERR_INVALID_ARG;
        seen[e] = true;
    }
    return SPLITZIP_OK;
}

int grid_for(uint64_t work_items, int sms, int blocks_per_sm) {
    const uint64_t cap = uint64_t(sms) * uint64_t(blocks_per_sm > 0 ? blocks_per_sm : 1);
    return int(std::max<uint64_t>(1, std::min<uint64_t>(work_items, cap)));
}

// Argument checks of splitzip_encode; fills the kernel arguments.
// cb is a host codebook (checked here) or, with device_cb, the device address
// of one (checked by the kernel).
int prepare_encode(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb, uint32_t chunk,
                   void* d_out, uint64_t out_capacity, void* d_ws, uint64_t ws_bytes, uint64_t* d_out_size,
                   int* d_status, EncodeArgs* a, Workspace* W, bool device_cb = false) {
    int st = check_geometry(n, dtype, chunk);
    if (st != SPLITZIP_OK) return st;
    if (device_cb ? !cb : (st = check_codebook(cb, dtype)) != SPLITZIP_OK) return device_cb ? SPLITZIP_ERR_INVALID_ARG : st;
    if (n > 0 && (!d_in || !aligned(d_in, 16))) return SPLITZIP_ERR_INVALID_ARG;
    if (!d_out || !aligned(d_out, 16)) return SPLITZIP_ERR_INVALID_ARG;
    if (!d_out_size || !aligned(d_out_size, 8) || !d_status || !aligned(d_status, 4))
        return SPLITZIP_ERR_INVALID_ARG;
    if (out_capacity < layout_for(n, dtype, chunk, n).size) return SPLITZIP_ERR_CAPACITY;
    *W = workspace_for(n, dtype, chunk);
    if (ws_bytes < W->bytes) return SPLITZIP_ERR_CAPACITY;
    if (W->bytes > 0 && (!d_ws || !aligned(d_ws, 16))) return SPLITZIP_ERR_INVALID_ARG;

    uint8_t* ws = static_cast<uint8_t*>(d_ws);
    a->in = d_in;
    a->n = n;
    a->out = static_cast<uint8_t*>(d_out);
    a->group_totals = reinterpret_cast<uint32_t*>(ws + W->group_off);
    a->warp_counts = reinterpret_cast<uint32_t*>(ws + W->warp_count_off);
    a->tile_first = reinterpret_cast<uint64_t*>(ws + W->tile_first_off);
    a->staging = reinterpret_cast<uint32_t*>(ws + W->staging_off);
    a->out_size = d_out_size;
    a->error = d_status;
    a->n_tiles = W->n_tiles;
    a->n_groups = W->n_groups;
    a->tile_elems = W->tile_elems;
    a->chunk_elems = chunk;
    a->n_chunks = layout_for(n, dtype, chunk, 0).n_chunks;
    a->dtype = dtype;
    if (device_cb) {
        std::memset(a->codebook, 0, 16);
        a->dev_codebook = reinterpret_cast<const uint8_t*>(cb);
    } else {
        std::memcpy(a->codebook, cb->exps, 16);
        a->dev_codebook = nullptr;
    }
    a->tensor_bytes = 0;
    a->box_bytes = 0;
    return SPLITZIP_OK;
}

// The driver's tensor-map encoder, fetched once through the runtime (the
// library does not link the driver library itself).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map of the encoder's input: a 2-D tensor of 128-byte rows (the
// input's whole rows; its last partial row, if any, is read by the consumers
// directly), one box = one tile.  Tiles of 128 bytes and more are copied with
// the 128-byte swizzle; the only smaller tile (E5M2 with 64-element chunks,
// 64 bytes) fits in one row and is copied unswizzled.  Row coordinates are
// 32-bit signed, so at most 2^31 - 256 rows are mapped; bytes past them are
// also read directly.
int make_input_map(const void* d_in, int dtype, EncodeArgs* a, CUtensorMap* map, uint64_t in_bytes) {
    std::memset(map, 0, sizeof(*map));
    const uint64_t eb = elem_bytes(dtype);
    const uint64_t rows = std::min<uint64_t>(in_bytes / 128u, (uint64_t(1) << 31) - 256u);
    if (rows == 0) return SPLITZIP_OK;  // every byte is read directly
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return SPLITZIP_ERR_CUDA;
    const uint32_t tile_bytes = a->tile_elems * uint32_t(eb);
    const uint32_t box_row_bytes = std::min<uint32_t>(tile_bytes, 128u);
    const cuuint64_t dims[2] = {128u / eb, rows};
    const cuuint64_t strides[1] = {128u};
    const cuuint32_t box[2] = {cuuint32_t(box_row_bytes / eb), cuuint32_t(tile_bytes / box_row_bytes)};
    const cuuint32_t elem_strides[2] = {1u, 1u};
    const CUresult r =
        encode(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
               const_cast<void*>(d_in), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
               box_row_bytes == 128u ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return SPLITZIP_ERR_CUDA;
    a->tensor_bytes = rows * 128u;
    a->box_bytes = tile_bytes;
    return SPLITZIP_OK;
}

}  // namespace

extern "C" {

const char* splitzip_status_string(int status) {
    switch (status) {
        case SPLITZIP_OK: return "ok";
        case SPLITZIP_ERR_INVALID_ARG: return "invalid argument";
        case SPLITZIP_ERR_CAPACITY: return "buffer too small";
        case SPLITZIP_ERR_CORRUPT: return "corrupt container";
        case SPLITZIP_ERR_CUDA: return "CUDA error";
        case SPLITZIP_ERR_TIMEOUT: return "device wait timed out";
        case SPLITZIP_ERR_UNSUPPORTED: return "unsupported device or size";
        default: return "unknown status";
    }
}

int splitzip_compressed_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t total_escapes,
                             uint64_t* out_bytes) {
    int st = check_geometry(n, dtype, chunk_elems);
    if (st != SPLITZIP_OK) return st;
    if (!out_bytes || total_escapes > n) return SPLITZIP_ERR_INVALID_ARG;
    *out_bytes = layout_for(n, dtype, chunk_elems, total_escapes).size;
    return SPLITZIP_OK;
}

int splitzip_max_compressed_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t* out_bytes) {
    return splitzip_compressed_size(n, dtype, chunk_elems, n, out_bytes);
}

int splitzip_encode_workspace_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t* out_bytes) {
    int st = check_geometry(n, dtype, chunk_elems);
    if (st != SPLITZIP_OK) return st;
    if (!out_bytes) return SPLITZIP_ERR_INVALID_ARG;
    *out_bytes = workspace_for(n, dtype, chunk_elems).bytes;
    return SPLITZIP_OK;
}

int splitzip_calibrate(const uint64_t* hist256, int hist_is_device, int dtype, splitzip_codebook_t* out_cb) {
    if (!hist256 || !out_cb || !valid_dtype(dtype)) return SPLITZIP_ERR_INVALID_ARG;
    uint64_t h[256];
    if (hist_is_device) {
        // A histogram enqueued on any stream of the device (non-blocking
        // streams and per-thread default streams included) is complete after a
        // device-wide synchronisation; a plain cudaMemcpy would order only
        // against the legacy default stream.
        if (cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(h, hist256, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return SPLITZIP_ERR_CUDA;
        }
    } else {
        std::memcpy(h, hist256, sizeof(h));
    }
    const uint32_t bins = exponent_bins(dtype);
    for (uint32_t b = bins; b < 256; ++b)
        if (h[b] != 0) return SPLITZIP_ERR_INVALID_ARG;
    // Most frequent first; the stable sort keeps ascending exponent order on ties.
    uint16_t order[256];
    for (uint32_t b = 0; b < bins; ++b) order[b] = uint16_t(b);
    std::stable_sort(order, order + bins, [&](uint16_t x, uint16_t y) { return h[x] > h[y]; });
    out_cb->dtype = uint8_t(dtype);
    for (int i = 0; i < 16; ++i) out_cb->exps[i] = uint8_t(order[i]);
    return SPLITZIP_OK;
}

int splitzip_exponent_histogram(const void* d_x, uint64_t n, int dtype, uint64_t* d_hist256,
                                cudaStream_t stream) {
    if (!valid_dtype(dtype) || !d_hist256 || !aligned(d_hist256, 16)) return SPLITZIP_ERR_INVALID_ARG;
    if (n > 0 && (!d_x || !aligned(d_x, 16))) return SPLITZIP_ERR_INVALID_ARG;
    if (n > kMaxElems) return SPLITZIP_ERR_UNSUPPORTED;
    DeviceState d;
    int st = device_state(&d);
    if (st != SPLITZIP_OK) return st;
    if (cudaMemsetAsync(d_hist256, 0, 256 * sizeof(uint64_t), stream) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    if (n == 0) return SPLITZIP_OK;
    const uint64_t vec_per_block = uint64_t(kHistThreads);
    const uint64_t vecs = n * elem_bytes(dtype) / 16;
    const int grid = grid_for((vecs + vec_per_block - 1) / vec_per_block, d.sms, d.hist_bpsm[dtype]);
    return launch_histogram(d_x, n, dtype, reinterpret_cast<unsigned long long*>(d_hist256), grid, stream) ==
                   cudaSuccess
               ? SPLITZIP_OK
               : SPLITZIP_ERR_CUDA;
}

namespace {

// Paged input for encode_call: the pool and its page list (null: contiguous).
struct PagedInput {
    const int32_t* pages = nullptr;
    uint64_t pool_pages = 0, page_elems = 0;
};

int encode_call(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb, uint32_t chunk_elems,
                void* d_out, uint64_t out_capacity, void* d_ws, uint64_t ws_bytes, uint64_t* d_out_size,
                int* d_status, cudaStream_t stream, bool device_cb, const PagedInput& paged = PagedInput()) {
    EncodeArgs a;
    Workspace W;
    int st = prepare_encode(d_in, n, dtype, cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes, d_out_size,
                            d_status, &a, &W, device_cb);
    if (st != SPLITZIP_OK) return st;
    const uint64_t eb = elem_bytes(dtype);
    a.pages = paged.pages;
    a.pool_pages = paged.pool_pages;
    a.page_tile_shift = 0;
    if (paged.pages) {
        const uint64_t tiles_per_page = paged.page_elems / a.tile_elems;
        while ((uint64_t(1) << a.page_tile_shift) < tiles_per_page) ++a.page_tile_shift;
        // the tensor map must reach every byte of the pool
        if (paged.pool_pages * paged.page_elems * eb > ((uint64_t(1) << 31) - 256u) * 128u)
            return SPLITZIP_ERR_UNSUPPORTED;
    }
    DeviceState d;
    if ((st = device_state(&d)) != SPLITZIP_OK) return st;
    if (!paged.pages && W.n_tiles > 0 && W.n_tiles <= kSmallEncodeTiles) {
        // a small tensor (batch.cu)
        const SmallEncodeItem item{d_in, n, d_out, d_out_size, d_ws};
        const uint8_t* host_cb = device_cb ? nullptr : cb->exps;
        const uint8_t* dev_cb = device_cb ? reinterpret_cast<const uint8_t*>(cb) : nullptr;
        const uint64_t resident = uint64_t(d.sms) * uint64_t(d.coop_encode_bpsm[dtype]);
        const cudaError_t e =
            W.n_tiles <= resident
                ? launch_coop_encode(item, dtype, host_cb, dev_cb, chunk_elems, d_status, int(W.n_tiles), stream)
                : launch_small_encode(&item, 1, dtype, host_cb, dev_cb, chunk_elems, d_status, stream);
        if (e != cudaSuccess) cudaGetLastError();
        return e == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
    }
    CUtensorMap map;
    const uint64_t mapped = paged.pages ? paged.pool_pages * paged.page_elems * eb : n * eb;
    if ((st = make_input_map(d_in, dtype, &a, &map, mapped)) != SPLITZIP_OK) return st;
    a.staged_bytes = paged.pages ? ~uint64_t(0) : a.tensor_bytes;
    EncodeLut lut;
    std::memset(lut.code, kEscapeFlag, sizeof(lut.code));
    if (!device_cb)
        for (int k = 0; k < 16; ++k) lut.code[cb->exps[k]] = uint8_t(k);
    // errors are recorded into the status word with compare-and-swap
    if (cudaMemsetAsync(d_status, 0, sizeof(int), stream) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    const int grid = grid_for(a.n_tiles, d.sms, d.encode_bpsm[dtype]);
    return launch_encode(a, lut, map, grid, stream) == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
}

}  // namespace

int splitzip_encode(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb, uint32_t chunk_elems,
                    void* d_out, uint64_t out_capacity, void* d_ws, uint64_t ws_bytes, uint64_t* d_out_size,
                    int* d_status, cudaStream_t stream) {
    return encode_call(d_in, n, dtype, cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes, d_out_size, d_status,
                       stream, false);
}

int splitzip_encode_device_codebook(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* d_cb,
                                    uint32_t chunk_elems, void* d_out, uint64_t out_capacity, void* d_ws,
                                    uint64_t ws_bytes, uint64_t* d_out_size, int* d_status, cudaStream_t stream) {
    return encode_call(d_in, n, dtype, d_cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes, d_out_size, d_status,
                       stream, true);
}

int splitzip_calibrate_device(const void* d_x, uint64_t n, int dtype, uint64_t* d_hist256,
                              splitzip_codebook_t* d_cb, cudaStream_t stream) {
    if (!d_cb) return SPLITZIP_ERR_INVALID_ARG;
    const int st = splitzip_exponent_histogram(d_x, n, dtype, d_hist256, stream);
    if (st != SPLITZIP_OK) return st;
    return launch_codebook(reinterpret_cast<const unsigned long long*>(d_hist256), dtype,
                           reinterpret_cast<uint8_t*>(d_cb), stream) == cudaSuccess
               ? SPLITZIP_OK
               : SPLITZIP_ERR_CUDA;
}

namespace {

int decode_call(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n, int dtype, int* d_status,
                cudaStream_t stream, const int32_t* pages, uint64_t pool_pages, uint32_t page_shift) {
    if (!valid_dtype(dtype) || !d_in || !aligned(d_in, 16) || !d_status || !aligned(d_status, 4))
        return SPLITZIP_ERR_INVALID_ARG;
    if (n > 0 && (!d_out || !aligned(d_out, 16))) return SPLITZIP_ERR_INVALID_ARG;
    if (n > kMaxElems) return SPLITZIP_ERR_UNSUPPORTED;
    if (in_bytes < kHeaderBytes) return SPLITZIP_ERR_CORRUPT;
    DeviceState d;
    int st = device_state(&d);
    if (st != SPLITZIP_OK) return st;
    if (!pages && n <= kSmallDecodeElems) {
        // a small tensor: a status clear and one CTA per 8,192 elements (batch.cu)
        const SmallDecodeItem item{d_in, in_bytes, d_out, n};
        const cudaError_t e = launch_small_decode(&item, 1, dtype, d_status, stream);
        if (e != cudaSuccess) cudaGetLastError();
        return e == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
    }
    if (cudaMemsetAsync(d_status, 0, sizeof(int), stream) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    DecodeArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.in_bytes = in_bytes;
    a.out = d_out;
    a.n = n;
    a.dtype = dtype;
    a.status = d_status;
    a.pages = pages;
    a.pool_pages = pool_pages;
    a.page_shift = page_shift;
    const int grid = grid_for((n + kMinChunk - 1) / kMinChunk, d.sms, d.decode_bpsm[dtype]);
    return launch_decode(a, grid, stream) == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
}

bool pow2(uint64_t x) { return x != 0 && (x & (x - 1)) == 0; }

uint32_t log2_of(uint64_t x) {
    uint32_t k = 0;
    while ((uint64_t(1) << k) < x) ++k;
    return k;
}

}  // namespace

int splitzip_decode(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n, int dtype, int* d_status,
                    cudaStream_t stream) {
    return decode_call(d_in, in_bytes, d_out, n, dtype, d_status, stream, nullptr, 0, 0);
}

int splitzip_encode_paged(const void* d_pool, uint64_t pool_pages, const int32_t* d_pages, uint64_t n_pages,
                          uint64_t page_elems, int dtype, const splitzip_codebook_t* cb, uint32_t chunk_elems,
                          void* d_out, uint64_t out_capacity, void* d_ws, uint64_t ws_bytes, uint64_t* d_out_size,
                          int* d_status, cudaStream_t stream) {
    if (!valid_dtype(dtype) || !valid_chunk(chunk_elems)) return SPLITZIP_ERR_INVALID_ARG;
    if (!d_pages || !aligned(d_pages, 4) || n_pages == 0 || pool_pages == 0 || !pow2(page_elems) ||
        page_elems % tile_elems_for(dtype, chunk_elems) != 0)
        return SPLITZIP_ERR_INVALID_ARG;
    if (n_pages > kMaxElems / page_elems || pool_pages > kMaxElems / page_elems) return SPLITZIP_ERR_UNSUPPORTED;
    PagedInput paged;
    paged.pages = d_pages;
    paged.pool_pages = pool_pages;
    paged.page_elems = page_elems;
    return encode_call(d_pool, n_pages * page_elems, dtype, cb, chunk_elems, d_out, out_capacity, d_ws, ws_bytes,
                       d_out_size, d_status, stream, false, paged);
}

int splitzip_decode_paged(const void* d_in, uint64_t in_bytes, void* d_pool, uint64_t pool_pages,
                          const int32_t* d_pages, uint64_t n_pages, uint64_t page_elems, int dtype, int* d_status,
                          cudaStream_t stream) {
    if (!valid_dtype(dtype) || !d_pages || !aligned(d_pages, 4) || n_pages == 0 || pool_pages == 0 ||
        !pow2(page_elems) || page_elems < 16)
        return SPLITZIP_ERR_INVALID_ARG;
    if (n_pages > kMaxElems / page_elems || pool_pages > kMaxElems / page_elems) return SPLITZIP_ERR_UNSUPPORTED;
    return decode_call(d_in, in_bytes, d_pool, n_pages * page_elems, dtype, d_status, stream, d_pages, pool_pages,
                       log2_of(page_elems));
}

int splitzip_encode_batch_workspace_size(const uint64_t* h_n, uint32_t count, int dtype, uint32_t chunk_elems,
                                         uint64_t* out_bytes) {
    if (!h_n || !out_bytes || count == 0 || count > SPLITZIP_MAX_BATCH) return SPLITZIP_ERR_INVALID_ARG;
    uint64_t total = 0;
    for (uint32_t i = 0; i < count; ++i) {
        const int st = check_geometry(h_n[i], dtype, chunk_elems);
        if (st != SPLITZIP_OK) return st;
        if (h_n[i] > SPLITZIP_MAX_BATCH_ITEM_ELEMS) return SPLITZIP_ERR_UNSUPPORTED;
        total += (workspace_for(h_n[i], dtype, chunk_elems).bytes + 255u) & ~uint64_t(255);
    }
    *out_bytes = total;
    return SPLITZIP_OK;
}

int splitzip_encode_batch(const splitzip_encode_item_t* h_items, uint32_t count, int dtype,
                          const splitzip_codebook_t* cb, uint32_t chunk_elems, void* d_ws, uint64_t ws_bytes,
                          int* d_status, cudaStream_t stream) {
    if (!h_items || count == 0 || count > SPLITZIP_MAX_BATCH) return SPLITZIP_ERR_INVALID_ARG;
    if (!valid_dtype(dtype) || !valid_chunk(chunk_elems)) return SPLITZIP_ERR_INVALID_ARG;
    int st = check_codebook(cb, dtype);
    if (st != SPLITZIP_OK) return st;
    if (!d_status || !aligned(d_status, 4)) return SPLITZIP_ERR_INVALID_ARG;
    SmallEncodeItem items[SPLITZIP_MAX_BATCH];
    uint64_t ws_off = 0;
    for (uint32_t i = 0; i < count; ++i) {
        const splitzip_encode_item_t& it = h_items[i];
        if ((st = check_geometry(it.n, dtype, chunk_elems)) != SPLITZIP_OK) return st;
        if (it.n > SPLITZIP_MAX_BATCH_ITEM_ELEMS) return SPLITZIP_ERR_UNSUPPORTED;
        if (it.n > 0 && (!it.d_in || !aligned(it.d_in, 16))) return SPLITZIP_ERR_INVALID_ARG;
        if (!it.d_out || !aligned(it.d_out, 16) || !it.d_out_size || !aligned(it.d_out_size, 8))
            return SPLITZIP_ERR_INVALID_ARG;
        if (it.out_capacity < layout_for(it.n, dtype, chunk_elems, it.n).size) return SPLITZIP_ERR_CAPACITY;
        items[i] = SmallEncodeItem{it.d_in, it.n, it.d_out, it.d_out_size, static_cast<uint8_t*>(d_ws) + ws_off};
        ws_off += (workspace_for(it.n, dtype, chunk_elems).bytes + 255u) & ~uint64_t(255);
    }
    if (ws_bytes < ws_off) return SPLITZIP_ERR_CAPACITY;
    if (ws_off > 0 && (!d_ws || !aligned(d_ws, 16))) return SPLITZIP_ERR_INVALID_ARG;
    DeviceState d;
    if ((st = device_state(&d)) != SPLITZIP_OK) return st;
    return launch_small_encode(items, count, dtype, cb->exps, nullptr, chunk_elems, d_status, stream) == cudaSuccess
               ? SPLITZIP_OK
               : SPLITZIP_ERR_CUDA;
}

int splitzip_decode_batch(const splitzip_decode_item_t* h_items, uint32_t count, int dtype, int* d_status,
                          cudaStream_t stream) {
    if (!h_items || count == 0 || count > SPLITZIP_MAX_BATCH || !valid_dtype(dtype)) return SPLITZIP_ERR_INVALID_ARG;
    if (!d_status || !aligned(d_status, 4)) return SPLITZIP_ERR_INVALID_ARG;
    SmallDecodeItem items[SPLITZIP_MAX_BATCH];
    for (uint32_t i = 0; i < count; ++i) {
        const splitzip_decode_item_t& it = h_items[i];
        if (!it.d_in || !aligned(it.d_in, 16)) return SPLITZIP_ERR_INVALID_ARG;
        if (it.n > 0 && (!it.d_out || !aligned(it.d_out, 16))) return SPLITZIP_ERR_INVALID_ARG;
        if (it.n > SPLITZIP_MAX_BATCH_ITEM_ELEMS) return SPLITZIP_ERR_UNSUPPORTED;
        if (it.in_bytes < kHeaderBytes) return SPLITZIP_ERR_CORRUPT;
        items[i] = SmallDecodeItem{it.d_in, it.in_bytes, it.d_out, it.n};
    }
    DeviceState d;
    const int st = device_state(&d);
    if (st != SPLITZIP_OK) return st;
    return launch_small_decode(items, count, dtype, d_status, stream) == cudaSuccess ? SPLITZIP_OK
                                                                                     : SPLITZIP_ERR_CUDA;
}

int splitzip_parse_header(const void* h_blob, uint64_t bytes, splitzip_header_t* out) {
    if (!h_blob || !out) return SPLITZIP_ERR_INVALID_ARG;
    if (bytes < kHeaderBytes) return SPLITZIP_ERR_CORRUPT;
    const uint8_t* b = static_cast<const uint8_t*>(h_blob);
    auto u16 = [&](int o) { return uint16_t(b[o] | (b[o + 1] << 8)); };
    auto u32 = [&](int o) {
        uint32_t v = 0;
        for (int i = 3; i >= 0; --i) v = (v << 8) | b[o + i];
        return v;
    };
    auto u64 = [&](int o) { return uint64_t(u32(o)) | (uint64_t(u32(o + 4)) << 32); };
    if (u32(0) != kMagic || u16(4) != kVersion || !valid_dtype(b[6]) || b[7] != 0) return SPLITZIP_ERR_CORRUPT;
    for (int i = 48; i < 64; ++i)
        if (b[i] != 0) return SPLITZIP_ERR_CORRUPT;
    splitzip_header_t h;
    h.dtype = b[6];
    h.n_elems = u64(8);
    h.chunk_elems = u32(16);
    h.n_chunks = u32(20);
    h.total_escapes = u64(24);
    std::memcpy(h.codebook, b + 32, 16);
    if (!valid_chunk(h.chunk_elems) || h.n_elems > kMaxElems) return SPLITZIP_ERR_CORRUPT;
    if ((h.n_elems + h.chunk_elems - 1u) / h.chunk_elems != h.n_chunks) return SPLITZIP_ERR_CORRUPT;
    if (h.total_escapes > h.n_elems) return SPLITZIP_ERR_CORRUPT;
    splitzip_codebook_t cb;
    cb.dtype = h.dtype;
    std::memcpy(cb.exps, h.codebook, 16);
    if (check_codebook(&cb, h.dtype) != SPLITZIP_OK) return SPLITZIP_ERR_CORRUPT;
    const Layout L = layout_for(h.n_elems, h.dtype, h.chunk_elems, h.total_escapes);
    if (L.size > bytes) return SPLITZIP_ERR_CORRUPT;
    h.size = L.size;
    h.index_off = L.index_off;
    h.counts_off = L.counts_off;
    h.nibble_off = L.nibble_off;
    h.signmant_off = L.signmant_off;
    h.escrec_off = L.escrec_off;
    *out = h;
    return SPLITZIP_OK;
}

}  // extern "C"
