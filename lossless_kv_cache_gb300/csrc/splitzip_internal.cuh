// Internal definitions shared by the SplitZip GB300 kernels and the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (types only; the encoder of tensor maps is fetched from the runtime)
#include <cuda_runtime.h>

#include "splitzip.h"

namespace splitzip {

constexpr uint32_t kMagic = 0x50495A53u;  // "SZIP" little-endian
constexpr uint16_t kVersion = 1;
constexpr uint64_t kHeaderBytes = 64;
constexpr uint32_t kMinChunk = 64;
constexpr uint32_t kMaxChunk = 65536;

// Work decomposition of the encoder.  A tile is the unit of work of one
// encode CTA trip: 16 KB of input (8,192 BF16 / FP16 or 16,384 E5M2 elements), or the
// chunk when chunks are smaller, so a tile never straddles a chunk (chunk
// sizes are powers of two >= 64).  Each of the 256 consumer threads of a CTA
// owns 64 contiguous bytes of the tile.
constexpr uint32_t kTileBytes = 16384;
constexpr uint32_t kEncodeWarps = 8;
constexpr uint32_t kThreadBytes = 64;
constexpr int kHistThreads = 256;

// Encoder table entry: low 4 bits = code, bit 4 = escape flag.
constexpr uint8_t kEscapeFlag = 0x10;

__host__ __device__ inline uint64_t align16(uint64_t x) { return (x + 15u) & ~uint64_t(15); }

__host__ __device__ inline uint32_t elem_bytes(int dtype) { return dtype == SPLITZIP_FP8_E5M2 ? 1u : 2u; }

// Bytes of the sign|mantissa stream: BF16 one byte per element, E5M2 3 bits
// and FP16 11 bits per element, packed in groups of 8 elements.
__host__ __device__ inline uint64_t signmant_bytes(int dtype, uint64_t n) {
    if (dtype == SPLITZIP_BF16) return n;
    return (dtype == SPLITZIP_FP16 ? 11u : 3u) * ((n + 7u) / 8u);
}

// Byte offsets of every section of a container (format v1, see splitzip.h).
struct Layout {
    uint64_t n_chunks;
    uint64_t index_off, counts_off, index_end, nibble_off, signmant_off, escrec_off, size;
};

__host__ __device__ inline Layout layout_for(uint64_t n, int dtype, uint32_t chunk, uint64_t E) {
    Layout L;
    L.n_chunks = (n + chunk - 1u) / chunk;
    L.index_off = kHeaderBytes;
    L.counts_off = L.index_off + 8u * L.n_chunks;
    L.index_end = L.counts_off + 4u * L.n_chunks;
    L.nibble_off = align16(L.index_end);
    L.signmant_off = L.nibble_off + align16((n + 1u) / 2u);
    L.escrec_off = L.signmant_off + align16(signmant_bytes(dtype, n));
    L.size = L.escrec_off + 3u * E;
    return L;
}

__host__ __device__ inline uint32_t tile_elems_for(int dtype, uint32_t chunk) {
    const uint32_t full = kTileBytes / elem_bytes(dtype);
    return chunk < full ? chunk : full;
}

// Encoder workspace: per-group escape totals (a group is kGroupTiles
// consecutive tiles), per-(tile, consumer warp) escape counts, then one
// staging slot of tile_elems records per tile; a record is (in-chunk position
// << 8) | exponent.  Consumer warp w stages its records contiguously from slot
// element w * (2,048 bytes / element size) on (its region of the tile).
constexpr uint32_t kGroupTiles = 256;

struct Workspace {
    uint64_t n_tiles, n_groups;
    uint32_t tile_elems;
    uint64_t group_off, warp_count_off, tile_first_off, staging_off, bytes;
};

__host__ __device__ inline Workspace workspace_for(uint64_t n, int dtype, uint32_t chunk) {
    Workspace W;
    W.tile_elems = tile_elems_for(dtype, chunk);
    W.n_tiles = (n + W.tile_elems - 1u) / W.tile_elems;
    W.n_groups = (W.n_tiles + kGroupTiles - 1u) / kGroupTiles;
    W.group_off = 0;
    W.warp_count_off = align16(4u * W.n_groups);
    W.tile_first_off = align16(W.warp_count_off + 4u * kEncodeWarps * W.n_tiles);
    W.staging_off = align16(W.tile_first_off + 8u * W.n_tiles);
    W.bytes = W.staging_off + 4u * W.n_tiles * W.tile_elems;
    return W;
}

// First error of a call: the status word keeps the first code written after
// it was cleared.
__device__ __forceinline__ void report(int* status, int code) { atomicCAS(status, SPLITZIP_OK, code); }

struct EncodeLut {
    uint8_t code[256];  // exponent -> code | kEscapeFlag
};

struct EncodeArgs {
    const void* in;
    uint64_t n;
    uint8_t* out;            // container base
    uint32_t* group_totals;  // workspace, per group of kGroupTiles tiles
    uint32_t* warp_counts;   // workspace, per tile and consumer warp
    uint64_t* tile_first;    // workspace, per tile: index of its first record
    uint32_t* staging;       // workspace, tile_elems records per tile
    uint64_t* out_size;
    int* error;              // device status word
    uint64_t n_tiles, n_groups;
    uint32_t tile_elems;
    uint32_t chunk_elems;
    uint64_t n_chunks;
    // Input bytes the tensor map covers (whole 128-byte rows from the start;
    // 0 = no tensor map) and the bytes one tensor-map load delivers.
    uint64_t tensor_bytes;
    uint32_t box_bytes;
    // tensor bytes (from the start) whose tiles arrive through the tensor map:
    // tensor_bytes, or every byte with paged input
    uint64_t staged_bytes;
    int dtype;
    uint8_t codebook[16];
    // a splitzip_codebook_t in device memory (dtype byte, then the 16
    // exponents) that replaces codebook[] and the host-built table, or null
    const uint8_t* dev_codebook;
    // paged input (null: `in` is the tensor): `in` is a pool of pool_pages
    // pages of 2^page_tile_shift tiles each, and tile t of the tensor is tile
    // t mod 2^page_tile_shift of pool page pages[t >> page_tile_shift]
    const int32_t* pages;
    uint64_t pool_pages;
    uint32_t page_tile_shift;
};

struct DecodeArgs {
    const uint8_t* in;
    uint64_t in_bytes;
    void* out;
    uint64_t n;
    int dtype;
    int* status;
    // paged output (null: `out` is the tensor): `out` is a pool of pool_pages
    // pages of 2^page_shift elements, and element g goes to element
    // g mod 2^page_shift of pool page pages[g >> page_shift]
    const int32_t* pages;
    uint64_t pool_pages;
    uint32_t page_shift;
};

// Launchers (encode.cu, decode.cu, histogram.cu).  Each returns the result of
// cudaGetLastError() after its launch.
cudaError_t launch_encode(const EncodeArgs& a, const EncodeLut& lut, const CUtensorMap& map, int grid,
                          cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s);
// One CTA: the Top-16 codebook of a device histogram into a device
// splitzip_codebook_t (count descending, exponent ascending on ties).
cudaError_t launch_codebook(const unsigned long long* hist, int dtype, uint8_t* cb, cudaStream_t s);
cudaError_t launch_histogram(const void* x, uint64_t n, int dtype, unsigned long long* hist, int grid,
                             cudaStream_t s);

// Small tensors and batches (batch.cu): one item of a call.  An encode item's
// workspace has the splitzip_encode layout for its n.
constexpr uint32_t kMaxBatch = 256;
struct SmallEncodeItem {
    const void* in;
    uint64_t n;
    void* out;
    uint64_t* out_size;
    void* ws;
};
struct SmallDecodeItem {
    const void* in;
    uint64_t in_bytes;
    void* out;
    uint64_t n;
};
// Batch encode: two kernels (one CTA per tile of every item; one per chunk)
// chained with programmatic dependent launch; the status word is set by the
// call.  codebook: host codebook bytes, or dev_codebook (then codebook is
// unused).
cudaError_t launch_small_encode(const SmallEncodeItem* items, uint32_t count, int dtype, const uint8_t* codebook,
                                const uint8_t* dev_codebook, uint32_t chunk, int* status, cudaStream_t s);
// Batch decode: a status clear, then one CTA per 8,192 elements of every item.
cudaError_t launch_small_decode(const SmallDecodeItem* items, uint32_t count, int dtype, int* status,
                                cudaStream_t s);
// One small tensor encoded by one cooperative kernel (grid <= the co-resident
// CTAs that occupancy_coop gives; n > 0).
cudaError_t launch_coop_encode(const SmallEncodeItem& item, int dtype, const uint8_t* codebook,
                               const uint8_t* dev_codebook, uint32_t chunk, int* status, int grid, cudaStream_t s);
cudaError_t occupancy_coop(int* encode_blocks_per_sm, int dtype);

// Resident CTAs per SM of each kernel; the encode/decode versions also raise
// the kernels' dynamic shared-memory limit (call once per device).
cudaError_t occupancy_encode(int* blocks_per_sm, int dtype);
cudaError_t occupancy_decode(int* blocks_per_sm, int dtype);
cudaError_t occupancy_histogram(int* blocks_per_sm, int dtype);

}  // namespace splitzip
