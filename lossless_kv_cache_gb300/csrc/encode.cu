// SplitZip encode kernels for sm_103a.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Encoding strategy".  Three kernels:
//
//   encode_streams_kernel  the dense pass over the input (HBM-bound): per
//       element split sign|mantissa from the exponent, map the exponent
//       through the Top-16 table to a 4-bit code, pack two codes per byte,
//       and detect escapes.  Each tile's escapes are ordered by a block scan
//       and written to the tile's own staging slot in the workspace together
//       with the tile's escape count.  No atomics, no inter-block waits.
//   encode_index_kernel    one CTA: per-chunk counts (sum of the chunk's tile
//       counts), their exclusive prefix (the container index), E, the size,
//       the status word and all section padding.
//   encode_gather_kernel   one warp per tile: copies the staged records of
//       the tile to their final place in the position and exponent arrays.
//
// The escape order inside a chunk is ascending position because tiles are
// chunk-aligned, tiles of a chunk are laid out in order, and inside a tile the
// block scan orders records by element index.
#include <type_traits>

#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kWarps = kEncodeThreads / 32;

// Units: BF16 8 elements (one 16-byte load), E5M2 16 elements.  Each thread
// handles kUnitsPerThread units per tile, unit u = j * 256 + threadIdx.x, so
// every warp-wide load covers 512 contiguous bytes.
template <int DT> struct Geometry;
template <> struct Geometry<SPLITZIP_BF16> {
    static constexpr int kElemBytes = 2, kUnitElems = 8, kUnitsPerThread = 4;
};
template <> struct Geometry<SPLITZIP_FP8_E5M2> {
    static constexpr int kElemBytes = 1, kUnitElems = 16, kUnitsPerThread = 2;
};
static_assert(kEncodeThreads * 8 * 4 == kTileElems, "BF16 tile");
static_assert(kEncodeThreads * 16 * 2 == kTileElems, "E5M2 tile");

// Load `nbytes` (< 16) bytes into a zero-filled vector (only the final unit
// of a tensor is partial).
__device__ __forceinline__ uint4 load_partial(const uint8_t* p, int nbytes) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i < nbytes) w[i >> 2] |= uint32_t(p[i]) << (8 * (i & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Four table entries (code | escape flag) for the four exponent bytes of `e`.
__device__ __forceinline__ uint32_t lookup4(const uint8_t* lut, uint32_t e) {
    return uint32_t(lut[e & 0xFFu]) | (uint32_t(lut[(e >> 8) & 0xFFu]) << 8) |
           (uint32_t(lut[(e >> 16) & 0xFFu]) << 16) | (uint32_t(lut[e >> 24]) << 24);
}

// Escape flags of four table entries -> 4-bit mask (bit k = byte k).
__device__ __forceinline__ uint32_t escape_bits4(uint32_t t) {
    const uint32_t f = (t >> 4) & 0x01010101u;
    return (f * 0x01020408u) >> 24;
}

// Two words of four codes each (low nibble of every byte) -> the 8 codes
// packed two per byte, even element in the low nibble.
__device__ __forceinline__ uint32_t pack_nibbles8(uint32_t t0, uint32_t t1) {
    const uint32_t k0 = t0 & 0x0F0F0F0Fu, k1 = t1 & 0x0F0F0F0Fu;
    return __byte_perm(k0 | (k0 >> 4), k1 | (k1 >> 4), 0x6420);
}

// One BF16 unit: 8 elements in v -> 8 nibbles, 8 sign|mantissa bytes, the
// escape mask and the 8 exponents (kept for the escape records).
__device__ __forceinline__ void encode_unit_bf16(const uint4 v, const uint8_t* lut, uint32_t& nib,
                                                 uint2& sm, uint32_t& esc, uint32_t& e0, uint32_t& e1) {
    const uint32_t lo0 = __byte_perm(v.x, v.y, 0x6420);  // low bytes of elements 0..3
    const uint32_t hi0 = __byte_perm(v.x, v.y, 0x7531);  // high bytes of elements 0..3
    const uint32_t lo1 = __byte_perm(v.z, v.w, 0x6420);
    const uint32_t hi1 = __byte_perm(v.z, v.w, 0x7531);
    // sign (bit 7 of the high byte) | mantissa (bits 6..0 of the low byte)
    sm.x = (hi0 & 0x80808080u) | (lo0 & 0x7F7F7F7Fu);
    sm.y = (hi1 & 0x80808080u) | (lo1 & 0x7F7F7F7Fu);
    // exponent = high byte bits 6..0 then low byte bit 7
    e0 = ((hi0 << 1) & 0xFEFEFEFEu) | ((lo0 >> 7) & 0x01010101u);
    e1 = ((hi1 << 1) & 0xFEFEFEFEu) | ((lo1 >> 7) & 0x01010101u);
    const uint32_t t0 = lookup4(lut, e0), t1 = lookup4(lut, e1);
    esc = escape_bits4(t0) | (escape_bits4(t1) << 4);
    nib = pack_nibbles8(t0, t1);
}

// Four E5M2 bytes -> their 3-bit sign|mantissa values packed LSB-first into
// 12 bits: s3 = (sign << 2) | mantissa2.
__device__ __forceinline__ uint32_t pack_s3x4(uint32_t w) {
    const uint32_t s = ((w >> 5) & 0x04040404u) | (w & 0x03030303u);
    const uint32_t x = s | (s >> 5);            // byte0: s0 | s1<<3, byte2: s2 | s3<<3
    return (x & 0x3Fu) | ((x >> 10) & 0xFC0u);  // 12 bits
}

// One E5M2 unit: 16 elements -> 16 nibbles (uint2), 6 bytes of s3 (lo32 +
// hi16), the escape mask and the exponents.
__device__ __forceinline__ void encode_unit_e5m2(const uint4 v, const uint8_t* lut, uint2& nib,
                                                 uint32_t& s3lo, uint32_t& s3hi, uint32_t& esc,
                                                 uint32_t (&e)[4]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        e[i] = (w[i] >> 2) & 0x1F1F1F1Fu;
        t[i] = lookup4(lut, e[i]);
    }
    esc = escape_bits4(t[0]) | (escape_bits4(t[1]) << 4) | (escape_bits4(t[2]) << 8) |
          (escape_bits4(t[3]) << 12);
    nib.x = pack_nibbles8(t[0], t[1]);
    nib.y = pack_nibbles8(t[2], t[3]);
    const uint32_t g0 = pack_s3x4(w[0]), g1 = pack_s3x4(w[1]), g2 = pack_s3x4(w[2]), g3 = pack_s3x4(w[3]);
    s3lo = g0 | (g1 << 12) | (g2 << 24);
    s3hi = (g2 >> 8) | (g3 << 4);
}

__device__ __forceinline__ void write_header(const EncodeArgs& a) {
    uint8_t* h = a.out;
    uint32_t* h32 = reinterpret_cast<uint32_t*>(h);
    h32[0] = kMagic;
    h32[1] = uint32_t(kVersion) | (uint32_t(a.dtype) << 16);  // version, dtype, reserved 0
    reinterpret_cast<uint64_t*>(h)[1] = a.n;
    h32[4] = a.chunk_elems;
    h32[5] = uint32_t(a.n_chunks);
    // h[24..31] (E) is written by the index kernel
    uint32_t cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        cb[i] = uint32_t(a.codebook[4 * i]) | (uint32_t(a.codebook[4 * i + 1]) << 8) |
                (uint32_t(a.codebook[4 * i + 2]) << 16) | (uint32_t(a.codebook[4 * i + 3]) << 24);
    reinterpret_cast<uint4*>(h)[2] = make_uint4(cb[0], cb[1], cb[2], cb[3]);
    reinterpret_cast<uint4*>(h)[3] = make_uint4(0u, 0u, 0u, 0u);
}

// Per-thread escape counts (<= 16 each) are scanned as 16-bit fields, two per
// word; a tile holds at most 8192 escapes so no field overflows.
template <int J>
struct PackedCounts {
    static constexpr int kWords = (J + 1) / 2;
    uint32_t w[kWords];
};

template <int DT>
__global__ void __launch_bounds__(kEncodeThreads)
encode_streams_kernel(const EncodeArgs a, const EncodeLut lut_in) {
    using G = Geometry<DT>;
    constexpr int J = G::kUnitsPerThread;
    constexpr int kWords = PackedCounts<J>::kWords;
    __shared__ uint8_t lut[256];
    __shared__ uint32_t warp_sums[2][kWarps][kWords];
    __shared__ __align__(16) uint8_t s3_stage[kWarps][192];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256; i += kEncodeThreads) lut[i] = lut_in.code[i];
    if (blockIdx.x == 0 && tid == 0) write_header(a);
    __syncthreads();

    const uint8_t* in = static_cast<const uint8_t*>(a.in);
    int parity = 0;
    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, parity ^= 1) {
        const uint64_t base = tile * a.tile_elems;  // first element of the tile
        const uint64_t rem = a.n - base;
        const uint32_t len_rt = rem < a.tile_elems ? uint32_t(rem) : a.tile_elems;
        const uint32_t pos0 = uint32_t(base & (a.chunk_elems - 1u));  // in-chunk position of element 0
        // Full 8192-element tiles (all but the last one) take a copy of the
        // body in which every bounds test folds away at compile time.
        auto body = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const uint32_t len = FULL ? kTileElems : len_rt;

            uint4 v[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t e = (uint32_t(j) * kEncodeThreads + tid) * G::kUnitElems;
                const uint8_t* p = in + (base + e) * G::kElemBytes;
                if (e + G::kUnitElems <= len)
                    v[j] = __ldcs(reinterpret_cast<const uint4*>(p));
                else if (e < len)
                    v[j] = load_partial(p, int(len - e) * G::kElemBytes);
                else
                    v[j] = make_uint4(0u, 0u, 0u, 0u);
            }

            uint32_t esc[J];
            uint32_t ex[J][4];  // exponents of each unit (BF16 uses [0..1])
#pragma unroll
            for (int j = 0; j < J; ++j) ex[j][2] = ex[j][3] = 0u;
            PackedCounts<J> cnt;
#pragma unroll
            for (int k = 0; k < kWords; ++k) cnt.w[k] = 0;

#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t e = (uint32_t(j) * kEncodeThreads + tid) * G::kUnitElems;
                const uint32_t valid = e < len ? min(len - e, uint32_t(G::kUnitElems)) : 0u;
                if constexpr (DT == SPLITZIP_BF16) {
                    uint32_t nib;
                    uint2 sm;
                    encode_unit_bf16(v[j], lut, nib, sm, esc[j], ex[j][0], ex[j][1]);
                    uint8_t* nb = a.nibbles + (base + e) / 2;
                    uint8_t* sb = a.signmant + (base + e);
                    if (valid == 8u) {
                        __stcs(reinterpret_cast<uint32_t*>(nb), nib);
                        __stcs(reinterpret_cast<uint2*>(sb), sm);
                    } else if (valid > 0u) {
                        esc[j] &= (1u << valid) - 1u;
                        nib &= (1u << (4u * valid)) - 1u;
                        for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nb[b] = uint8_t(nib >> (8u * b));
                        const uint64_t smw = uint64_t(sm.x) | (uint64_t(sm.y) << 32);
                        for (uint32_t b = 0; b < valid; ++b) sb[b] = uint8_t(smw >> (8u * b));
                    } else {
                        esc[j] = 0u;
                    }
                } else {
                    uint2 nib;
                    uint32_t s3lo, s3hi;
                    encode_unit_e5m2(v[j], lut, nib, s3lo, s3hi, esc[j], ex[j]);
                    uint8_t* nb = a.nibbles + (base + e) / 2;
                    // s3 bytes of this unit start at 3 * (element index) / 8
                    uint8_t* sb = a.signmant + (base + e) / 8 * 3;
                    // fast path: the warp's 32 units are full and the tile is a
                    // multiple of 512 elements, so its 192 s3 bytes are 16-aligned
                    const uint32_t warp_e0 = (uint32_t(j) * kEncodeThreads + warp * 32u) * G::kUnitElems;
                    const bool warp_full = (FULL || a.tile_elems % 512u == 0u) && (warp_e0 + 512u <= len);
                    if (valid == 16u) {
                        __stcs(reinterpret_cast<uint2*>(nb), nib);
                    } else if (valid > 0u) {
                        esc[j] &= (1u << valid) - 1u;
                        uint64_t nw = uint64_t(nib.x) | (uint64_t(nib.y) << 32);
                        nw &= (uint64_t(1) << (4u * valid)) - 1u;
                        for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nb[b] = uint8_t(nw >> (8u * b));
                    } else {
                        esc[j] = 0u;
                    }
                    if (warp_full) {  // warp-uniform
                        uint16_t* st = reinterpret_cast<uint16_t*>(&s3_stage[warp][6 * lane]);
                        st[0] = uint16_t(s3lo);
                        st[1] = uint16_t(s3lo >> 16);
                        st[2] = uint16_t(s3hi);
                        __syncwarp();
                        if (lane < 12) {
                            const uint4 q = reinterpret_cast<const uint4*>(s3_stage[warp])[lane];
                            uint8_t* dst = a.signmant + (base + warp_e0) / 8 * 3 + 16 * lane;
                            __stcs(reinterpret_cast<uint4*>(dst), q);
                        }
                        __syncwarp();
                    } else if (valid > 0u) {
                        // 3 bytes per started group of 8 elements (pad bits are 0)
                        const uint32_t nbytes = 3u * ((valid + 7u) / 8u);
                        uint16_t* d16 = reinterpret_cast<uint16_t*>(sb);  // 6*unit is even
                        if (nbytes == 6u) {
                            d16[0] = uint16_t(s3lo);
                            d16[1] = uint16_t(s3lo >> 16);
                            d16[2] = uint16_t(s3hi);
                        } else {
                            d16[0] = uint16_t(s3lo);
                            sb[2] = uint8_t(s3lo >> 16);
                        }
                    }
                }
                const uint32_t c = __popc(esc[j]);
                cnt.w[j >> 1] |= c << (16 * (j & 1));
            }

            // ---- block-wide exclusive scan of the per-thread escape counts, in
            // element order (unit group j major, then thread) ----
            uint32_t incl[kWords];
#pragma unroll
            for (int k = 0; k < kWords; ++k) incl[k] = cnt.w[k];
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
                for (int k = 0; k < kWords; ++k) {
                    const uint32_t y = __shfl_up_sync(kFull, incl[k], d);
                    if (lane >= d) incl[k] += y;
                }
            }
            if (lane == 31) {
#pragma unroll
                for (int k = 0; k < kWords; ++k) warp_sums[parity][warp][k] = incl[k];
            }
            __syncthreads();
            uint32_t before[kWords], total[kWords];
#pragma unroll
            for (int k = 0; k < kWords; ++k) before[k] = total[k] = 0u;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
#pragma unroll
                for (int k = 0; k < kWords; ++k) {
                    const uint32_t s = warp_sums[parity][w][k];
                    if (w < warp) before[k] += s;
                    total[k] += s;
                }
            }

            uint32_t group_base = 0;  // escapes of the tile in unit groups < j
            uint32_t* slot = a.staging + tile * a.tile_elems;
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int k = j >> 1, sh = 16 * (j & 1);
                const uint32_t excl = ((before[k] + incl[k] - cnt.w[k]) >> sh) & 0xFFFFu;
                uint32_t idx = group_base + excl;
                uint32_t m = esc[j];
                const uint32_t upos = pos0 + (uint32_t(j) * kEncodeThreads + tid) * G::kUnitElems;
                while (m) {
                    const uint32_t b = __ffs(m) - 1;
                    m &= m - 1;
                    const uint32_t q = b >> 2;  // which exponent word (select, no local memory)
                    const uint32_t ew = q == 0 ? ex[j][0] : q == 1 ? ex[j][1] : q == 2 ? ex[j][2] : ex[j][3];
                    const uint32_t exponent = (ew >> (8u * (b & 3u))) & 0xFFu;
                    slot[idx++] = ((upos + b) << 8) | exponent;
                }
                group_base += (total[k] >> sh) & 0xFFFFu;
            }
            if (tid == 0) a.tile_counts[tile] = group_base;
        };
        if (len_rt == kTileElems)
            body(std::true_type{});
        else
            body(std::false_type{});
    }
}

// ---------------------------------------------------------------------------
// index: per-chunk counts, exclusive prefix, E, size, status, padding

__device__ __forceinline__ void zero_bytes(uint8_t* p, uint64_t from, uint64_t to) {
    for (uint64_t i = from; i < to; ++i) p[i] = 0;
}

__global__ void __launch_bounds__(kIndexThreads)
encode_index_kernel(const EncodeArgs a, uint64_t* out_size, int* status) {
    __shared__ uint64_t sums[kIndexThreads];
    const int tid = threadIdx.x;
    const uint64_t C = a.n_chunks;
    const uint32_t tpc = a.chunk_elems / a.tile_elems;
    const Layout L = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    uint32_t* counts = reinterpret_cast<uint32_t*>(a.out + L.counts_off);
    uint64_t* offsets = reinterpret_cast<uint64_t*>(a.out + L.index_off);

    // phase 1: chunk counts, coalesced over chunks
    for (uint64_t c = tid; c < C; c += kIndexThreads) {
        const uint64_t t0 = c * tpc;
        const uint64_t t1 = min(t0 + tpc, a.n_tiles);
        uint32_t s = 0;
        for (uint64_t t = t0; t < t1; ++t) s += a.tile_counts[t];
        counts[c] = s;
    }
    __syncthreads();
    // phase 2: each thread owns a contiguous range of chunks
    const uint64_t per = (C + kIndexThreads - 1) / kIndexThreads;
    const uint64_t c0 = min(C, uint64_t(tid) * per), c1 = min(C, c0 + per);
    uint64_t mine = 0;
    for (uint64_t c = c0; c < c1; ++c) mine += counts[c];
    sums[tid] = mine;
    __syncthreads();
    // Hillis-Steele inclusive scan over the block
    for (int d = 1; d < kIndexThreads; d <<= 1) {
        const uint64_t y = tid >= d ? sums[tid - d] : 0;
        __syncthreads();
        sums[tid] += y;
        __syncthreads();
    }
    uint64_t run = sums[tid] - mine;
    for (uint64_t c = c0; c < c1; ++c) {
        offsets[c] = run;
        run += counts[c];
    }
    if (tid == 0) {
        const uint64_t E = sums[kIndexThreads - 1];
        const Layout F = layout_for(a.n, a.dtype, a.chunk_elems, E);
        reinterpret_cast<uint64_t*>(a.out)[3] = E;
        zero_bytes(a.out, F.index_end, F.nibble_off);
        zero_bytes(a.out, F.nibble_off + (a.n + 1) / 2, F.signmant_off);
        zero_bytes(a.out, F.signmant_off + signmant_bytes(a.dtype, a.n), F.escpos_off);
        zero_bytes(a.out, F.escpos_off + 2 * E, F.escexp_off);
        *out_size = F.size;
        *status = SPLITZIP_OK;
    }
}

// ---------------------------------------------------------------------------
// gather: one warp per tile moves the staged records to the escape arrays

__global__ void __launch_bounds__(kGatherThreads) encode_gather_kernel(const EncodeArgs a) {
    const int lane = threadIdx.x & 31;
    const uint64_t warps = uint64_t(gridDim.x) * (kGatherThreads / 32);
    const uint64_t first_warp = uint64_t(blockIdx.x) * (kGatherThreads / 32) + (threadIdx.x >> 5);
    const uint64_t E = reinterpret_cast<const uint64_t*>(a.out)[3];
    const Layout L = layout_for(a.n, a.dtype, a.chunk_elems, E);
    const uint64_t* offsets = reinterpret_cast<const uint64_t*>(a.out + L.index_off);
    uint16_t* pos = reinterpret_cast<uint16_t*>(a.out + L.escpos_off);
    uint8_t* exps = a.out + L.escexp_off;
    const uint32_t tpc = a.chunk_elems / a.tile_elems;

    for (uint64_t tile = first_warp; tile < a.n_tiles; tile += warps) {
        const uint32_t cnt = a.tile_counts[tile];
        if (cnt == 0) continue;
        const uint64_t c = tile / tpc, first = c * tpc;
        // escapes of the earlier tiles of the same chunk (fewer than 32 tiles)
        const uint32_t earlier = uint32_t(tile - first);
        uint32_t s = (uint32_t(lane) < earlier) ? a.tile_counts[first + lane] : 0u;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(kFull, s, d);
        const uint64_t off = offsets[c] + s;
        const uint32_t* slot = a.staging + tile * a.tile_elems;
        for (uint32_t i = lane; i < cnt; i += 32) {
            const uint32_t r = slot[i];
            pos[off + i] = uint16_t(r >> 8);
            exps[off + i] = uint8_t(r & 0xFFu);
        }
    }
}

}  // namespace

cudaError_t launch_encode_streams(const EncodeArgs& a, const EncodeLut& lut, int grid, cudaStream_t s) {
    if (a.dtype == SPLITZIP_BF16)
        encode_streams_kernel<SPLITZIP_BF16><<<grid, kEncodeThreads, 0, s>>>(a, lut);
    else
        encode_streams_kernel<SPLITZIP_FP8_E5M2><<<grid, kEncodeThreads, 0, s>>>(a, lut);
    return cudaGetLastError();
}

cudaError_t launch_encode_escapes(const EncodeArgs& a, uint64_t* d_out_size, int* d_status, int grid,
                                  cudaStream_t s) {
    encode_index_kernel<<<1, kIndexThreads, 0, s>>>(a, d_out_size, d_status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.n_tiles == 0) return err;
    encode_gather_kernel<<<grid, kGatherThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t occupancy_encode(int* blocks_per_sm, int dtype) {
    if (dtype == SPLITZIP_BF16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                             encode_streams_kernel<SPLITZIP_BF16>,
                                                             kEncodeThreads, 0);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                         encode_streams_kernel<SPLITZIP_FP8_E5M2>,
                                                         kEncodeThreads, 0);
}

cudaError_t occupancy_gather(int* blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, encode_gather_kernel,
                                                         kGatherThreads, 0);
}

}  // namespace splitzip
