// SplitZip encode kernels for sm_103a.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Encoding strategy": each element's
// exponent goes through the offline-calibrated Top-16 codebook to a 4-bit code,
// two codes per byte ("Fixed-length coding"); sign and mantissa are kept raw
// ("Sign/mantissa preservation"); an exponent outside the codebook becomes a
// (16-bit position, 8-bit exponent) escape record ("Escape stream").
//
// Two kernels, no inter-block waits:
//   encode_kernel (the streaming pass, persistent CTAs of 8 consumer warps +
//     1 producer warp): the producer streams each of the CTA's tiles into a
//     4-stage shared-memory ring with bulk copies (TMA, cp.async.bulk +
//     mbarrier); consumers split, code and pack the tile from shared memory
//     and write the nibble and sign|mantissa streams with coalesced stores; a
//     block scan orders the tile's escapes by element index and writes them
//     to the tile's staging slot; the tile's count goes to the workspace and,
//     by an integer atomic add, to its group's total.
//   encode_index_kernel (one CTA per group of 256 tiles): the sum of the
//     earlier groups' totals plus a block scan of the group's tile counts give
//     every tile's first record index; the CTA writes them and the index
//     entries of the group's chunks; the last group writes E and the size.
//   encode_records_kernel (a warp per 4 tiles): moves every tile's staged
//     records to their place in the escape stream.
#include <type_traits>

#include "splitzip_internal.cuh"
#include "tma_pipeline.cuh"

namespace splitzip {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kBlock = kConsumers + 32;  // + one producer warp
constexpr int kStages = 4;
constexpr uint32_t kStageBytes = kTileElems * 2;  // one BF16 tile
constexpr uint32_t kEncodeSmem = kStages * kStageBytes;
constexpr int kFinishThreads = kGroupTiles;  // one thread per tile of the group

// Units: BF16 8 elements, E5M2 16 elements (16 bytes either way).  Thread t
// handles units j * 256 + t of a tile, so each warp reads 512 contiguous bytes.
template <int DT> struct Geometry;
template <> struct Geometry<SPLITZIP_BF16> {
    static constexpr int kElemBytes = 2, kUnitElems = 8, kUnitsPerThread = 4;
};
template <> struct Geometry<SPLITZIP_FP8_E5M2> {
    static constexpr int kElemBytes = 1, kUnitElems = 16, kUnitsPerThread = 2;
};
static_assert(kConsumers * 8 * 4 == kTileElems, "BF16 tile");
static_assert(kConsumers * 16 * 2 == kTileElems, "E5M2 tile");

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

// Header fields known before any tile is encoded (E is written at the end),
// and the zero padding between sections, whose places depend only on n.
__device__ void write_header_and_padding(const EncodeArgs& a) {
    uint8_t* h = a.out;
    uint32_t* h32 = reinterpret_cast<uint32_t*>(h);
    h32[0] = kMagic;
    h32[1] = uint32_t(kVersion) | (uint32_t(a.dtype) << 16);  // version, dtype, reserved 0
    reinterpret_cast<uint64_t*>(h)[1] = a.n;
    h32[4] = a.chunk_elems;
    h32[5] = uint32_t(a.n_chunks);
    uint32_t cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        cb[i] = uint32_t(a.codebook[4 * i]) | (uint32_t(a.codebook[4 * i + 1]) << 8) |
                (uint32_t(a.codebook[4 * i + 2]) << 16) | (uint32_t(a.codebook[4 * i + 3]) << 24);
    reinterpret_cast<uint4*>(h)[2] = make_uint4(cb[0], cb[1], cb[2], cb[3]);
    reinterpret_cast<uint4*>(h)[3] = make_uint4(0u, 0u, 0u, 0u);
    const Layout L = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    for (uint64_t i = L.index_end; i < L.nibble_off; ++i) h[i] = 0;
    for (uint64_t i = L.nibble_off + (a.n + 1) / 2; i < L.signmant_off; ++i) h[i] = 0;
    for (uint64_t i = L.signmant_off + signmant_bytes(a.dtype, a.n); i < L.escrec_off; ++i) h[i] = 0;
    if (a.n_tiles == 0) {  // no tile will finish the header
        reinterpret_cast<uint64_t*>(h)[3] = 0;
        *a.out_size = L.size;
    }
}

__device__ __forceinline__ void report(int* status, int code) { atomicCAS(status, SPLITZIP_OK, code); }

template <int DT>
__global__ void __launch_bounds__(kBlock, 3) encode_kernel(const EncodeArgs a, const EncodeLut lut_in) {
    using G = Geometry<DT>;
    constexpr int J = G::kUnitsPerThread;
    constexpr int kWords = (J + 1) / 2;  // per-thread counts as 16-bit fields, two per word
    extern __shared__ __align__(128) uint8_t stages[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ uint8_t lut[256];
    __shared__ uint32_t warp_sums[2][kConsumerWarps][kWords];
    __shared__ __align__(16) uint8_t s3_stage[kConsumerWarps][192];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 256; i += kBlock) lut[i] = lut_in.code[i];
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumerWarps);
        }
        mbar_init_fence();
        if (blockIdx.x == 0) write_header_and_padding(a);
    }
    __syncthreads();

    const uint8_t* in = static_cast<const uint8_t*>(a.in);
    if (warp == kConsumerWarps) {
        // ---- producer: stream the CTA's tiles (blockIdx.x + k * gridDim.x) ----
        if (lane != 0) return;
        uint32_t it = 0;
        for (uint64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++it) {
            const uint32_t stage = it % kStages, use = it / kStages;
            if (use > 0 && !mbar_wait(&empty_bar[stage], (use - 1) & 1u)) report(a.error, SPLITZIP_ERR_TIMEOUT);
            const uint64_t base = t * a.tile_elems;
            const uint64_t len = min(uint64_t(a.tile_elems), a.n - base);
            // whole 16-byte units only: the input has no padding after element n-1
            const uint32_t bytes = uint32_t(len * G::kElemBytes) & ~15u;
            mbar_arrive_expect_tx(&full_bar[stage], bytes);
            if (bytes) bulk_load(stages + stage * kStageBytes, in + base * G::kElemBytes, bytes, &full_bar[stage]);
        }
        if (!drain_stages(full_bar, kStages, it)) report(a.error, SPLITZIP_ERR_TIMEOUT);
        return;
    }

    // ---- consumers ----
    const Layout L0 = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    uint8_t* nibbles = a.out + L0.nibble_off;
    uint8_t* signmant = a.out + L0.signmant_off;

    uint32_t it = 0;
    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++it) {
        const uint32_t stage = it % kStages, use = it / kStages, parity = it & 1u;
        // on a time-out the tile is processed anyway (its addresses do not
        // depend on the data), so every consumer still meets every barrier
        if (!mbar_wait(&full_bar[stage], use & 1u)) report(a.error, SPLITZIP_ERR_TIMEOUT);
        const uint64_t base = tile * a.tile_elems;
        const uint64_t rem = a.n - base;
        const uint32_t len_rt = rem < a.tile_elems ? uint32_t(rem) : a.tile_elems;
        const uint32_t pos0 = uint32_t(base & (a.chunk_elems - 1u));  // in-chunk position of element 0
        const uint8_t* tile_smem = stages + stage * kStageBytes;

        // Full 8192-element tiles take a copy of the body in which every
        // bounds test folds away at compile time.
        auto body = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const uint32_t len = FULL ? kTileElems : len_rt;

            uint4 v[J];
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t e = (uint32_t(j) * kConsumers + tid) * G::kUnitElems;
                if (e + G::kUnitElems <= len)
                    v[j] = *reinterpret_cast<const uint4*>(tile_smem + e * G::kElemBytes);
                else if (e < len)  // the tensor's final bytes were not bulk-copied
                    v[j] = load_partial(in + (base + e) * G::kElemBytes, int(len - e) * G::kElemBytes);
                else
                    v[j] = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);  // the stage may be refilled

            uint32_t esc[J];
            uint32_t ex[J][4];  // exponents of each unit (BF16 uses [0..1])
            uint32_t cnt[kWords];
#pragma unroll
            for (int j = 0; j < J; ++j) ex[j][2] = ex[j][3] = 0u;
#pragma unroll
            for (int k = 0; k < kWords; ++k) cnt[k] = 0;

#pragma unroll
            for (int j = 0; j < J; ++j) {
                const uint32_t e = (uint32_t(j) * kConsumers + tid) * G::kUnitElems;
                const uint32_t valid = e < len ? min(len - e, uint32_t(G::kUnitElems)) : 0u;
                if constexpr (DT == SPLITZIP_BF16) {
                    uint32_t nib;
                    uint2 sm;
                    encode_unit_bf16(v[j], lut, nib, sm, esc[j], ex[j][0], ex[j][1]);
                    uint8_t* nb = nibbles + (base + e) / 2;
                    uint8_t* sb = signmant + (base + e);
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
                    uint8_t* nb = nibbles + (base + e) / 2;
                    uint8_t* sb = signmant + (base + e) / 8 * 3;  // 6 s3 bytes per unit
                    // fast path: the warp's 32 units are full and the tile is a
                    // multiple of 512 elements, so its 192 s3 bytes are 16-aligned
                    const uint32_t warp_e0 = (uint32_t(j) * kConsumers + warp * 32u) * G::kUnitElems;
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
                            uint8_t* dst = signmant + (base + warp_e0) / 8 * 3 + 16 * lane;
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
                cnt[j >> 1] |= uint32_t(__popc(esc[j])) << (16 * (j & 1));
            }

            // ---- block-wide exclusive scan of the per-thread escape counts,
            // in element order (unit group j major, then thread) ----
            uint32_t incl[kWords];
#pragma unroll
            for (int k = 0; k < kWords; ++k) incl[k] = cnt[k];
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
            named_barrier(1, kConsumers);
            uint32_t before[kWords], total[kWords];
#pragma unroll
            for (int k = 0; k < kWords; ++k) before[k] = total[k] = 0u;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
#pragma unroll
                for (int k = 0; k < kWords; ++k) {
                    const uint32_t s = warp_sums[parity][w][k];
                    if (w < warp) before[k] += s;
                    total[k] += s;
                }
            }
            uint32_t tile_total = 0;
#pragma unroll
            for (int j = 0; j < J; ++j) tile_total += (total[j >> 1] >> (16 * (j & 1))) & 0xFFFFu;

            if (tid == 0) {
                a.tile_counts[tile] = tile_total;
                if (tile_total) atomicAdd(a.group_totals + tile / kGroupTiles, tile_total);
            }

            // ---- escape records, in element order, to the tile's staging slot ----
            uint32_t* slot = a.staging + tile * a.tile_elems;
            uint32_t group_base = 0;  // escapes of the tile in unit groups < j
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int k = j >> 1, sh = 16 * (j & 1);
                const uint32_t excl = ((before[k] + incl[k] - cnt[k]) >> sh) & 0xFFFFu;
                uint32_t idx = group_base + excl;
                uint32_t m = esc[j];
                const uint32_t upos = pos0 + (uint32_t(j) * kConsumers + tid) * G::kUnitElems;
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
        };
        if (len_rt == kTileElems)
            body(std::true_type{});
        else
            body(std::false_type{});
    }
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

// One CTA per group of kGroupTiles tiles (groups are chunk-aligned: tiles per
// chunk is a power of two <= 8): the first record index of every tile of the
// group, the index entries of the group's chunks, and E from the last group.
__global__ void __launch_bounds__(kFinishThreads) encode_index_kernel(const EncodeArgs a) {
    constexpr int kWarps = kFinishThreads / 32;
    __shared__ uint64_t warp_part[kWarps];
    __shared__ uint32_t warp_incl[kWarps];
    __shared__ uint32_t tile_off[kFinishThreads + 1];  // exclusive prefix of the group's tile counts
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t g = blockIdx.x;

    // records of all earlier groups
    uint64_t before = 0;
    for (uint64_t q = tid; q < g; q += kFinishThreads) before += a.group_totals[q];
    before = warp_sum_u64(before);
    if (lane == 0) warp_part[warp] = before;

    // exclusive scan of the group's tile counts
    const uint64_t t = g * kGroupTiles + tid;
    const uint32_t c = t < a.n_tiles ? a.tile_counts[t] : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) warp_incl[warp] = incl;
    __syncthreads();
    uint64_t group_base = 0;
    uint32_t warp_before = 0, group_total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        group_base += warp_part[w];
        if (w < warp) warp_before += warp_incl[w];
        group_total += warp_incl[w];
    }
    tile_off[tid] = warp_before + incl - c;
    if (tid == 0) tile_off[kFinishThreads] = group_total;
    __syncthreads();
    if (t < a.n_tiles) a.tile_first[t] = group_base + tile_off[tid];

    // index entries of the chunks that start in this group
    const Layout L0 = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    const uint32_t tpc = a.chunk_elems / a.tile_elems;
    if (t < a.n_tiles && t % tpc == 0) {
        const uint64_t chunk = t / tpc;
        reinterpret_cast<uint64_t*>(a.out + L0.index_off)[chunk] = group_base + tile_off[tid];
        reinterpret_cast<uint32_t*>(a.out + L0.counts_off)[chunk] = tile_off[tid + tpc] - tile_off[tid];
    }
    if (g + 1 == a.n_groups && tid == 0) {  // the last group knows E
        const uint64_t E = group_base + group_total;
        reinterpret_cast<uint64_t*>(a.out)[3] = E;
        *a.out_size = layout_for(a.n, a.dtype, a.chunk_elems, E).size;
    }
}

// Staged records -> 3-byte records in the escape stream.  Each warp serves
// kRecordTiles consecutive tiles and interleaves them, so every lane keeps
// kRecordTiles independent loads in flight per round.
constexpr int kRecordTiles = 4;
constexpr int kRecordThreads = 256;

__global__ void __launch_bounds__(kRecordThreads) encode_records_kernel(const EncodeArgs a) {
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = (uint64_t(blockIdx.x) * (kRecordThreads / 32) + (threadIdx.x >> 5)) * kRecordTiles;
    if (t0 >= a.n_tiles) return;
    uint64_t first = 0;
    uint32_t cnt = 0;
    if (lane < kRecordTiles && t0 + lane < a.n_tiles) {
        first = a.tile_first[t0 + lane];
        cnt = a.tile_counts[t0 + lane];
    }
    uint64_t f[kRecordTiles];
    uint32_t c[kRecordTiles], most = 0;
#pragma unroll
    for (int k = 0; k < kRecordTiles; ++k) {
        f[k] = __shfl_sync(kFull, first, k);
        c[k] = __shfl_sync(kFull, cnt, k);
        most = max(most, c[k]);
    }
    const Layout L0 = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    uint8_t* records = a.out + L0.escrec_off;
    for (uint32_t i = lane; i < most; i += 32) {
        uint32_t r[kRecordTiles];
#pragma unroll
        for (int k = 0; k < kRecordTiles; ++k)
            r[k] = i < c[k] ? __ldcs(a.staging + (t0 + k) * a.tile_elems + i) : 0u;
#pragma unroll
        for (int k = 0; k < kRecordTiles; ++k) {
            if (i < c[k]) {
                uint8_t* d = records + 3 * (f[k] + i);
                d[0] = uint8_t(r[k] >> 8);
                d[1] = uint8_t(r[k] >> 16);
                d[2] = uint8_t(r[k]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_encode(const EncodeArgs& a, const EncodeLut& lut, int grid, cudaStream_t s) {
    if (a.dtype == SPLITZIP_BF16)
        encode_kernel<SPLITZIP_BF16><<<grid, kBlock, kEncodeSmem, s>>>(a, lut);
    else
        encode_kernel<SPLITZIP_FP8_E5M2><<<grid, kBlock, kEncodeSmem, s>>>(a, lut);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.n_groups == 0) return e;
    encode_index_kernel<<<unsigned(a.n_groups), kFinishThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const uint64_t warps = (a.n_tiles + kRecordTiles - 1) / kRecordTiles;
    encode_records_kernel<<<unsigned((warps + kRecordThreads / 32 - 1) / (kRecordThreads / 32)), kRecordThreads, 0,
                            s>>>(a);
    return cudaGetLastError();
}

cudaError_t occupancy_encode(int* blocks_per_sm, int dtype) {
    auto k = dtype == SPLITZIP_BF16 ? encode_kernel<SPLITZIP_BF16> : encode_kernel<SPLITZIP_FP8_E5M2>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kEncodeSmem));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kBlock, kEncodeSmem);
}

}  // namespace splitzip
