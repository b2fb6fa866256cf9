// Per-element encoder arithmetic shared by the streaming encoder (encode.cu)
// and the one-tile-per-CTA encoder of small tensors and batches (batch.cu):
// the position tables, the per-dtype packing of a 16-byte piece, the header.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Encoding strategy".
#pragma once

#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

// Position table entries (four tables, one per position k = 0..3 of an
// element within its group of four consecutive elements):
//   bits 16 + 4k .. 19 + 4k  the element's code (0 when it escapes)
//   bit  12 + k              the element's escape flag
//   bits 3k .. 3k + 1        E5M2 only: the element's 2 mantissa bits
// BF16 and FP16 tables are indexed by the exponent, E5M2 tables by the byte without
// its sign (exponent and mantissa: 128 entries, so elements that differ only
// in sign hit the same entry instead of another bank).  The four entries of a
// group have disjoint bits, so their sum -- plus, for E5M2, the four sign bits
// moved to bits 3k + 2 -- is the group's two nibble bytes (bits 16..31, even
// element in the low nibble), its escape mask (bits 12..15) and its 12 bits of
// packed 3-bit sign|mantissa values (bits 0..11).
__device__ __forceinline__ uint32_t table_entry(int dtype, int k, uint32_t index, const uint8_t* code) {
    uint32_t e = index, s3 = 0;
    if (dtype == SPLITZIP_FP8_E5M2) {  // index = exponent << 2 | mantissa
        e = (index >> 2) & 31u;
        s3 = index & 3u;
    }
    const uint32_t t = code[e];
    const uint32_t c = (t & kEscapeFlag) ? (1u << (12 + k)) : (uint32_t(t & 15u) << (16 + 4 * k));
    return c | (s3 << (3 * k));
}

// Entry of table k at byte offset `off` (index * 4).
__device__ __forceinline__ uint32_t tab_at(const uint32_t* tab, int k, uint32_t off) {
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(tab + 256 * k) + off);
}

// BF16: the group of four elements in words x (elements 0, 1) and y (2, 3);
// the table index is the exponent (bits 7..14 of each 16-bit element).
__device__ __forceinline__ uint32_t group_bf16(const uint32_t* tab, uint32_t x, uint32_t y) {
    return tab_at(tab, 0, (x >> 5) & 0x3FCu) + tab_at(tab, 1, (x >> 21) & 0x3FCu) +
           tab_at(tab, 2, (y >> 5) & 0x3FCu) + tab_at(tab, 3, (y >> 21) & 0x3FCu);
}

// FP16: the group of four elements in words x (elements 0, 1) and y (2, 3);
// the table index is the exponent (bits 10..14 of each 16-bit element).
__device__ __forceinline__ uint32_t group_fp16(const uint32_t* tab, uint32_t x, uint32_t y) {
    return tab_at(tab, 0, (x >> 8) & 0x7Cu) + tab_at(tab, 1, (x >> 24) & 0x7Cu) +
           tab_at(tab, 2, (y >> 8) & 0x7Cu) + tab_at(tab, 3, (y >> 24) & 0x7Cu);
}

// E5M2: the group of four elements in word w.  The sign of byte k (bit
// 8k + 7) belongs at bit 3k + 2: the high word of (signs * 0x08421000) has it
// there (term k is shifted by 27 - 5k), and every other product term lands on
// a bit of its own (checked for all 16 terms: no carries), so one mask keeps
// exactly the four signs.
__device__ __forceinline__ uint32_t group_e5m2(const uint32_t* tab, uint32_t w) {
    const uint32_t signs = __umulhi(w & 0x80808080u, 0x08421000u) & 0x924u;
    return tab_at(tab, 0, (w << 2) & 0x1FCu) + tab_at(tab, 1, (w >> 6) & 0x1FCu) +
           tab_at(tab, 2, (w >> 14) & 0x1FCu) + tab_at(tab, 3, (w >> 22) & 0x1FCu) + signs;
}

// Stage position of byte L of a tile: the tensor-map copy stores every
// 128-byte row r with its 16-byte pieces permuted by XOR with (r mod 8).
__device__ __forceinline__ uint32_t swizzled(uint32_t L) { return L ^ (((L >> 7) & 7u) << 4); }

// Load `nbytes` (< 16) bytes into a zero-filled vector (only the last bytes
// of a tensor are not covered by whole rows of the tensor map).
__device__ __forceinline__ uint4 load_partial(const uint8_t* p, uint32_t nbytes) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (uint32_t i = 0; i < 16; ++i)
        if (i < nbytes) w[i >> 2] |= uint32_t(p[i]) << (8 * (i & 3));
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Header fields known before any tile is encoded (E is written at the end),
// and the zero padding between sections, whose places depend only on n.  An
// empty tensor has no tile to finish the header, so its E and size go here.
__device__ void write_header_and_padding(uint8_t* h, int dtype, uint64_t n, uint32_t chunk_elems,
                                         uint64_t n_chunks, const uint8_t* codebook, uint64_t* out_size) {
    uint32_t* h32 = reinterpret_cast<uint32_t*>(h);
    h32[0] = kMagic;
    h32[1] = uint32_t(kVersion) | (uint32_t(dtype) << 16);  // version, dtype, reserved 0
    reinterpret_cast<uint64_t*>(h)[1] = n;
    h32[4] = chunk_elems;
    h32[5] = uint32_t(n_chunks);
    uint32_t cb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        cb[i] = uint32_t(codebook[4 * i]) | (uint32_t(codebook[4 * i + 1]) << 8) |
                (uint32_t(codebook[4 * i + 2]) << 16) | (uint32_t(codebook[4 * i + 3]) << 24);
    reinterpret_cast<uint4*>(h)[2] = make_uint4(cb[0], cb[1], cb[2], cb[3]);
    reinterpret_cast<uint4*>(h)[3] = make_uint4(0u, 0u, 0u, 0u);
    const Layout L = layout_for(n, dtype, chunk_elems, 0);
    for (uint64_t i = L.index_end; i < L.nibble_off; ++i) h[i] = 0;
    for (uint64_t i = L.nibble_off + (n + 1) / 2; i < L.signmant_off; ++i) h[i] = 0;
    for (uint64_t i = L.signmant_off + signmant_bytes(dtype, n); i < L.escrec_off; ++i) h[i] = 0;
    if (n == 0) {  // no tile will finish the header
        reinterpret_cast<uint64_t*>(h)[3] = 0;
        *out_size = L.size;
    }
}

// Per-thread results of one tile: BF16 32 elements, E5M2 64 elements.
template <int DT> struct ThreadOut;
template <> struct ThreadOut<SPLITZIP_BF16> {
    static constexpr uint32_t kElems = 32;
    uint32_t nib[4];  // 16 nibble bytes
    uint32_t sm[8];   // 32 sign|mantissa bytes
    uint32_t mask;    // escape flags, bit b = element b
};
template <> struct ThreadOut<SPLITZIP_FP16> {
    static constexpr uint32_t kElems = 32;
    uint32_t nib[4];  // 16 nibble bytes
    uint32_t sm[11];  // 44 bytes: 32 sign|mantissa fields of 11 bits, LSB-first
    uint32_t mask;
};
template <> struct ThreadOut<SPLITZIP_FP8_E5M2> {
    static constexpr uint32_t kElems = 64;
    uint32_t nib[8];  // 32 nibble bytes
    uint32_t s3[6];   // 24 bytes of packed 3-bit sign|mantissa
    uint32_t mask[2];
};

// One 16-byte piece (BF16: 8 elements) into slot i of the thread's results.
__device__ __forceinline__ void encode_piece(const uint32_t* tab, uint4 v, int i, ThreadOut<SPLITZIP_BF16>& o) {
    const uint32_t s0 = group_bf16(tab, v.x, v.y), s1 = group_bf16(tab, v.z, v.w);
    o.nib[i] = __byte_perm(s0, s1, 0x7632);
    o.mask |= (((s0 >> 12) & 0xFu) | ((s1 >> 8) & 0xF0u)) << (8 * i);
    // sign (bit 7 of the high byte) | mantissa (bits 6..0 of the low byte)
    const uint32_t lo0 = __byte_perm(v.x, v.y, 0x6420), hi0 = __byte_perm(v.x, v.y, 0x7531);
    const uint32_t lo1 = __byte_perm(v.z, v.w, 0x6420), hi1 = __byte_perm(v.z, v.w, 0x7531);
    o.sm[2 * i] = (hi0 & 0x80808080u) | (lo0 & 0x7F7F7F7Fu);
    o.sm[2 * i + 1] = (hi1 & 0x80808080u) | (lo1 & 0x7F7F7F7Fu);
}

// One 16-byte piece (FP16: 8 elements) into slot i of the thread's results.
// The sign|mantissa fields of a word's two elements form one 22-bit value
// (s11 of the even element | s11 of the odd one << 11): the even element's
// sign (bit 15) moves to bit 10 and the odd element's mantissa (bits 16..25)
// to bits 11..20 with the same shift by 5, its sign (bit 31) to bit 21.  Pair
// j of the thread's 16 lands at bit 22 j of its 352-bit run (o.sm, zeroed by
// the caller), possibly across two words.
__device__ __forceinline__ void encode_piece(const uint32_t* tab, uint4 v, int i, ThreadOut<SPLITZIP_FP16>& o) {
    const uint32_t s0 = group_fp16(tab, v.x, v.y), s1 = group_fp16(tab, v.z, v.w);
    o.nib[i] = __byte_perm(s0, s1, 0x7632);
    o.mask |= (((s0 >> 12) & 0xFu) | ((s1 >> 8) & 0xF0u)) << (8 * i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t x = w[j];
        const uint32_t pair = (x & 0x3FFu) | ((x >> 5) & 0x1FFC00u) | ((x >> 10) & 0x200000u);
        const int bit = 22 * (4 * i + j);
        o.sm[bit >> 5] |= pair << (bit & 31);
        if ((bit & 31) > 10) o.sm[(bit >> 5) + 1] |= pair >> (32 - (bit & 31));
    }
}

// One 16-byte piece (E5M2: 16 elements); the packed sign|mantissa of the
// piece (48 bits) is left in p[2i], p[2i+1] (24 bits each).
__device__ __forceinline__ void encode_piece(const uint32_t* tab, uint4 v, int i, ThreadOut<SPLITZIP_FP8_E5M2>& o,
                                             uint32_t* p) {
    const uint32_t s0 = group_e5m2(tab, v.x), s1 = group_e5m2(tab, v.y);
    const uint32_t s2 = group_e5m2(tab, v.z), s3 = group_e5m2(tab, v.w);
    o.nib[2 * i] = __byte_perm(s0, s1, 0x7632);
    o.nib[2 * i + 1] = __byte_perm(s2, s3, 0x7632);
    const uint32_t f = ((s0 >> 12) & 0xFu) | ((s1 >> 8) & 0xF0u) | ((s2 >> 4) & 0xF00u) | (s3 & 0xF000u);
    o.mask[i >> 1] |= f << (16 * (i & 1));
    p[2 * i] = (s0 & 0xFFFu) | ((s1 & 0xFFFu) << 12);
    p[2 * i + 1] = (s2 & 0xFFFu) | ((s3 & 0xFFFu) << 12);
}

// Eight 24-bit groups -> 24 bytes of the 3-bit stream.
__device__ __forceinline__ void pack_s3_stream(const uint32_t* p, uint32_t* out) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t* q = p + 4 * h;
        out[3 * h] = q[0] | (q[1] << 24);
        out[3 * h + 1] = (q[1] >> 8) | (q[2] << 16);
        out[3 * h + 2] = (q[2] >> 16) | (q[3] << 8);
    }
}

template <int DT>
__device__ __forceinline__ void clear_out(ThreadOut<DT>& o) {
    if constexpr (DT == SPLITZIP_BF16) {
        o.mask = 0u;
    } else if constexpr (DT == SPLITZIP_FP16) {
        o.mask = 0u;
#pragma unroll
        for (int k = 0; k < 11; ++k) o.sm[k] = 0u;
    } else {
        o.mask[0] = o.mask[1] = 0u;
    }
}

// The nibble and sign|mantissa bytes of a thread's run of elements, from
// element `first` of the tensor (a multiple of 32): all TE of them with
// 16-byte (BF16, E5M2) or 4-byte (FP16) streaming stores, or only the first
// `ne` (the end of the tensor) byte by byte, whose escape mask is then cut to
// those elements.  p: E5M2's packed sign|mantissa groups.
template <int DT, bool FULL>
__device__ __forceinline__ void store_streams(ThreadOut<DT>& o, const uint32_t* p, uint8_t* nibbles,
                                              uint8_t* signmant, uint64_t first, uint32_t ne) {
    constexpr uint32_t TE = ThreadOut<DT>::kElems;
    uint8_t* nb = nibbles + first / 2;
    if constexpr (DT == SPLITZIP_BF16) {
        uint8_t* sb = signmant + first;
        if (FULL || ne == TE) {
            __stcs(reinterpret_cast<uint4*>(nb), make_uint4(o.nib[0], o.nib[1], o.nib[2], o.nib[3]));
            __stcs(reinterpret_cast<uint4*>(sb), make_uint4(o.sm[0], o.sm[1], o.sm[2], o.sm[3]));
            __stcs(reinterpret_cast<uint4*>(sb) + 1, make_uint4(o.sm[4], o.sm[5], o.sm[6], o.sm[7]));
        } else if (ne > 0u) {
            o.mask &= (1u << (ne & 31u)) - 1u;  // ne < 32 here
            for (uint32_t b = 0; b < ne; b += 2) {
                const uint32_t w = o.nib[b >> 3] >> (4 * (b & 7u));
                nb[b >> 1] = uint8_t(b + 1 < ne ? (w & 0xFFu) : (w & 0xFu));
            }
            for (uint32_t b = 0; b < ne; ++b) sb[b] = uint8_t(o.sm[b >> 2] >> (8 * (b & 3u)));
        } else {
            o.mask = 0u;
        }
    } else if constexpr (DT == SPLITZIP_FP16) {
        // 44 bytes from byte 44 t of the tile's run: 4-byte aligned
        uint8_t* sb = signmant + first / 8 * 11;
        if (FULL || ne == TE) {
            __stcs(reinterpret_cast<uint4*>(nb), make_uint4(o.nib[0], o.nib[1], o.nib[2], o.nib[3]));
#pragma unroll
            for (int k = 0; k < 11; ++k) __stcs(reinterpret_cast<unsigned int*>(sb) + k, o.sm[k]);
        } else if (ne > 0u) {
            o.mask &= (1u << (ne & 31u)) - 1u;  // ne < 32 here
            for (uint32_t b = 0; b < ne; b += 2) {
                const uint32_t w = o.nib[b >> 3] >> (4 * (b & 7u));
                nb[b >> 1] = uint8_t(b + 1 < ne ? (w & 0xFFu) : (w & 0xFu));
            }
            // 11 bytes per started group of 8 elements (pad bits are 0)
            for (uint32_t b = 0; b < 11u * ((ne + 7u) / 8u); ++b) sb[b] = uint8_t(o.sm[b >> 2] >> (8 * (b & 3u)));
        } else {
            o.mask = 0u;
        }
    } else {
        uint32_t s3[6];
        pack_s3_stream(p, s3);
        uint8_t* sb = signmant + first / 8 * 3;
        if (FULL || ne == TE) {
            __stcs(reinterpret_cast<uint4*>(nb), make_uint4(o.nib[0], o.nib[1], o.nib[2], o.nib[3]));
            __stcs(reinterpret_cast<uint4*>(nb) + 1, make_uint4(o.nib[4], o.nib[5], o.nib[6], o.nib[7]));
#pragma unroll
            for (int k = 0; k < 3; ++k) __stcs(reinterpret_cast<uint2*>(sb) + k, make_uint2(s3[2 * k], s3[2 * k + 1]));
        } else if (ne > 0u) {
            if (ne < 32u) {  // ne < 64 here
                o.mask[0] &= (1u << (ne & 31u)) - 1u;
                o.mask[1] = 0u;
            } else {
                o.mask[1] &= (1u << ((ne - 32u) & 31u)) - 1u;
            }
            for (uint32_t b = 0; b < ne; b += 2) {
                const uint32_t w = o.nib[b >> 3] >> (4 * (b & 7u));
                nb[b >> 1] = uint8_t(b + 1 < ne ? (w & 0xFFu) : (w & 0xFu));
            }
            // 3 bytes per started group of 8 elements (pad bits are 0)
            for (uint32_t b = 0; b < 3u * ((ne + 7u) / 8u); ++b) sb[b] = uint8_t(s3[b >> 2] >> (8 * (b & 3u)));
        } else {
            o.mask[0] = o.mask[1] = 0u;
        }
    }
}

template <int DT>
__device__ __forceinline__ uint32_t escape_count(const ThreadOut<DT>& o) {
    if constexpr (DT != SPLITZIP_FP8_E5M2)
        return __popc(o.mask);
    else
        return __popc(o.mask[0]) + __popc(o.mask[1]);
}

// The escape flags of a thread's elements (element b = bit b of m[b / 32]).
template <int DT>
__device__ __forceinline__ void escape_masks(const ThreadOut<DT>& o, uint32_t* m) {
    if constexpr (DT != SPLITZIP_FP8_E5M2) {
        m[0] = o.mask;
        m[1] = 0u;
    } else {
        m[0] = o.mask[0];
        m[1] = o.mask[1];
    }
}

// The thread's escapes (flags m as from escape_masks), in element order, as
// 4-byte records (in-chunk position << 8) | exponent from slot[0] on; pos =
// in-chunk position of the thread's first element; bits(b) = the raw bits of
// its element b.
template <int DT, typename Bits>
__device__ __forceinline__ void stage_records_masked(const uint32_t* mask, uint32_t* slot, uint32_t pos, Bits bits) {
    auto record = [&](uint32_t b, uint32_t x) -> uint32_t {
        const uint32_t exponent = DT == SPLITZIP_BF16   ? (x >> 7) & 0xFFu
                                  : DT == SPLITZIP_FP16 ? (x >> 10) & 0x1Fu
                                                        : (x >> 2) & 0x1Fu;
        return ((pos + b) << 8) | exponent;
    };
#pragma unroll
    for (int h = 0; h < (DT == SPLITZIP_FP8_E5M2 ? 2 : 1); ++h) {
        uint32_t m = mask[h];
        // two escapes per round, so their two element reads overlap
        while (m) {
            const uint32_t b0 = 32u * h + uint32_t(__ffs(m) - 1);
            m &= m - 1u;
            const bool two = m != 0u;
            const uint32_t b1 = two ? 32u * h + uint32_t(__ffs(m) - 1) : b0;
            m &= two ? m - 1u : m;
            const uint32_t x0 = bits(b0), x1 = bits(b1);
            slot[0] = record(b0, x0);
            if (two) slot[1] = record(b1, x1);
            slot += two ? 2 : 1;
        }
    }
}

template <int DT, typename Bits>
__device__ __forceinline__ void stage_records(const ThreadOut<DT>& o, uint32_t* slot, uint32_t pos, Bits bits) {
    uint32_t m[2];
    escape_masks<DT>(o, m);
    stage_records_masked<DT>(m, slot, pos, bits);
}

}  // namespace
}  // namespace splitzip
