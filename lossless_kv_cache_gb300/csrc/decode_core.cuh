// Per-unit decoder arithmetic shared by the persistent decoder (decode.cu)
// and the one-sub-tile-per-CTA decoder of small tensors and batches
// (batch.cu): header checks, the per-dtype recombination of a unit, where an
// output element lives, and the escape patch.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Decoding strategy" (Parallelism,
// Correction).
#pragma once

#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

struct Header {
    uint64_t n, E, n_chunks;
    uint32_t chunk;
    Layout L;
    uint8_t codebook[16];
};

// Header checks (format v1): magic, version, dtype and n as given, reserved
// bytes zero, chunk size, chunk count, E <= n, codebook distinct and in range,
// container size within in_bytes.
__device__ __forceinline__ bool read_header(const DecodeArgs& a, Header& h) {
    if (a.in_bytes < kHeaderBytes) return false;
    const uint4* p = reinterpret_cast<const uint4*>(a.in);
    const uint4 q0 = p[0], q1 = p[1], q2 = p[2], q3 = p[3];
    if (q0.x != kMagic) return false;
    if ((q0.y & 0xFFFFu) != kVersion || ((q0.y >> 16) & 0xFFu) != uint32_t(a.dtype) || (q0.y >> 24) != 0u)
        return false;
    if ((q3.x | q3.y | q3.z | q3.w) != 0u) return false;
    h.n = uint64_t(q0.z) | (uint64_t(q0.w) << 32);
    h.chunk = q1.x;
    h.n_chunks = q1.y;
    h.E = uint64_t(q1.z) | (uint64_t(q1.w) << 32);
    if (h.n != a.n) return false;
    if (h.chunk < kMinChunk || h.chunk > kMaxChunk || (h.chunk & (h.chunk - 1u)) != 0u) return false;
    if ((h.n + h.chunk - 1u) / h.chunk != h.n_chunks) return false;
    if (h.E > h.n) return false;
    const uint32_t bins = a.dtype == SPLITZIP_BF16 ? 256u : 32u;
    uint64_t seen[4] = {0u, 0u, 0u, 0u};  // set of exponents met so far (constant indices only)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t w = i < 4 ? q2.x : i < 8 ? q2.y : i < 12 ? q2.z : q2.w;
        const uint32_t e = (w >> (8 * (i & 3))) & 0xFFu;
        const uint64_t bit = uint64_t(1) << (e & 63u);
        bool dup = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if ((e >> 6) == uint32_t(q)) {
                dup = (seen[q] & bit) != 0;
                seen[q] |= bit;
            }
        }
        if (e >= bins || dup) return false;
        h.codebook[i] = uint8_t(e);
    }
    h.L = layout_for(h.n, a.dtype, h.chunk, h.E);
    return h.L.size <= a.in_bytes;
}

// BF16: 8 elements from 8 codes (one nibble word) and 8 sign|mantissa bytes.
__device__ __forceinline__ uint4 decode_unit_bf16(uint32_t nib, uint2 sm, const uint16_t* lut2) {
    const uint32_t e0 = uint32_t(lut2[nib & 0xFFu]) | (uint32_t(lut2[(nib >> 8) & 0xFFu]) << 16);
    const uint32_t e1 = uint32_t(lut2[(nib >> 16) & 0xFFu]) | (uint32_t(lut2[nib >> 24]) << 16);
    // low byte = exponent bit 0 | mantissa; high byte = sign | exponent bits 7..1
    const uint32_t lo0 = ((e0 << 7) & 0x80808080u) | (sm.x & 0x7F7F7F7Fu);
    const uint32_t hi0 = (sm.x & 0x80808080u) | ((e0 >> 1) & 0x7F7F7F7Fu);
    const uint32_t lo1 = ((e1 << 7) & 0x80808080u) | (sm.y & 0x7F7F7F7Fu);
    const uint32_t hi1 = (sm.y & 0x80808080u) | ((e1 >> 1) & 0x7F7F7F7Fu);
    return make_uint4(__byte_perm(lo0, hi0, 0x5140), __byte_perm(lo0, hi0, 0x7362),
                      __byte_perm(lo1, hi1, 0x5140), __byte_perm(lo1, hi1, 0x7362));
}

// E5M2: 16 elements from 16 codes (8 nibble bytes) and 48 bits of s3.  The
// E5M2 table holds each exponent already at bits 2..6 of its byte.  For four
// elements with s3 values v0..v3 (12 bits g, v_k = sign << 2 | mantissa at bits
// 3k..3k+2), y = g[0:6] | g[6:12] << 16 puts v0, v1 at bits 0..5 and v2, v3
// at bits 16..21; from there every sign and mantissa field moves left by 0, 5
// or 10 bits to its place in the output bytes (sign bit 7, mantissa bits 0..1).
// The fields never overlap, so the moves are multiply-adds.
__device__ __forceinline__ uint32_t merge_e5m2(uint32_t g, uint32_t e) {
    const uint32_t y = (g & 0xFC0u) * 1024u + (g & 0x3Fu);
    const uint32_t t = (y & 0x00200020u) * 32u + (y & 0x001C001Cu);  // moved by 5 more, then all by 5
    return t * 32u + ((y & 0x00030003u) | e);
}

// FP16: a 22-bit pair value p (s11 of the even element | s11 of the odd one
// << 11) and both elements' exponents e already at bits 10..14 and 26..30 give
// the output word: mantissas stay at bits 0..9 / move to 16..25, signs move
// from bits 10 and 21 to 15 and 31 (fields never overlap).
__device__ __forceinline__ uint32_t merge_fp16(uint32_t p, uint32_t e) {
    return e | (p & 0x3FFu) | ((p << 5) & 0x03FF8000u) | ((p << 10) & 0x80000000u);
}

// FP16: 8 elements from 8 codes (one nibble word) and the unit's 88 bits of
// s11 (f0, f1, f2 = the 96 bits from the unit's first byte): pair k sits at
// bits [22k, 22k + 22).  lut4 maps a nibble byte to both exponents in place.
__device__ __forceinline__ uint4 decode_unit_fp16(uint32_t nib, uint32_t f0, uint32_t f1, uint32_t f2,
                                                  const uint32_t* lut4) {
    const uint32_t p0 = f0 & 0x3FFFFFu;
    const uint32_t p1 = __funnelshift_r(f0, f1, 22) & 0x3FFFFFu;
    const uint32_t p2 = __funnelshift_r(f1, f2, 12) & 0x3FFFFFu;
    const uint32_t p3 = (f2 >> 2) & 0x3FFFFFu;
    return make_uint4(merge_fp16(p0, lut4[nib & 0xFFu]), merge_fp16(p1, lut4[(nib >> 8) & 0xFFu]),
                      merge_fp16(p2, lut4[(nib >> 16) & 0xFFu]), merge_fp16(p3, lut4[nib >> 24]));
}

__device__ __forceinline__ uint16_t lut_at(const uint16_t* lut2, uint32_t byte) {
    return *reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(lut2) + 2u * byte);
}

__device__ __forceinline__ uint4 decode_unit_e5m2(uint2 nib, uint32_t s3lo, uint32_t s3hi, const uint16_t* lut2) {
    const uint32_t nb[2] = {nib.x, nib.y};
    uint32_t e[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t w = nb[i];
        e[2 * i] = __byte_perm(lut_at(lut2, __byte_perm(w, 0u, 0x4440u)), lut_at(lut2, __byte_perm(w, 0u, 0x4441u)),
                               0x5410u);
        e[2 * i + 1] = __byte_perm(lut_at(lut2, __byte_perm(w, 0u, 0x4442u)), lut_at(lut2, w >> 24), 0x5410u);
    }
    // only bits 0..11 of each g are used
    return make_uint4(merge_e5m2(s3lo, e[0]), merge_e5m2(s3lo >> 12, e[1]),
                      merge_e5m2(__funnelshift_r(s3lo, s3hi, 24), e[2]), merge_e5m2(s3hi >> 4, e[3]));
}

// Where element g of the tensor is written: itself (contiguous output) or,
// with paged output, element g mod 2^shift of pool page pages[g >> shift].
// A page index outside the pool is reported and its elements are not
// written.  The 16-byte units and the 4-byte words the decoder writes never
// straddle a page (pages hold a power of two >= 16 elements).
template <bool PAGED>
struct OutMap {
    uint8_t* base;
    uint64_t limit;  // bytes of the output (tensor or pool)
    const int32_t* pages;
    uint64_t pool_pages;
    uint32_t shift;
    int* status;
    __device__ __forceinline__ bool at(uint64_t g, uint32_t eb, uint64_t& off) const {
        if constexpr (!PAGED) {
            off = g * eb;
            return true;
        } else {
            const int64_t p = pages[g >> shift];
            if (p < 0 || uint64_t(p) >= pool_pages) {
                atomicCAS(status, SPLITZIP_OK, SPLITZIP_ERR_INVALID_ARG);
                return false;
            }
            off = ((uint64_t(p) << shift) | (g & ((uint64_t(1) << shift) - 1u))) * eb;
            return true;
        }
    }
};

// FP16: the 96 bits from smem byte address a (four aligned words, shifted)
__device__ __forceinline__ void load96(const uint8_t* a, uint32_t& f0, uint32_t& f1, uint32_t& f2) {
    const uint32_t* w = reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(a) & ~uintptr_t(3));
    const uint32_t sh = 8u * uint32_t(reinterpret_cast<uintptr_t>(a) & 3u);
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3];
    f0 = __funnelshift_r(w0, w1, sh);
    f1 = __funnelshift_r(w1, w2, sh);
    f2 = __funnelshift_r(w2, w3, sh);
}

// Escape-record check and patch of one element (returns false on a corrupt
// record).  `prev` is the previous record's position in the chunk (or -1).
// The exponent field is rewritten with two atomic reductions on the 32-bit
// word that holds the element (AND clears the field, OR sets it; the results
// are unused, so neither waits for memory, and one thread's two operations on
// one address stay in order).  Other elements of the word are left as they
// are; a word that would reach past the output's last byte (only at the very
// end of an odd-sized output) is patched by a plain read-modify-write.
template <int DT, bool PAGED>
__device__ __forceinline__ bool patch_one(const OutMap<PAGED>& om, uint64_t base, uint32_t len, int64_t prev,
                                          uint32_t pos, uint32_t ex) {
    if (pos >= len || int64_t(pos) <= prev || ex >= (DT == SPLITZIP_BF16 ? 256u : 32u)) return false;
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    // bit of the exponent field within a 16-bit (BF16, FP16) or 8-bit element
    constexpr uint32_t kExpShift = DT == SPLITZIP_BF16 ? 7u : DT == SPLITZIP_FP16 ? 10u : 2u;
    uint64_t byte;
    if (!om.at(base + pos, EB, byte)) return true;  // (reported: a page outside the pool)
    uint8_t* o = om.base;
    if ((byte | 3u) < om.limit) {
        const uint32_t sh = uint32_t(byte & 3u) * 8u + kExpShift;
        const uint32_t field = (DT == SPLITZIP_BF16 ? 0xFFu : 0x1Fu) << sh;
        unsigned int* w = reinterpret_cast<unsigned int*>(o + (byte & ~uint64_t(3)));
        atomicAnd(w, ~field);
        atomicOr(w, ex << sh);
    } else if constexpr (DT == SPLITZIP_BF16) {
        uint16_t* e = reinterpret_cast<uint16_t*>(o + byte);
        *e = uint16_t((*e & 0x807Fu) | (ex << 7));
    } else if constexpr (DT == SPLITZIP_FP16) {
        uint16_t* e = reinterpret_cast<uint16_t*>(o + byte);
        *e = uint16_t((*e & 0x83FFu) | (ex << 10));
    } else {
        o[byte] = uint8_t((o[byte] & 0x83u) | (ex << 2));
    }
    return true;
}

__device__ __forceinline__ uint32_t rec_pos(const uint8_t* r) { return uint32_t(r[0]) | (uint32_t(r[1]) << 8); }

}  // namespace
}  // namespace splitzip
