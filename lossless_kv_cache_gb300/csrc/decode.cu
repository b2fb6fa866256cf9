// SplitZip decode kernel for sm_103a.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Decoding strategy":
//   Parallelism — every byte of the nibble stream is unpacked into two 4-bit
//     codes and mapped through the 16-entry codebook in parallel; the result
//     is joined with the raw sign|mantissa bits.  Here one shared-memory table
//     lookup maps a whole nibble byte to its two exponents, so the dense path
//     has no branch on the data.
//   Correction — after the dense writes of a chunk (same CTA, after a
//     barrier), the chunk's escape records overwrite the exponent field of the
//     escaped elements, making the output bit-exact.
//
// Persistent grid: each CTA loops over chunks.  Every CTA validates the header
// first; each chunk validates its index entry and each escape record, and
// errors go to the status word without any out-of-bounds access.
#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

struct Header {
    uint64_t n, E, n_chunks;
    uint32_t chunk;
    Layout L;
    uint8_t codebook[16];
};

__device__ __forceinline__ void report(int* status, int code) { atomicCAS(status, SPLITZIP_OK, code); }

// Header checks (format v1): magic, version, dtype and n as given, reserved
// bytes zero, chunk size, chunk count, E <= n, codebook distinct and in range,
// container size within in_bytes.
__device__ bool read_header(const DecodeArgs& a, Header& h) {
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
    const uint32_t cbw[4] = {q2.x, q2.y, q2.z, q2.w};
    const uint32_t bins = a.dtype == SPLITZIP_BF16 ? 256u : 32u;
    uint32_t seen[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    for (int i = 0; i < 16; ++i) {
        const uint32_t e = (cbw[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        if (e >= bins || (seen[e >> 5] >> (e & 31)) & 1u) return false;
        seen[e >> 5] |= 1u << (e & 31);
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

// 12 bits of four packed s3 values -> one value per byte.
__device__ __forceinline__ uint32_t unpack_s3x4(uint32_t g) {
    const uint32_t y = (g & 0x3Fu) | ((g & 0xFC0u) << 10);       // groups of 2 at bytes 0 and 2
    return (y & 0x00070007u) | ((y << 5) & 0x07000700u);         // one value per byte
}

// E5M2: 16 elements from 16 codes (8 nibble bytes) and 48 bits of s3.
__device__ __forceinline__ uint4 decode_unit_e5m2(uint2 nib, uint32_t s3lo, uint32_t s3hi,
                                                  const uint16_t* lut2) {
    const uint32_t nb[2] = {nib.x, nib.y};
    uint32_t e[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        e[2 * i] = uint32_t(lut2[nb[i] & 0xFFu]) | (uint32_t(lut2[(nb[i] >> 8) & 0xFFu]) << 16);
        e[2 * i + 1] = uint32_t(lut2[(nb[i] >> 16) & 0xFFu]) | (uint32_t(lut2[nb[i] >> 24]) << 16);
    }
    const uint32_t g[4] = {s3lo & 0xFFFu, (s3lo >> 12) & 0xFFFu, (s3lo >> 24) | ((s3hi & 0xFu) << 8),
                           (s3hi >> 4) & 0xFFFu};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t s = unpack_s3x4(g[i]);
        o[i] = ((s << 5) & 0x80808080u) | ((e[i] << 2) & 0x7C7C7C7Cu) | (s & 0x03030303u);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int DT>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(const DecodeArgs a) {
    constexpr int kUnitElems = DT == SPLITZIP_BF16 ? 8 : 16;
    constexpr int kWarps = kDecodeThreads / 32;
    __shared__ Header hdr;
    __shared__ int header_ok;
    __shared__ uint16_t lut2[256];  // nibble byte -> (exponent of low code) | (exponent of high code) << 8
    __shared__ __align__(16) uint8_t s3_stage[kWarps][192];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        header_ok = read_header(a, hdr);
        if (!header_ok) report(a.status, SPLITZIP_ERR_CORRUPT);
    }
    __syncthreads();
    if (!header_ok) return;
    for (int b = tid; b < 256; b += kDecodeThreads)
        lut2[b] = uint16_t(hdr.codebook[b & 15]) | uint16_t(hdr.codebook[b >> 4] << 8);
    __syncthreads();

    const uint8_t* in = a.in;
    const Layout L = hdr.L;
    const uint8_t* nibbles = in + L.nibble_off;
    const uint8_t* signmant = in + L.signmant_off;
    const uint64_t* offsets = reinterpret_cast<const uint64_t*>(in + L.index_off);
    const uint32_t* counts = reinterpret_cast<const uint32_t*>(in + L.counts_off);
    const uint16_t* esc_pos = reinterpret_cast<const uint16_t*>(in + L.escpos_off);
    const uint8_t* esc_exp = in + L.escexp_off;
    const uint64_t chunk = hdr.chunk, C = hdr.n_chunks, E = hdr.E;

    for (uint64_t c = blockIdx.x; c < C; c += gridDim.x) {
        const uint64_t base = c * chunk;
        const uint32_t len = uint32_t(min(chunk, a.n - base));
        // ---- dense path ----
        for (uint32_t e = uint32_t(tid) * kUnitElems; e < len; e += kDecodeThreads * kUnitElems) {
            const uint32_t valid = min(len - e, uint32_t(kUnitElems));
            const uint64_t g = base + e;  // global element index of the unit
            if constexpr (DT == SPLITZIP_BF16) {
                uint32_t nib;
                uint2 sm;
                if (valid == 8u) {
                    nib = __ldcs(reinterpret_cast<const uint32_t*>(nibbles + g / 2));
                    sm = __ldcs(reinterpret_cast<const uint2*>(signmant + g));
                } else {
                    nib = 0u;
                    uint64_t smw = 0;
                    for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nib |= uint32_t(nibbles[g / 2 + b]) << (8u * b);
                    for (uint32_t b = 0; b < valid; ++b) smw |= uint64_t(signmant[g + b]) << (8u * b);
                    sm = make_uint2(uint32_t(smw), uint32_t(smw >> 32));
                }
                const uint4 o = decode_unit_bf16(nib, sm, lut2);
                uint16_t* out = static_cast<uint16_t*>(a.out) + g;
                if (valid == 8u) {
                    __stcs(reinterpret_cast<uint4*>(out), o);
                } else {
                    for (uint32_t k = 0; k < valid; ++k) {
                        const uint32_t q = k >> 1;
                        const uint32_t w = q == 0 ? o.x : q == 1 ? o.y : q == 2 ? o.z : o.w;
                        out[k] = uint16_t(w >> (16u * (k & 1u)));
                    }
                }
            } else {
                // s3 bytes of this unit: 6 per unit starting at 3 * g / 8.
                // Fast path: the warp's 32 units are full and 512-aligned in the
                // chunk, so the warp's 192 bytes are 16-aligned.
                const uint32_t warp_e0 = e - uint32_t(lane) * kUnitElems;
                const bool warp_full = (chunk % 512u == 0u) && (warp_e0 + 512u <= len);
                uint32_t s3lo, s3hi;
                if (warp_full) {  // warp-uniform
                    if (lane < 12) {
                        const uint8_t* src = signmant + (base + warp_e0) / 8 * 3 + 16 * lane;
                        reinterpret_cast<uint4*>(s3_stage[warp])[lane] = __ldcs(reinterpret_cast<const uint4*>(src));
                    }
                    __syncwarp();
                    const uint16_t* st = reinterpret_cast<const uint16_t*>(&s3_stage[warp][6 * lane]);
                    s3lo = uint32_t(st[0]) | (uint32_t(st[1]) << 16);
                    s3hi = st[2];
                    __syncwarp();
                } else {
                    const uint8_t* src = signmant + g / 8 * 3;
                    const uint32_t nbytes = 3u * ((valid + 7u) / 8u);
                    uint64_t w = 0;
                    for (uint32_t b = 0; b < nbytes; ++b) w |= uint64_t(src[b]) << (8u * b);
                    s3lo = uint32_t(w);
                    s3hi = uint32_t(w >> 32);
                }
                uint2 nib;
                if (valid == 16u) {
                    nib = __ldcs(reinterpret_cast<const uint2*>(nibbles + g / 2));
                } else {
                    uint64_t w = 0;
                    for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) w |= uint64_t(nibbles[g / 2 + b]) << (8u * b);
                    nib = make_uint2(uint32_t(w), uint32_t(w >> 32));
                }
                const uint4 o = decode_unit_e5m2(nib, s3lo, s3hi, lut2);
                uint8_t* out = static_cast<uint8_t*>(a.out) + g;
                if (valid == 16u) {
                    __stcs(reinterpret_cast<uint4*>(out), o);
                } else {
                    for (uint32_t k = 0; k < valid; ++k) {
                        const uint32_t q = k >> 2;
                        const uint32_t w = q == 0 ? o.x : q == 1 ? o.y : q == 2 ? o.z : o.w;
                        out[k] = uint8_t(w >> (8u * (k & 3u)));
                    }
                }
            }
        }
        __syncthreads();  // the chunk's dense writes are visible to the whole CTA

        // ---- correction: escape records of this chunk ----
        const uint64_t off = offsets[c];
        const uint64_t cnt = counts[c];
        const uint64_t expect_off = c == 0 ? 0 : offsets[c - 1] + counts[c - 1];
        const bool index_ok = off == expect_off && cnt <= len && off <= E && cnt <= E - off &&
                              (c + 1 < C || off + cnt == E);
        if (!index_ok) {
            if (tid == 0) report(a.status, SPLITZIP_ERR_CORRUPT);
            continue;
        }
        for (uint64_t i = tid; i < cnt; i += kDecodeThreads) {
            const uint32_t pos = esc_pos[off + i];
            const uint32_t ex = esc_exp[off + i];
            const bool ascending = i == 0 || esc_pos[off + i - 1] < pos;
            if (pos >= len || !ascending || ex >= (DT == SPLITZIP_BF16 ? 256u : 32u)) {
                report(a.status, SPLITZIP_ERR_CORRUPT);
                continue;
            }
            if constexpr (DT == SPLITZIP_BF16) {
                uint16_t* o = static_cast<uint16_t*>(a.out) + base + pos;
                *o = uint16_t((*o & 0x807Fu) | (ex << 7));
            } else {
                uint8_t* o = static_cast<uint8_t*>(a.out) + base + pos;
                *o = uint8_t((*o & 0x83u) | (ex << 2));
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s) {
    if (a.dtype == SPLITZIP_BF16)
        decode_kernel<SPLITZIP_BF16><<<grid, kDecodeThreads, 0, s>>>(a);
    else
        decode_kernel<SPLITZIP_FP8_E5M2><<<grid, kDecodeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t occupancy_decode(int* blocks_per_sm, int dtype) {
    if (dtype == SPLITZIP_BF16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<SPLITZIP_BF16>,
                                                             kDecodeThreads, 0);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<SPLITZIP_FP8_E5M2>,
                                                         kDecodeThreads, 0);
}

}  // namespace splitzip
