// The page's ablation formats on sm_103a (section "Results", "Ablation
// Studies"; Method, the design choice of Top-16 over Top-15): Top-8 (8 coded
// exponents, 3-bit codes, explicit escape records) and Top-15 + sentinel
// (code 15 marks an escape; the escape stream holds only the exponents, their
// positions found from the sentinels).  Containers: the main format's header,
// index and sign|mantissa stream; header byte 7 names the variant (0 = Top-16,
// the main format, 1 = Top-8, 2 = Top-15 + sentinel); the code stream is 3 bits
// per element (Top-8, LSB-first, 3 bytes per 8 elements) or one nibble; the
// escape stream is 3-byte (position, exponent) records (Top-16, Top-8) or one
// exponent byte per escape (sentinel).
//
// One kernel family serves the three formats, so that their measured speeds
// differ only by what the formats ask for: plain 16-byte loads and stores, one
// CTA per chunk, 32-element units, unit u of a chunk handled by thread u mod 256
// in round u / 256.  Encode: per-chunk escape counts, one CTA's prefix scan
// (the index, E, the header), then the streams, with a block scan per round
// placing each escape in element order.  Decode: the dense pass, then, for
// explicit records, the patch after a barrier; the sentinel format instead
// ranks each unit's sentinels by a block scan per round and gathers their
// exponents.  (The production Top-16 path is encode.cu / decode.cu.)
#include <algorithm>
#include <cstring>

#include "splitzip.h"
#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

constexpr int kAblThreads = 256;
constexpr uint32_t kUnit = 32;     // elements per unit
constexpr uint8_t kNoCode = 0xFF;  // exponent outside the codebook

__host__ __device__ inline uint32_t abl_codes(int variant) { return variant == 1 ? 8u : variant == 2 ? 15u : 16u; }

struct AblLayout {
    uint64_t n_chunks, index_off, counts_off, code_off, sm_off, esc_off, size;
};

__host__ __device__ inline AblLayout abl_layout(uint64_t n, int dtype, uint32_t chunk, int variant, uint64_t E) {
    AblLayout L;
    L.n_chunks = (n + chunk - 1u) / chunk;
    L.index_off = kHeaderBytes;
    L.counts_off = L.index_off + 8u * L.n_chunks;
    L.code_off = align16(L.counts_off + 4u * L.n_chunks);
    const uint64_t code_bytes = variant == 1 ? 3u * ((n + 7u) / 8u) : (n + 1u) / 2u;
    const uint64_t sm_bytes = dtype == SPLITZIP_BF16 ? n : 3u * ((n + 7u) / 8u);
    L.sm_off = L.code_off + align16(code_bytes);
    L.esc_off = L.sm_off + align16(sm_bytes);
    L.size = L.esc_off + (variant == 2 ? 1u : 3u) * E;
    return L;
}

struct AblEncodeArgs {
    const uint8_t* in;
    uint64_t n;
    uint8_t* out;
    uint64_t* out_size;
    int* status;
    uint32_t chunk;
    int dtype, variant;
    uint8_t codebook[16];
    uint8_t code_of[256];  // exponent -> code, or kNoCode
};

struct AblDecodeArgs {
    const uint8_t* in;
    uint64_t in_bytes;
    uint8_t* out;
    uint64_t n;
    int* status;
    int dtype, variant;
};

__device__ __forceinline__ void abl_report(int* status, int code) { atomicCAS(status, SPLITZIP_OK, code); }

// Exclusive scan of v over the CTA (all kAblThreads threads call it); also
// returns the CTA's total.  `tmp`: kAblThreads / 32 + 1 words of shared memory.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* tmp, uint32_t& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += y;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t run = 0;
        for (int w = 0; w < kAblThreads / 32; ++w) {
            const uint32_t t = tmp[w];
            tmp[w] = run;
            run += t;
        }
        tmp[kAblThreads / 32] = run;
    }
    __syncthreads();
    const uint32_t r = tmp[warp] + incl - v;
    total = tmp[kAblThreads / 32];
    __syncthreads();  // tmp may be reused right away
    return r;
}

// element i's raw bits
template <int DT>
__device__ __forceinline__ uint32_t abl_load(const uint8_t* in, uint64_t i) {
    if constexpr (DT == SPLITZIP_BF16)
        return uint32_t(reinterpret_cast<const uint16_t*>(in)[i]);
    else
        return uint32_t(in[i]);
}

template <int DT>
__device__ __forceinline__ uint32_t abl_exponent(uint32_t v) {
    return DT == SPLITZIP_BF16 ? (v >> 7) & 0xFFu : (v >> 2) & 0x1Fu;
}

// sign|mantissa field (BF16 byte (s << 7) | m7; E5M2 3 bits (s << 2) | m2)
template <int DT>
__device__ __forceinline__ uint32_t abl_signmant(uint32_t v) {
    return DT == SPLITZIP_BF16 ? ((v >> 8) & 0x80u) | (v & 0x7Fu) : ((v >> 5) & 4u) | (v & 3u);
}

template <int DT>
__device__ __forceinline__ uint32_t abl_join(uint32_t sm, uint32_t e) {
    return DT == SPLITZIP_BF16 ? ((sm & 0x80u) << 8) | (e << 7) | (sm & 0x7Fu)
                               : ((sm & 4u) << 5) | (e << 2) | (sm & 3u);
}

// ---- encode pass 1: each chunk's escape count, into the index's count slots
template <int DT>
__global__ void __launch_bounds__(kAblThreads) abl_count_kernel(const AblEncodeArgs a) {
    __shared__ uint8_t code_s[256];
    __shared__ uint32_t tmp[kAblThreads / 32 + 1];
    for (int i = threadIdx.x; i < 256; i += kAblThreads) code_s[i] = a.code_of[i];
    __syncthreads();
    const uint64_t c = blockIdx.x, base = c * a.chunk;
    const uint32_t len = uint32_t(min(uint64_t(a.chunk), a.n - base));
    uint32_t cnt = 0;
    for (uint32_t e = threadIdx.x; e < len; e += kAblThreads)
        cnt += code_s[abl_exponent<DT>(abl_load<DT>(a.in, base + e))] == kNoCode;
    uint32_t total;
    block_excl_scan(cnt, tmp, total);
    const AblLayout L = abl_layout(a.n, a.dtype, a.chunk, a.variant, 0);
    if (threadIdx.x == 0) reinterpret_cast<uint32_t*>(a.out + L.counts_off)[c] = total;
}

// ---- encode pass 2 (one CTA): the offsets (exclusive prefix of the counts),
// the header, E, the size and the zero padding between sections
__global__ void __launch_bounds__(kAblThreads) abl_index_kernel(const AblEncodeArgs a) {
    __shared__ uint32_t tmp[kAblThreads / 32 + 1];
    const AblLayout L = abl_layout(a.n, a.dtype, a.chunk, a.variant, 0);
    const uint32_t* counts = reinterpret_cast<const uint32_t*>(a.out + L.counts_off);
    uint64_t* offsets = reinterpret_cast<uint64_t*>(a.out + L.index_off);
    uint64_t running = 0;
    for (uint64_t c0 = 0; c0 < L.n_chunks; c0 += kAblThreads) {
        const uint64_t c = c0 + threadIdx.x;
        const uint32_t v = c < L.n_chunks ? counts[c] : 0u;
        uint32_t total;
        const uint32_t excl = block_excl_scan(v, tmp, total);
        if (c < L.n_chunks) offsets[c] = running + excl;
        running += total;
    }
    uint8_t* h = a.out;
    if (threadIdx.x == 0) {
        reinterpret_cast<uint32_t*>(h)[0] = kMagic;
        reinterpret_cast<uint16_t*>(h)[2] = uint16_t(kVersion);
        h[6] = uint8_t(a.dtype);
        h[7] = uint8_t(a.variant);
        reinterpret_cast<uint64_t*>(h)[1] = a.n;
        reinterpret_cast<uint32_t*>(h)[4] = a.chunk;
        reinterpret_cast<uint32_t*>(h)[5] = uint32_t(L.n_chunks);
        reinterpret_cast<uint64_t*>(h)[3] = running;
        *a.out_size = abl_layout(a.n, a.dtype, a.chunk, a.variant, running).size;
    }
    if (threadIdx.x < 16) h[32 + threadIdx.x] = a.codebook[threadIdx.x];
    if (threadIdx.x < 16) h[48 + threadIdx.x] = 0;
    const uint64_t code_end = L.code_off + (a.variant == 1 ? 3u * ((a.n + 7u) / 8u) : (a.n + 1u) / 2u);
    const uint64_t sm_end = L.sm_off + (a.dtype == SPLITZIP_BF16 ? a.n : 3u * ((a.n + 7u) / 8u));
    for (uint64_t i = L.counts_off + 4u * L.n_chunks + threadIdx.x; i < L.code_off; i += kAblThreads) h[i] = 0;
    for (uint64_t i = code_end + threadIdx.x; i < L.sm_off; i += kAblThreads) h[i] = 0;
    for (uint64_t i = sm_end + threadIdx.x; i < L.esc_off; i += kAblThreads) h[i] = 0;
}

// ---- encode pass 3: the code and sign|mantissa streams and the escapes, unit
// by unit; a block scan per round gives each unit's first escape index
template <int DT, int VAR>
__global__ void __launch_bounds__(kAblThreads) abl_write_kernel(const AblEncodeArgs a) {
    constexpr uint32_t EB = DT == SPLITZIP_BF16 ? 2u : 1u;
    __shared__ uint8_t code_s[256];
    __shared__ uint32_t tmp[kAblThreads / 32 + 1];
    for (int i = threadIdx.x; i < 256; i += kAblThreads) code_s[i] = a.code_of[i];
    __syncthreads();
    const uint64_t c = blockIdx.x, base = c * a.chunk;
    const uint32_t len = uint32_t(min(uint64_t(a.chunk), a.n - base));
    const AblLayout L = abl_layout(a.n, a.dtype, a.chunk, VAR, 0);
    uint64_t next = reinterpret_cast<const uint64_t*>(a.out + L.index_off)[c];  // this chunk's first escape
    const uint32_t units = (len + kUnit - 1u) / kUnit;
    const uint32_t rounds = (units + kAblThreads - 1u) / kAblThreads;
    for (uint32_t r = 0; r < rounds; ++r) {
        const uint32_t e0 = (r * kAblThreads + threadIdx.x) * kUnit;  // first element of the unit in the chunk
        const uint32_t m = e0 < len ? min(kUnit, len - e0) : 0u;
        const uint64_t g = base + e0;
        uint32_t mask = 0;
#pragma unroll
        for (uint32_t j = 0; j < kUnit; ++j)
            if (j < m && code_s[abl_exponent<DT>(abl_load<DT>(a.in, g + j))] == kNoCode) mask |= 1u << j;
        uint32_t total;
        const uint64_t rank = next + block_excl_scan(__popc(mask), tmp, total);
        next += total;
        if (m == 0) continue;
        uint32_t cw[4] = {0u, 0u, 0u, 0u};       // code bits of the unit (128 or 96)
        uint32_t sw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // sign|mantissa bits (256 or 96)
        uint32_t k = 0;
#pragma unroll
        for (uint32_t j = 0; j < kUnit; ++j) {
            if (j >= m) continue;
            const uint32_t v = abl_load<DT>(a.in, g + j);
            const uint32_t ex = abl_exponent<DT>(v), sm = abl_signmant<DT>(v);
            uint32_t code = code_s[ex];
            if (code == kNoCode) {
                if constexpr (VAR == 2) {
                    a.out[L.esc_off + rank + k] = uint8_t(ex);
                    code = 15u;
                } else {
                    uint8_t* rec = a.out + L.esc_off + 3u * (rank + k);
                    rec[0] = uint8_t((e0 + j) & 0xFFu);
                    rec[1] = uint8_t((e0 + j) >> 8);
                    rec[2] = uint8_t(ex);
                    code = 0u;
                }
                ++k;
            }
            if constexpr (VAR == 1) {
                const uint32_t bit = 3u * j;
                cw[bit >> 5] |= code << (bit & 31u);
                if ((bit & 31u) > 29u) cw[(bit >> 5) + 1] |= code >> (32u - (bit & 31u));
            } else {
                cw[j >> 3] |= code << (4u * (j & 7u));
            }
            if constexpr (DT == SPLITZIP_BF16) {
                sw[j >> 2] |= sm << (8u * (j & 3u));
            } else {
                const uint32_t bit = 3u * j;
                sw[bit >> 5] |= sm << (bit & 31u);
                if ((bit & 31u) > 29u) sw[(bit >> 5) + 1] |= sm >> (32u - (bit & 31u));
            }
        }
        uint8_t* cd = a.out + L.code_off + (VAR == 1 ? g / 8u * 3u : g / 2u);
        uint8_t* sd = a.out + L.sm_off + (DT == SPLITZIP_BF16 ? g : g / 8u * 3u);
        if (m == kUnit) {
            if constexpr (VAR == 1) {
                for (int w = 0; w < 3; ++w) reinterpret_cast<uint32_t*>(cd)[w] = cw[w];
            } else {
                *reinterpret_cast<uint4*>(cd) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            }
            if constexpr (DT == SPLITZIP_BF16) {
                reinterpret_cast<uint4*>(sd)[0] = make_uint4(sw[0], sw[1], sw[2], sw[3]);
                reinterpret_cast<uint4*>(sd)[1] = make_uint4(sw[4], sw[5], sw[6], sw[7]);
            } else {
                for (int w = 0; w < 3; ++w) reinterpret_cast<uint32_t*>(sd)[w] = sw[w];
            }
        } else {  // the tensor's last, short unit: only the bytes its elements reach
            const uint32_t cbytes = VAR == 1 ? 3u * ((m + 7u) / 8u) : (m + 1u) / 2u;
#pragma unroll
            for (uint32_t b = 0; b < 16; ++b)
                if (b < cbytes) cd[b] = uint8_t(cw[b >> 2] >> (8u * (b & 3u)));
            const uint32_t sbytes = DT == SPLITZIP_BF16 ? m : 3u * ((m + 7u) / 8u);
#pragma unroll
            for (uint32_t b = 0; b < 32; ++b)
                if (b < sbytes) sd[b] = uint8_t(sw[b >> 2] >> (8u * (b & 3u)));
        }
        (void)EB;
    }
}

// ---- decode: persistent CTAs, chunk c to CTA c mod G (the chunk count comes
// from the header).  Thread 0 checks the header, then each chunk's index
// entry; the dense pass writes every element (the sentinel format takes
// the exponents of its escapes from the escape stream in element order); the
// explicit formats then patch their escapes after a barrier.
template <int DT, int VAR>
__global__ void __launch_bounds__(kAblThreads) abl_decode_kernel(const AblDecodeArgs a) {
    constexpr uint32_t EB = DT == SPLITZIP_BF16 ? 2u : 1u;
    constexpr uint32_t kBins = DT == SPLITZIP_BF16 ? 256u : 32u;
    __shared__ uint32_t lut[16];
    __shared__ uint32_t tmp[kAblThreads / 32 + 1];
    __shared__ int hdr_ok, ok_s;
    __shared__ uint32_t chunk_s, C_s;
    __shared__ uint64_t off_s, cnt_s, E_s;
    if (threadIdx.x == 0) {
        const uint8_t* h = a.in;
        bool ok = a.in_bytes >= kHeaderBytes && reinterpret_cast<const uint32_t*>(h)[0] == kMagic &&
                  reinterpret_cast<const uint16_t*>(h)[2] == kVersion && h[6] == uint8_t(a.dtype) && h[7] == VAR;
        for (int b = 48; ok && b < 64; ++b) ok = h[b] == 0;
        const uint64_t n = ok ? reinterpret_cast<const uint64_t*>(h)[1] : 0;
        const uint32_t chunk = ok ? reinterpret_cast<const uint32_t*>(h)[4] : 64u;
        const uint32_t C = ok ? reinterpret_cast<const uint32_t*>(h)[5] : 0u;
        const uint64_t E = ok ? reinterpret_cast<const uint64_t*>(h)[3] : 0;
        ok = ok && n == a.n && chunk >= kMinChunk && chunk <= kMaxChunk && (chunk & (chunk - 1u)) == 0 &&
             (n + chunk - 1u) / chunk == C && E <= n;
        // codebook: the first k exponents distinct and in range, the rest zero
        const uint32_t k = abl_codes(VAR);
        uint64_t seen_e[4] = {0, 0, 0, 0};
        for (uint32_t i = 0; ok && i < 16; ++i) {
            const uint32_t e = h[32 + i];
            if (i >= k) {
                ok = e == 0;
                continue;
            }
            const uint64_t bit = uint64_t(1) << (e & 63u);
            ok = e < kBins && !(seen_e[e >> 6] & bit);
            seen_e[e >> 6] |= bit;
        }
        ok = ok && abl_layout(n, a.dtype, chunk, VAR, E).size <= a.in_bytes;
        for (uint32_t i = 0; i < 16; ++i) lut[i] = h[32 + i];
        chunk_s = chunk;
        C_s = ok ? C : 0u;
        E_s = E;
        hdr_ok = ok;
        if (!ok) abl_report(a.status, SPLITZIP_ERR_CORRUPT);
    }
    __syncthreads();
    if (!hdr_ok) return;
    const uint32_t chunk = chunk_s;
    const AblLayout L = abl_layout(a.n, a.dtype, chunk, VAR, E_s);
    for (uint64_t c = blockIdx.x; c < C_s; c += gridDim.x) {
    if (threadIdx.x == 0) {
        // the chunk's index entry: offset = the prefix, count within the chunk
        const uint64_t* offs = reinterpret_cast<const uint64_t*>(a.in + L.index_off);
        const uint32_t* cnts = reinterpret_cast<const uint32_t*>(a.in + L.counts_off);
        const uint64_t off = offs[c], cnt = cnts[c], E = E_s;
        const uint64_t len = min(uint64_t(chunk), a.n - c * chunk);
        const uint64_t expect = c == 0 ? 0 : offs[c - 1] + cnts[c - 1];
        const bool ok = off == expect && cnt <= len && off <= E && cnt <= E - off && (c + 1 < C_s || off + cnt == E);
        off_s = off;
        cnt_s = cnt;
        ok_s = ok;
        if (!ok) abl_report(a.status, SPLITZIP_ERR_CORRUPT);
    }
    __syncthreads();
    if (ok_s) {
    const uint64_t base = c * chunk, off = off_s, cnt = cnt_s;
    const uint32_t len = uint32_t(min(uint64_t(chunk), a.n - base));
    const uint8_t* esc = a.in + L.esc_off;
    bool bad = false;
    uint64_t seen = 0;  // sentinels met so far in this chunk (the sentinel format)
    const uint32_t units = (len + kUnit - 1u) / kUnit;
    const uint32_t rounds = (units + kAblThreads - 1u) / kAblThreads;
    for (uint32_t r = 0; r < rounds; ++r) {
        const uint32_t e0 = (r * kAblThreads + threadIdx.x) * kUnit;
        const uint32_t m = e0 < len ? min(kUnit, len - e0) : 0u;
        const uint64_t g = base + e0;
        const uint8_t* cs = a.in + L.code_off + (VAR == 1 ? g / 8u * 3u : g / 2u);
        const uint8_t* ss = a.in + L.sm_off + (DT == SPLITZIP_BF16 ? g : g / 8u * 3u);
        uint32_t cw[4] = {0u, 0u, 0u, 0u}, sw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (m == kUnit) {
            if constexpr (VAR == 1) {
                for (int w = 0; w < 3; ++w) cw[w] = reinterpret_cast<const uint32_t*>(cs)[w];
            } else {
                const uint4 q = *reinterpret_cast<const uint4*>(cs);
                cw[0] = q.x; cw[1] = q.y; cw[2] = q.z; cw[3] = q.w;
            }
            if constexpr (DT == SPLITZIP_BF16) {
                const uint4 q0 = reinterpret_cast<const uint4*>(ss)[0], q1 = reinterpret_cast<const uint4*>(ss)[1];
                sw[0] = q0.x; sw[1] = q0.y; sw[2] = q0.z; sw[3] = q0.w;
                sw[4] = q1.x; sw[5] = q1.y; sw[6] = q1.z; sw[7] = q1.w;
            } else {
                for (int w = 0; w < 3; ++w) sw[w] = reinterpret_cast<const uint32_t*>(ss)[w];
            }
        } else if (m > 0) {
            const uint32_t cbytes = VAR == 1 ? 3u * ((m + 7u) / 8u) : (m + 1u) / 2u;
#pragma unroll
            for (uint32_t b = 0; b < 16; ++b)
                if (b < cbytes) cw[b >> 2] |= uint32_t(cs[b]) << (8u * (b & 3u));
            const uint32_t sbytes = DT == SPLITZIP_BF16 ? m : 3u * ((m + 7u) / 8u);
#pragma unroll
            for (uint32_t b = 0; b < 32; ++b)
                if (b < sbytes) sw[b >> 2] |= uint32_t(ss[b]) << (8u * (b & 3u));
        }
        auto code_at = [&](uint32_t j) -> uint32_t {
            if constexpr (VAR == 1) {
                const uint32_t bit = 3u * j, w = bit >> 5, s = bit & 31u;
                uint32_t v = cw[w] >> s;
                if (s > 29u) v |= cw[w + 1] << (32u - s);
                return v & 7u;
            } else {
                return (cw[j >> 3] >> (4u * (j & 7u))) & 15u;
            }
        };
        uint64_t rank = 0;
        if constexpr (VAR == 2) {
            // this unit's sentinels, ranked in element order over the chunk
            uint32_t mask = 0;
#pragma unroll
            for (uint32_t j = 0; j < kUnit; ++j)
                if (j < m && code_at(j) == 15u) mask |= 1u << j;
            uint32_t total;
            rank = seen + block_excl_scan(__popc(mask), tmp, total);
            seen += total;
        }
        if (m == 0) continue;
        uint32_t ow[16] = {};  // the unit's output: 64 bytes (BF16) or 32 (E5M2)
#pragma unroll
        for (uint32_t j = 0; j < kUnit; ++j) {
            if (j >= m) continue;
            const uint32_t code = code_at(j);
            uint32_t e;
            if (VAR == 2 && code == 15u) {
                if (rank < cnt) {
                    e = esc[off + rank];
                    bad |= e >= kBins;
                    e &= kBins - 1u;
                } else {
                    bad = true;
                    e = 0;
                }
                ++rank;
            } else {
                e = lut[code];
            }
            uint32_t sm;
            if constexpr (DT == SPLITZIP_BF16) {
                sm = (sw[j >> 2] >> (8u * (j & 3u))) & 0xFFu;
                ow[j >> 1] |= abl_join<DT>(sm, e) << (16u * (j & 1u));
            } else {
                const uint32_t bit = 3u * j, w = bit >> 5, s = bit & 31u;
                uint32_t v = sw[w] >> s;
                if (s > 29u) v |= sw[w + 1] << (32u - s);
                sm = v & 7u;
                ow[j >> 2] |= abl_join<DT>(sm, e) << (8u * (j & 3u));
            }
        }
        uint8_t* od = a.out + g * EB;
        if (m == kUnit) {
            if constexpr (DT == SPLITZIP_BF16) {
                for (int q = 0; q < 4; ++q)
                    reinterpret_cast<uint4*>(od)[q] = make_uint4(ow[4 * q], ow[4 * q + 1], ow[4 * q + 2], ow[4 * q + 3]);
            } else {
                reinterpret_cast<uint4*>(od)[0] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                reinterpret_cast<uint4*>(od)[1] = make_uint4(ow[4], ow[5], ow[6], ow[7]);
            }
        } else {
#pragma unroll
            for (uint32_t b = 0; b < kUnit * EB; ++b)
                if (b < m * EB) od[b] = uint8_t(ow[b >> 2] >> (8u * (b & 3u)));
        }
    }
    if constexpr (VAR == 2) {
        if (seen != cnt) bad = true;
    } else {
        __syncthreads();  // the chunk's dense stores, visible to every thread of the CTA
        for (uint64_t i = threadIdx.x; i < cnt; i += kAblThreads) {
            const uint8_t* rec = esc + 3u * (off + i);
            const uint32_t pos = uint32_t(rec[0]) | (uint32_t(rec[1]) << 8), e = rec[2];
            const bool in_order = i == 0 || pos > (uint32_t(rec[-3]) | (uint32_t(rec[-2]) << 8));
            if (pos >= len || e >= kBins || !in_order) {
                bad = true;
                continue;
            }
            const uint64_t byte = (base + pos) * EB;
            const uint32_t sh = uint32_t(byte & 3u) * 8u + (DT == SPLITZIP_BF16 ? 7u : 2u);
            const uint32_t field = (DT == SPLITZIP_BF16 ? 0xFFu : 0x1Fu) << sh;
            if ((byte | 3u) < a.n * EB) {
                unsigned int* w = reinterpret_cast<unsigned int*>(a.out + (byte & ~uint64_t(3)));
                atomicAnd(w, ~field);
                atomicOr(w, e << sh);
            } else if constexpr (DT == SPLITZIP_BF16) {
                uint16_t* p = reinterpret_cast<uint16_t*>(a.out + byte);
                *p = uint16_t((*p & 0x807Fu) | (e << 7));
            } else {
                a.out[byte] = uint8_t((a.out[byte] & 0x83u) | (e << 2));
            }
        }
    }
    if (bad) abl_report(a.status, SPLITZIP_ERR_CORRUPT);
    }  // ok_s
    __syncthreads();  // before thread 0 reads the next chunk's index entry into shared memory
    }  // chunks
}

template <int DT>
void abl_launch_write(const AblEncodeArgs& a, unsigned grid, cudaStream_t s) {
    if (a.variant == 0)
        abl_write_kernel<DT, 0><<<grid, kAblThreads, 0, s>>>(a);
    else if (a.variant == 1)
        abl_write_kernel<DT, 1><<<grid, kAblThreads, 0, s>>>(a);
    else
        abl_write_kernel<DT, 2><<<grid, kAblThreads, 0, s>>>(a);
}

template <int DT>
void abl_launch_decode(const AblDecodeArgs& a, unsigned grid, cudaStream_t s) {
    if (a.variant == 0)
        abl_decode_kernel<DT, 0><<<grid, kAblThreads, 0, s>>>(a);
    else if (a.variant == 1)
        abl_decode_kernel<DT, 1><<<grid, kAblThreads, 0, s>>>(a);
    else
        abl_decode_kernel<DT, 2><<<grid, kAblThreads, 0, s>>>(a);
}

bool abl_geometry_ok(int dtype, uint32_t chunk, int variant) {
    return (dtype == SPLITZIP_BF16 || dtype == SPLITZIP_FP8_E5M2) && variant >= 0 && variant <= 2 &&
           chunk >= kMinChunk && chunk <= kMaxChunk && (chunk & (chunk - 1u)) == 0;
}

bool abl_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1u)) == 0; }

int abl_fail_cuda() {
    cudaGetLastError();
    return SPLITZIP_ERR_CUDA;
}

}  // namespace
}  // namespace splitzip

using namespace splitzip;

extern "C" int splitzip_ablation_max_size(uint64_t n, int dtype, uint32_t chunk_elems, int variant,
                                          uint64_t* out_bytes) {
    if (!out_bytes || !abl_geometry_ok(dtype, chunk_elems, variant)) return SPLITZIP_ERR_INVALID_ARG;
    if (n > (uint64_t(1) << 48) || (n + chunk_elems - 1u) / chunk_elems > 0x7FFFFFFFull)
        return SPLITZIP_ERR_UNSUPPORTED;
    *out_bytes = abl_layout(n, dtype, chunk_elems, variant, n).size;
    return SPLITZIP_OK;
}

extern "C" int splitzip_ablation_encode(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                                        uint32_t chunk_elems, int variant, void* d_out, uint64_t out_capacity,
                                        uint64_t* d_out_size, int* d_status, cudaStream_t stream) {
    uint64_t need = 0;
    int st = splitzip_ablation_max_size(n, dtype, chunk_elems, variant, &need);
    if (st != SPLITZIP_OK) return st;
    if ((n > 0 && (!d_in || !abl_aligned(d_in, 16))) || !d_out || !abl_aligned(d_out, 16) || !d_out_size ||
        !abl_aligned(d_out_size, 8) || !d_status || !abl_aligned(d_status, 4) || !cb || cb->dtype != dtype)
        return SPLITZIP_ERR_INVALID_ARG;
    if (out_capacity < need) return SPLITZIP_ERR_CAPACITY;
    // codebook: the first k exponents distinct and in range, the rest zero
    AblEncodeArgs a;
    std::memset(a.code_of, kNoCode, sizeof(a.code_of));
    const uint32_t k = abl_codes(variant), bins = dtype == SPLITZIP_BF16 ? 256u : 32u;
    for (uint32_t i = 0; i < 16; ++i) {
        const uint32_t e = cb->exps[i];
        if (i >= k) {
            if (e != 0) return SPLITZIP_ERR_INVALID_ARG;
            continue;
        }
        if (e >= bins || a.code_of[e] != kNoCode) return SPLITZIP_ERR_INVALID_ARG;
        a.code_of[e] = uint8_t(i);
    }
    a.in = static_cast<const uint8_t*>(d_in);
    a.n = n;
    a.out = static_cast<uint8_t*>(d_out);
    a.out_size = d_out_size;
    a.status = d_status;
    a.chunk = chunk_elems;
    a.dtype = dtype;
    a.variant = variant;
    std::memcpy(a.codebook, cb->exps, 16);
    if (cudaMemsetAsync(d_status, 0, sizeof(int), stream) != cudaSuccess) return abl_fail_cuda();
    const unsigned C = unsigned((n + chunk_elems - 1u) / chunk_elems);
    if (C > 0) {
        if (dtype == SPLITZIP_BF16)
            abl_count_kernel<SPLITZIP_BF16><<<C, kAblThreads, 0, stream>>>(a);
        else
            abl_count_kernel<SPLITZIP_FP8_E5M2><<<C, kAblThreads, 0, stream>>>(a);
    }
    abl_index_kernel<<<1, kAblThreads, 0, stream>>>(a);
    if (C > 0) {
        if (dtype == SPLITZIP_BF16)
            abl_launch_write<SPLITZIP_BF16>(a, C, stream);
        else
            abl_launch_write<SPLITZIP_FP8_E5M2>(a, C, stream);
    }
    return cudaGetLastError() == cudaSuccess ? SPLITZIP_OK : abl_fail_cuda();
}

extern "C" int splitzip_ablation_decode(const void* d_in, uint64_t in_bytes, void* d_out, uint64_t n, int dtype,
                                        int variant, int* d_status, cudaStream_t stream) {
    if (!abl_geometry_ok(dtype, kMinChunk, variant) || !d_in || !abl_aligned(d_in, 16) || !d_status ||
        !abl_aligned(d_status, 4) || (n > 0 && (!d_out || !abl_aligned(d_out, 16))))
        return SPLITZIP_ERR_INVALID_ARG;
    if (n > (uint64_t(1) << 48)) return SPLITZIP_ERR_UNSUPPORTED;
    if (in_bytes < kHeaderBytes) return SPLITZIP_ERR_CORRUPT;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return abl_fail_cuda();
    if (cudaMemsetAsync(d_status, 0, sizeof(int), stream) != cudaSuccess) return abl_fail_cuda();
    if (n == 0) return SPLITZIP_OK;
    AblDecodeArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.in_bytes = in_bytes;
    a.out = static_cast<uint8_t*>(d_out);
    a.n = n;
    a.status = d_status;
    a.dtype = dtype;
    a.variant = variant;
    // persistent: 8 CTAs of 256 threads per SM, never more CTAs than the
    // smallest chunk size allows chunks
    const uint64_t most = (n + kMinChunk - 1u) / kMinChunk;
    const unsigned grid = unsigned(std::min<uint64_t>(most, uint64_t(sms) * 8u));
    if (dtype == SPLITZIP_BF16)
        abl_launch_decode<SPLITZIP_BF16>(a, grid, stream);
    else
        abl_launch_decode<SPLITZIP_FP8_E5M2>(a, grid, stream);
    return cudaGetLastError() == cudaSuccess ? SPLITZIP_OK : abl_fail_cuda();
}
