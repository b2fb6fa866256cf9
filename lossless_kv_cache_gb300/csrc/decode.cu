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
// Persistent grid: each CTA loops over its chunks.  A producer warp streams
// the chunks' nibble and sign|mantissa bytes into a shared-memory ring (one or two stages)
// with bulk copies (TMA); eight consumer warps decode from shared memory and
// write 16-byte streaming stores.  Every CTA validates the header first; each
// chunk validates its index entry and each escape record, and errors go to the
// status word without any out-of-bounds access.
#include "decode_core.cuh"
#include "splitzip_internal.cuh"
#include "tma_pipeline.cuh"

namespace splitzip {
namespace {

// Decode work: each CTA walks its chunks (c = blockIdx.x, +gridDim.x, ...)
// as a sequence of sub-tiles of up to kSub elements.  Producer and consumers
// walk the same sequence, so sub-tile i always lives in stage i % kStages.
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kBlock = kConsumers + 32;  // + one producer warp
// Sub-tile size, ring depth and resident CTAs per SM, measured on the
// 2.1 G-element BF16 and 4.3 G-element E5M2 caches: both run fastest with
// 16,384-element sub-tiles at 3 CTAs per SM, BF16 (24 KB a sub-tile) with a
// single stage, E5M2 (14 KB) with two; the other CTAs of the SM keep its
// copies in flight while one decodes (BF16 1.21 ms vs 1.27 ms with four
// 8,192-element stages at 2 CTAs; E5M2 1.44 ms vs 1.63 ms with four
// 8,192-element stages, 1.44 ms at 32,768 elements and 2 CTAs).
// FP16 (8 nibble + 22 sign|mantissa KB a sub-tile) takes BF16's single stage.
template <int DT> constexpr int kStages = DT == SPLITZIP_FP8_E5M2 ? 2 : 1;
template <int DT> constexpr uint32_t kSub = 16384u;
template <int DT> constexpr uint32_t kNibCap = kSub<DT> / 2 + 32;  // + room for a 16-byte window shift
// sign|mantissa bytes of a sub-tile: BF16 one per element, E5M2 3 and FP16
// 11 per 8 elements
template <int DT> constexpr uint32_t kSmCap =
    (DT == SPLITZIP_BF16 ? kSub<DT> : (DT == SPLITZIP_FP16 ? 11 : 3) * kSub<DT> / 8) + 32;
template <int DT> constexpr uint32_t kStageBytes = (kNibCap<DT> + kSmCap<DT> + 127u) & ~127u;
template <int DT> constexpr uint32_t kRingBytes = kStages<DT> * kStageBytes<DT>;
// A chunk's escape records are brought into shared memory with one bulk copy
// when they fit (at most kRecCap records: BF16 8,192 = 12.5 % of a 65,536-element
// chunk, E5M2 7,680 = 11.7 %, within each dtype's shared-memory budget at its
// CTAs per SM);
// a chunk with more escapes reads them from the escape stream instead.  Either
// way each sub-tile is patched right after its stores, while its lines are
// still in L2.
template <int DT> constexpr uint32_t kRecCap = DT == SPLITZIP_BF16 ? 8192u : DT == SPLITZIP_FP16 ? 6144u : 7680u;
// resident CTAs per SM the kernel is compiled for (register budget)
template <int DT> constexpr int kDecodeMinBlocks = 3;
// per buffer: 3 bytes a record + room for a 16-byte window shift
template <int DT> constexpr uint32_t kRecBytes = 3 * kRecCap<DT> + 32;
// dynamic shared memory: the sub-tile ring, then two record buffers
template <int DT> constexpr uint32_t kDecodeSmem = kRingBytes<DT> + 2 * kRecBytes<DT>;
// the CTAs of one SM share its 228 KB (each also takes ~1 KB static + 1 KB reserved)
static_assert(kDecodeMinBlocks<SPLITZIP_BF16> * (kDecodeSmem<SPLITZIP_BF16> + 2048) <= 228 * 1024, "smem");
static_assert(kDecodeMinBlocks<SPLITZIP_FP8_E5M2> * (kDecodeSmem<SPLITZIP_FP8_E5M2> + 2048) <= 228 * 1024, "smem");
static_assert(kDecodeMinBlocks<SPLITZIP_FP16> * (kDecodeSmem<SPLITZIP_FP16> + 3072) <= 228 * 1024, "smem");

struct SubTile {
    Window nib, sm;
};

template <int DT>
__device__ __forceinline__ SubTile subtile_windows(const uint8_t* nibbles, const uint8_t* signmant, uint64_t g,
                                                   uint32_t cnt) {
    SubTile t;
    t.nib = window_of(nibbles + g / 2, (cnt + 1u) / 2u);
    if constexpr (DT == SPLITZIP_BF16)
        t.sm = window_of(signmant + g, cnt);
    else if constexpr (DT == SPLITZIP_FP16)
        t.sm = window_of(signmant + g / 8u * 11u, 11u * ((cnt + 7u) / 8u));
    else
        t.sm = window_of(signmant + g / 8u * 3u, 3u * ((cnt + 7u) / 8u));
    return t;
}

// Dense decode of one sub-tile from shared memory; results go straight to
// global memory with 16-byte streaming stores.  Unit u (UE elements) of the
// sub-tile is decoded by thread u mod 256 in round u / 256.
template <int DT, bool PAGED>
__device__ __forceinline__ void decode_subtile(const uint8_t* nb, const uint8_t* sb, const OutMap<PAGED>& om,
                                               uint64_t g, uint32_t cnt, int tid, const uint16_t* lut2,
                                               const uint32_t* lut4) {
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    constexpr uint32_t UE = DT == SPLITZIP_FP8_E5M2 ? 16u : 8u;
    const uint32_t units = (cnt + UE - 1u) / UE;
    const uint32_t rounds = (units + kConsumers - 1u) / kConsumers;
    // paged output: a sub-tile that lies in one page takes one page-table
    // lookup for all its units (the same decision in every thread)
    [[maybe_unused]] bool one_page = false, page_ok = true;
    [[maybe_unused]] uint64_t page_off = 0;
    if constexpr (PAGED) {
        if (cnt > 0 && (g >> om.shift) == ((g + cnt - 1u) >> om.shift)) {
            one_page = true;
            page_ok = om.at(g, EB, page_off);
        }
    }
    auto out_at = [&](uint32_t e, uint64_t& off) -> bool {
        if constexpr (PAGED) {
            if (one_page) {
                off = page_off + uint64_t(e) * EB;
                return page_ok;
            }
        }
        return om.at(g + e, EB, off);
    };
#pragma unroll 2
    for (uint32_t k = 0; k < rounds; ++k) {
        const uint32_t u = k * kConsumers + uint32_t(tid);
        const uint32_t e = UE * u;
        if (e + UE <= cnt) {
            uint4 o;
            if constexpr (DT == SPLITZIP_BF16) {
                const uint32_t nib = *reinterpret_cast<const uint32_t*>(nb + e / 2);
                const uint2 sm = *reinterpret_cast<const uint2*>(sb + e);
                o = decode_unit_bf16(nib, sm, lut2);
            } else if constexpr (DT == SPLITZIP_FP16) {
                // 11 bytes of s11 per unit, at any byte of the stage
                const uint32_t nib = *reinterpret_cast<const uint32_t*>(nb + e / 2);
                uint32_t f0, f1, f2;
                load96(sb + 11u * u, f0, f1, f2);
                o = decode_unit_fp16(nib, f0, f1, f2, lut4);
            } else {
                // 6 bytes of s3 per unit, 2-byte aligned in the stage
                const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sb + 6u * u);
                const uint2 nib = *reinterpret_cast<const uint2*>(nb + e / 2);
                const uint32_t s3lo = uint32_t(s16[0]) | (uint32_t(s16[1]) << 16), s3hi = s16[2];
                o = decode_unit_e5m2(nib, s3lo, s3hi, lut2);
            }
            uint64_t off;
            if (out_at(e, off)) __stcs(reinterpret_cast<uint4*>(om.base + off), o);
        } else if (e < cnt) {
            const uint32_t valid = cnt - e;
            uint4 o;
            if constexpr (DT == SPLITZIP_BF16) {
                uint32_t nib = 0;
                uint64_t smw = 0;
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nib |= uint32_t(nb[e / 2 + b]) << (8u * b);
                for (uint32_t b = 0; b < valid; ++b) smw |= uint64_t(sb[e + b]) << (8u * b);
                o = decode_unit_bf16(nib, make_uint2(uint32_t(smw), uint32_t(smw >> 32)), lut2);
            } else if constexpr (DT == SPLITZIP_FP16) {
                uint32_t nib = 0, f[3] = {0u, 0u, 0u};
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nib |= uint32_t(nb[e / 2 + b]) << (8u * b);
                const uint8_t* s8 = sb + 11u * u;
                for (uint32_t b = 0; b < 11u; ++b) f[b >> 2] |= uint32_t(s8[b]) << (8u * (b & 3u));
                o = decode_unit_fp16(nib, f[0], f[1], f[2], lut4);
            } else {
                uint64_t nw = 0, sw = 0;
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nw |= uint64_t(nb[e / 2 + b]) << (8u * b);
                const uint8_t* s8 = sb + 6u * u;
                for (uint32_t b = 0; b < 3u * ((valid + 7u) / 8u); ++b) sw |= uint64_t(s8[b]) << (8u * b);
                o = decode_unit_e5m2(make_uint2(uint32_t(nw), uint32_t(nw >> 32)), uint32_t(sw), uint32_t(sw >> 32),
                                     lut2);
            }
            uint64_t off;
            if (out_at(e, off)) {
                for (uint32_t b = 0; b < valid; ++b) {
                    const uint32_t q = EB == 2 ? b >> 1 : b >> 2;
                    const uint32_t w = q == 0 ? o.x : q == 1 ? o.y : q == 2 ? o.z : o.w;
                    if constexpr (EB == 2)
                        reinterpret_cast<uint16_t*>(om.base + off)[b] = uint16_t(w >> (16u * (b & 1u)));
                    else
                        (om.base + off)[b] = uint8_t(w >> (8u * (b & 3u)));
                }
            }
        }
    }
}

template <int DT, bool PAGED>
__global__ void __launch_bounds__(kBlock, kDecodeMinBlocks<DT>) decode_kernel(const DecodeArgs a) {
    extern __shared__ __align__(128) uint8_t stages[];
    __shared__ __align__(8) uint64_t full_bar[kStages<DT>];
    __shared__ __align__(8) uint64_t empty_bar[kStages<DT>];
    __shared__ __align__(8) uint64_t rec_full[2];
    __shared__ __align__(8) uint64_t rec_empty[2];
    // record buffer b (0, 1) of the double buffer
    auto rec_buf = [&](uint32_t b) { return stages + kRingBytes<DT> + b * kRecBytes<DT>; };
    __shared__ uint32_t rec_offset[2];  // window shift of the records in rec_buf, or kNoRecords
    __shared__ Header hdr;
    __shared__ int header_ok;
    // nibble byte -> (exponent of low code) | (exponent of high code) << 8,
    // both shifted left by 2 for E5M2 (their place in the output byte)
    __shared__ uint16_t lut2[256];
    // FP16: nibble byte -> (exponent of low code) << 10 | (of high code) << 26
    __shared__ uint32_t lut4[DT == SPLITZIP_FP16 ? 256 : 1];
    constexpr uint32_t kNoRecords = 0xFFFFFFFFu;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        header_ok = read_header(a, hdr);
        if (!header_ok) report(a.status, SPLITZIP_ERR_CORRUPT);
        for (int s = 0; s < kStages<DT>; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumerWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&rec_full[b], 1);
            mbar_init(&rec_empty[b], kConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    if (!header_ok) return;
    for (int b = tid; b < 256; b += kBlock) {
        if constexpr (DT == SPLITZIP_FP16)
            lut4[b] = (uint32_t(hdr.codebook[b & 15]) << 10) | (uint32_t(hdr.codebook[b >> 4]) << 26);
        else
            lut2[b] = uint16_t((hdr.codebook[b & 15] | (hdr.codebook[b >> 4] << 8)) << (DT == SPLITZIP_BF16 ? 0 : 2));
    }
    __syncthreads();

    const uint8_t* in = a.in;
    const Layout L = hdr.L;
    const uint8_t* nibbles = in + L.nibble_off;
    const uint8_t* signmant = in + L.signmant_off;
    const uint64_t* offsets = reinterpret_cast<const uint64_t*>(in + L.index_off);
    const uint32_t* counts = reinterpret_cast<const uint32_t*>(in + L.counts_off);
    const uint8_t* records = in + L.escrec_off;  // 3 bytes each: position u16 LE, exponent
    const uint64_t chunk = hdr.chunk, C = hdr.n_chunks, E = hdr.E;
    const uint32_t EBo = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    const OutMap<PAGED> om{static_cast<uint8_t*>(a.out),
                           PAGED ? (a.pool_pages << a.page_shift) * EBo : a.n * EBo,
                           a.pages, a.pool_pages, a.page_shift, a.status};
    const uint32_t sub = uint32_t(min(uint64_t(kSub<DT>), chunk));

    if (warp == kConsumerWarps) {
        // ---- producer: per chunk its escape records (when they fit), then
        // its sub-tiles, streamed into shared memory ----
        if (lane != 0) return;
        uint32_t it = 0, ci = 0;
        for (uint64_t c = blockIdx.x; c < C; c += gridDim.x, ++ci) {
            const uint64_t base = c * chunk;
            const uint32_t len = uint32_t(min(chunk, a.n - base));
            const uint32_t rb = ci & 1u;
            if (ci >= 2 && !mbar_wait(&rec_empty[rb], ((ci >> 1) - 1) & 1u)) report(a.status, SPLITZIP_ERR_TIMEOUT);
            const uint64_t off = offsets[c], cnt = counts[c];
            // only a range that lies inside the escape stream is copied, and
            // only when its 16-byte-aligned window stays inside the caller's
            // buffer (the stream ends the container unpadded); the consumers
            // check the index entry in full
            const Window w = window_of(records + 3 * min(off, E), 3 * min(cnt, uint64_t(kRecCap<DT>)));
            if (cnt > 0 && cnt <= kRecCap<DT> && cnt <= len && off <= E && cnt <= E - off &&
                w.src + w.bytes <= in + a.in_bytes) {
                rec_offset[rb] = w.offset;
                mbar_arrive_expect_tx(&rec_full[rb], w.bytes);
                bulk_load(rec_buf(rb), w.src, w.bytes, &rec_full[rb]);
            } else {
                rec_offset[rb] = cnt == 0 ? 0u : kNoRecords;
                mbar_arrive(&rec_full[rb]);
            }
            for (uint32_t s0 = 0; s0 < len; s0 += sub, ++it) {
                const uint32_t stage = it % kStages<DT>, use = it / kStages<DT>;
                if (use > 0 && !mbar_wait(&empty_bar[stage], (use - 1) & 1u)) report(a.status, SPLITZIP_ERR_TIMEOUT);
                const SubTile t = subtile_windows<DT>(nibbles, signmant, base + s0, min(sub, len - s0));
                uint8_t* dst = stages + stage * kStageBytes<DT>;
                mbar_arrive_expect_tx(&full_bar[stage], t.nib.bytes + t.sm.bytes);
                bulk_load(dst, t.nib.src, t.nib.bytes, &full_bar[stage]);
                bulk_load(dst + kNibCap<DT>, t.sm.src, t.sm.bytes, &full_bar[stage]);
            }
        }
        bool ok = drain_stages(full_bar, kStages<DT>, it);
        ok &= drain_stages(rec_full, 2, ci);
        if (!ok) report(a.status, SPLITZIP_ERR_TIMEOUT);
        return;
    }

    // ---- consumers: dense decode per sub-tile, each sub-tile patched right
    // after its stores ----
    uint32_t it = 0, ci = 0;
    for (uint64_t c = blockIdx.x; c < C; c += gridDim.x, ++ci) {
        const uint64_t base = c * chunk;
        const uint32_t len = uint32_t(min(chunk, a.n - base));
        const uint32_t rb = ci & 1u;
        const uint64_t off = offsets[c];
        const uint64_t cnt = counts[c];
        const uint64_t expect_off = c == 0 ? 0 : offsets[c - 1] + counts[c - 1];
        const bool index_ok = off == expect_off && cnt <= len && off <= E && cnt <= E - off &&
                              (c + 1 < C || off + cnt == E);
        if (!mbar_wait(&rec_full[rb], (ci >> 1) & 1u)) report(a.status, SPLITZIP_ERR_TIMEOUT);
        const uint32_t shift = rec_offset[rb];
        // the chunk's records: in shared memory when they fit, else read from
        // the escape stream; either way each sub-tile is patched right after
        // its stores (the same decision in every consumer)
        const bool in_smem = index_ok && shift != kNoRecords;
        const bool patch = index_ok && cnt > 0;
        uint32_t cursor = 0;  // records of this chunk already applied
        bool bad = false;
        // records are sorted, so a sub-tile's are the next ones with position
        // < end; the counting barrier also makes the sub-tile's stores visible
        // to every consumer
        auto patch_upto = [&](const uint8_t* recs, uint32_t end) {
            while (true) {
                const uint32_t i = cursor + tid;
                const bool mine = i < cnt && rec_pos(recs + 3 * i) < end;
                const uint32_t n_in = named_barrier_popc(1, kConsumers, mine);
                if (mine) {
                    const int64_t prev = i == 0 ? -1 : int64_t(rec_pos(recs + 3 * (i - 1)));
                    bad |= !patch_one<DT, PAGED>(om, base, len, prev, rec_pos(recs + 3 * i), recs[3 * i + 2]);
                }
                cursor += n_in;
                if (n_in < kConsumers) break;
            }
        };
        for (uint32_t s0 = 0; s0 < len; s0 += sub, ++it) {
            const uint32_t stage = it % kStages<DT>, use = it / kStages<DT>;
            const uint32_t n_sub = min(sub, len - s0);
            if (!mbar_wait(&full_bar[stage], use & 1u)) report(a.status, SPLITZIP_ERR_TIMEOUT);
            const SubTile t = subtile_windows<DT>(nibbles, signmant, base + s0, n_sub);
            const uint8_t* src = stages + stage * kStageBytes<DT>;
            decode_subtile<DT, PAGED>(src + t.nib.offset, src + kNibCap<DT> + t.sm.offset, om, base + s0, n_sub, tid,
                                      lut2, lut4);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[stage]);
            if (!patch) continue;
            if (in_smem)
                patch_upto(rec_buf(rb) + shift, s0 + n_sub);
            else
                patch_upto(records + 3 * off, s0 + n_sub);
        }
        if (patch && cursor != cnt) bad = true;  // a record outside the chunk or out of order
        if (bad) report(a.status, SPLITZIP_ERR_CORRUPT);
        if (!index_ok && tid == 0) report(a.status, SPLITZIP_ERR_CORRUPT);
        __syncwarp();
        if (lane == 0) mbar_arrive(&rec_empty[rb]);
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t s) {
    const bool paged = a.pages != nullptr;
    if (a.dtype == SPLITZIP_BF16) {
        if (paged)
            decode_kernel<SPLITZIP_BF16, true><<<grid, kBlock, kDecodeSmem<SPLITZIP_BF16>, s>>>(a);
        else
            decode_kernel<SPLITZIP_BF16, false><<<grid, kBlock, kDecodeSmem<SPLITZIP_BF16>, s>>>(a);
    } else if (a.dtype == SPLITZIP_FP16) {
        if (paged)
            decode_kernel<SPLITZIP_FP16, true><<<grid, kBlock, kDecodeSmem<SPLITZIP_FP16>, s>>>(a);
        else
            decode_kernel<SPLITZIP_FP16, false><<<grid, kBlock, kDecodeSmem<SPLITZIP_FP16>, s>>>(a);
    } else {
        if (paged)
            decode_kernel<SPLITZIP_FP8_E5M2, true><<<grid, kBlock, kDecodeSmem<SPLITZIP_FP8_E5M2>, s>>>(a);
        else
            decode_kernel<SPLITZIP_FP8_E5M2, false><<<grid, kBlock, kDecodeSmem<SPLITZIP_FP8_E5M2>, s>>>(a);
    }
    return cudaGetLastError();
}

// Also raises the kernels' dynamic shared-memory limit (once per device, for
// the contiguous and the paged instances); the occupancy is the contiguous
// instance's.
cudaError_t occupancy_decode(int* blocks_per_sm, int dtype) {
    const bool bf16 = dtype == SPLITZIP_BF16, fp16 = dtype == SPLITZIP_FP16;
    auto k = bf16 ? decode_kernel<SPLITZIP_BF16, false>
             : fp16 ? decode_kernel<SPLITZIP_FP16, false> : decode_kernel<SPLITZIP_FP8_E5M2, false>;
    auto kp = bf16 ? decode_kernel<SPLITZIP_BF16, true>
              : fp16 ? decode_kernel<SPLITZIP_FP16, true> : decode_kernel<SPLITZIP_FP8_E5M2, true>;
    const int smem = int(bf16 ? kDecodeSmem<SPLITZIP_BF16>
                         : fp16 ? kDecodeSmem<SPLITZIP_FP16> : kDecodeSmem<SPLITZIP_FP8_E5M2>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kBlock, smem);
}

}  // namespace splitzip
