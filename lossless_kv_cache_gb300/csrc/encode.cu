// SplitZip encode kernels for sm_103a.
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip", "Encoding strategy": each element's
// exponent goes through the offline-calibrated Top-16 codebook to a 4-bit code,
// two codes per byte ("Fixed-length coding"); sign and mantissa are kept raw
// ("Sign/mantissa preservation"); an exponent outside the codebook becomes a
// (16-bit position, 8-bit exponent) escape record ("Escape stream").
//
// Four kernels, no inter-block waits:
//   encode_kernel (the streaming pass, persistent CTAs of 8 consumer warps +
//     1 producer warp): the producer streams each of the CTA's 16 KB tiles
//     into a shared-memory ring (BF16 8 stages at one CTA per SM, E5M2 and
//     FP16 4 stages at two) with tensor-map copies (TMA,
//     cp.async.bulk.tensor, 128-byte swizzle, mbarrier); every consumer
//     thread owns 64 contiguous bytes of the tile.  Per element it does one
//     shared-memory lookup in a table for the element's position within its
//     group of four; the table entries already sit at their final bit
//     positions, so the sum of four entries is the group's two nibble bytes,
//     its escape flags and (E5M2) its packed 3-bit sign|mantissa values.  The
//     nibble and sign|mantissa streams go out with 16-byte stores (FP16's
//     11-bit stream by way of a per-warp shared-memory transpose); a warp
//     scan orders the warp's escapes, each thread writes its own contiguously
//     into the warp's region of the tile's staging slot after those of the
//     lower lanes, and the warp's count goes to the workspace; no
//     synchronisation between the warps.
//   encode_group_kernel (one CTA per group of 256 tiles): the group's total.
//   encode_index_kernel (one CTA per group of 256 tiles): the sum of the
//     earlier groups' totals plus a block scan of the group's tile counts give
//     every tile's first record index; the CTA writes them and the index
//     entries of the group's chunks; the last group writes E and the size.
//   encode_records_kernel (a warp per 4 tiles): moves every tile's staged
//     records to their place in the escape stream.
// The three short kernels are launched with programmatic stream
// serialization: each is scheduled while its predecessor drains (the
// streaming kernel lets it once every CTA has issued its last copy) and waits
// in griddepcontrol.wait for that grid to complete before it reads its
// results (BF16 cache encode 1.327 -> 1.305 ms, same-box timing).
#include <type_traits>

#include "encode_core.cuh"
#include "splitzip_internal.cuh"
#include "tma_pipeline.cuh"

namespace splitzip {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kConsumerWarps = int(kEncodeWarps);
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kBlock = kConsumers + 32;  // + one producer warp
constexpr uint32_t kStageBytes = kTileBytes;
// Ring depth and resident CTAs per SM (register budget) per dtype, measured on
// the 2.1 G-element BF16 and 4.3 G-element E5M2 caches: BF16 runs fastest as
// one CTA per SM with an 8-stage ring (1.18 ms; 1.25-1.28 ms at 2 or 3 CTAs),
// E5M2 with 2 CTAs of 4 stages (1.50 ms; 1.84 ms at one CTA).
// FP16 (more integer work per element than BF16: the 11-bit sign|mantissa
// packing) runs fastest with E5M2's shape: 2 CTAs of 4 stages measured 6.7 %
// faster than BF16's one CTA of 8 (3 CTAs of 3 stages: 3.7 %).
template <int DT> constexpr int kStages = DT == SPLITZIP_BF16 ? 8 : 4;
template <int DT> constexpr int kMinBlocks = DT == SPLITZIP_BF16 ? 1 : 2;
// + room to align the ring to 1024 bytes, which the 128-byte swizzle needs
template <int DT> constexpr uint32_t kEncodeSmem = kStages<DT> * kStageBytes + 1024;
constexpr int kFinishThreads = kGroupTiles;  // one thread per tile of the group
static_assert(kConsumers * kThreadBytes == kTileBytes, "one tile = 64 bytes per consumer thread");

template <int DT>
__global__ void __launch_bounds__(kBlock, kMinBlocks<DT>)
    encode_kernel(const __grid_constant__ EncodeArgs a, const __grid_constant__ CUtensorMap map,
                  const __grid_constant__ EncodeLut lut) {
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    using Out = ThreadOut<DT>;
    constexpr uint32_t TE = Out::kElems;  // elements per consumer thread per tile
    constexpr int kStages = splitzip::kStages<DT>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(16) uint32_t tab[4 * 256];
    __shared__ uint8_t code_s[256];  // exponent -> code | kEscapeFlag
    __shared__ uint8_t cb_s[16];     // code -> exponent (the header's codebook)
    // FP16: each consumer warp's 1,408 sign|mantissa bytes of a full tile
    __shared__ __align__(16) uint32_t fp16_run[DT == SPLITZIP_FP16 ? kConsumerWarps : 1][352];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the ring starts on a 1024-byte boundary of the shared window
    uint8_t* ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    if (a.dev_codebook) {
        // a codebook in device memory (online calibration): checked here, on
        // the GPU (its dtype, every exponent in range, all distinct); a bad
        // one is reported and leaves the output unspecified
        for (int i = tid; i < 256; i += kBlock) code_s[i] = kEscapeFlag;
        if (tid < 16) cb_s[tid] = a.dev_codebook[1 + tid];
        __syncthreads();
        if (tid == 0) {
            bool ok = a.dev_codebook[0] == uint8_t(a.dtype);
            for (int k = 0; k < 16; ++k) {
                const uint32_t e = cb_s[k];
                ok &= e < (DT == SPLITZIP_BF16 ? 256u : 32u) && code_s[e] == kEscapeFlag;
                code_s[e] = uint8_t(k);
            }
            if (!ok) report(a.error, SPLITZIP_ERR_INVALID_ARG);
        }
    } else {
        for (int i = tid; i < 256; i += kBlock) code_s[i] = lut.code[i];
        if (tid < 16) cb_s[tid] = a.codebook[tid];
    }
    __syncthreads();
    for (int i = tid; i < 4 * 256; i += kBlock) tab[i] = table_entry(DT, i >> 8, uint32_t(i & 255), code_s);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], kConsumerWarps);
        }
        mbar_init_fence();
        if (blockIdx.x == 0)
            write_header_and_padding(a.out, a.dtype, a.n, a.chunk_elems, a.n_chunks, cb_s, a.out_size);
    }
    __syncthreads();

    const uint8_t* in = static_cast<const uint8_t*>(a.in);
    const uint32_t tile_bytes = a.tile_elems * EB;
    // ---- the producer warp ----
    if constexpr (DT == SPLITZIP_BF16) {
        // BF16, bound by HBM, is sensitive to its producer's pace: paged input
        // gets the page indices loaded 32 tiles ahead by the whole warp (a
        // one-tile lookahead whose check waited on the load cost paged BF16
        // 9 %), and contiguous input a loop with no page lookup at all.  E5M2
        // and FP16, whose consumers are bound by integer work, measured 0.5-1 %
        // slower with the warp-wide lookup and keep the single-lane producer.
        if (warp == kConsumerWarps && a.pages) {
            // ---- producer warp, paged input: lane 0 streams the CTA's tiles
            // (blockIdx.x + k * gridDim.x) from the pool; the whole warp loads the
            // page indices of the CTA's tiles 32 to 63 tiles ahead, so lane 0
            // never waits on a page-table load ----
            const uint64_t G = gridDim.x;
            auto raw_page = [&](uint64_t t) -> int32_t {  // checked where it is used
                return t < a.n_tiles ? a.pages[t >> a.page_tile_shift] : 0;
            };
            // page of tile (batch + lane) of this and of the next batch of 32
            int32_t pg_cur = raw_page(blockIdx.x + uint64_t(lane) * G);
            int32_t pg_next = raw_page(blockIdx.x + uint64_t(32 + lane) * G);
            uint32_t it = 0;
            for (uint64_t t = blockIdx.x; t < a.n_tiles; t += G, ++it) {
                const uint32_t stage = it % kStages, use = it / kStages, j = it & 31u;
                if (j == 0 && it > 0) {
                    pg_cur = pg_next;
                    pg_next = raw_page(t + uint64_t(32 + lane) * G);
                }
                // the pool tile that holds tile t; a page index outside the pool
                // is reported and read as page 0, inside the pool
                int64_t p = __shfl_sync(kFull, pg_cur, int(j));
                if (p < 0 || uint64_t(p) >= a.pool_pages) {
                    if (lane == 0) report(a.error, SPLITZIP_ERR_INVALID_ARG);
                    p = 0;
                }
                const uint64_t src =
                    (uint64_t(p) << a.page_tile_shift) | (t & ((uint64_t(1) << a.page_tile_shift) - 1u));
                if (use > 0 && !mbar_wait(&empty_bar[stage], (use - 1) & 1u) && lane == 0)
                    report(a.error, SPLITZIP_ERR_TIMEOUT);
                if (lane == 0) {
                    const uint64_t tb = src * tile_bytes;
                    if (tb < a.tensor_bytes) {
                        mbar_arrive_expect_tx(&full_bar[stage], a.box_bytes);
                        tensor_load_2d(ring + stage * kStageBytes, &map, int32_t((tb & 127u) / EB), int32_t(tb >> 7),
                                       &full_bar[stage]);
                    } else {
                        mbar_arrive(&full_bar[stage]);  // the consumers read this tile from global memory
                    }
                }
                __syncwarp();
            }
            if (lane == 0) {
                // every copy of this CTA is issued: the call's next kernel may be
                // scheduled (it waits for this grid to complete before it reads)
                asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
                if (!drain_stages(full_bar, kStages, it)) report(a.error, SPLITZIP_ERR_TIMEOUT);
            }
            return;
        }

        if (warp == kConsumerWarps) {
            // ---- producer, contiguous input: stream the CTA's tiles
            // (blockIdx.x + k * gridDim.x) ----
            if (lane != 0) return;
            uint32_t it = 0;
            for (uint64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++it) {
                const uint32_t stage = it % kStages, use = it / kStages;
                if (use > 0 && !mbar_wait(&empty_bar[stage], (use - 1) & 1u)) report(a.error, SPLITZIP_ERR_TIMEOUT);
                const uint64_t tb = t * tile_bytes;
                if (tb < a.tensor_bytes) {
                    mbar_arrive_expect_tx(&full_bar[stage], a.box_bytes);
                    tensor_load_2d(ring + stage * kStageBytes, &map, int32_t((tb & 127u) / EB), int32_t(tb >> 7),
                                   &full_bar[stage]);
                } else {
                    mbar_arrive(&full_bar[stage]);  // the consumers read this tile from global memory
                }
            }
            // every copy of this CTA is issued: the call's next kernel may be
            // scheduled (it waits for this grid to complete before it reads)
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            if (!drain_stages(full_bar, kStages, it)) report(a.error, SPLITZIP_ERR_TIMEOUT);
            return;
        }
    } else {
        if (warp == kConsumerWarps) {
            // ---- producer: stream the CTA's tiles (blockIdx.x + k * gridDim.x) ----
            if (lane != 0) return;
            // the pool tile that holds tile t (paged input; a page index outside
            // the pool is reported and read as page 0, inside the pool)
            auto source_tile = [&](uint64_t t) -> uint64_t {
                if (!a.pages) return t;
                int64_t p = a.pages[t >> a.page_tile_shift];
                if (p < 0 || uint64_t(p) >= a.pool_pages) {
                    report(a.error, SPLITZIP_ERR_INVALID_ARG);
                    p = 0;
                }
                return (uint64_t(p) << a.page_tile_shift) | (t & ((uint64_t(1) << a.page_tile_shift) - 1u));
            };
            uint32_t it = 0;
            uint64_t src_next = blockIdx.x < a.n_tiles ? source_tile(blockIdx.x) : 0;
            for (uint64_t t = blockIdx.x; t < a.n_tiles; t += gridDim.x, ++it) {
                const uint32_t stage = it % kStages, use = it / kStages;
                const uint64_t src = src_next;
                // the next tile's page lookup is issued before this stage's wait
                if (t + gridDim.x < a.n_tiles) src_next = source_tile(t + gridDim.x);
                if (use > 0 && !mbar_wait(&empty_bar[stage], (use - 1) & 1u)) report(a.error, SPLITZIP_ERR_TIMEOUT);
                const uint64_t tb = src * tile_bytes;
                if (tb < a.tensor_bytes) {
                    mbar_arrive_expect_tx(&full_bar[stage], a.box_bytes);
                    tensor_load_2d(ring + stage * kStageBytes, &map, int32_t((tb & 127u) / EB), int32_t(tb >> 7),
                                   &full_bar[stage]);
                } else {
                    mbar_arrive(&full_bar[stage]);  // the consumers read this tile from global memory
                }
            }
            // every copy of this CTA is issued: the call's next kernel may be
            // scheduled (it waits for this grid to complete before it reads)
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            if (!drain_stages(full_bar, kStages, it)) report(a.error, SPLITZIP_ERR_TIMEOUT);
            return;
        }
    }

    // ---- consumers: thread `tid` owns bytes [64 tid, 64 tid + 64) of a tile ----
    const Layout L0 = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    uint8_t* nibbles = a.out + L0.nibble_off;
    uint8_t* signmant = a.out + L0.signmant_off;
    const uint32_t my_byte = kThreadBytes * uint32_t(tid);
    const uint32_t my_elem = my_byte / EB;  // first element of the thread in a tile
    uint32_t piece_off[4];                  // stage offsets of the thread's four 16-byte pieces
#pragma unroll
    for (int i = 0; i < 4; ++i) piece_off[i] = swizzled(my_byte + 16u * i);

    uint32_t it = 0;
    for (uint64_t tile = blockIdx.x; tile < a.n_tiles; tile += gridDim.x, ++it) {
        const uint32_t stage = it % kStages, use = it / kStages;
        // on a time-out the tile is processed anyway (its addresses do not
        // depend on the data), so every consumer still reaches every barrier
        if (!mbar_wait(&full_bar[stage], use & 1u)) report(a.error, SPLITZIP_ERR_TIMEOUT);
        const uint64_t base = tile * a.tile_elems;
        const uint64_t rem = a.n - base;
        const uint32_t len = rem < a.tile_elems ? uint32_t(rem) : a.tile_elems;
        const uint64_t tb = base * EB;
        // bytes of this tile that the tensor-map copy delivered (paged input:
        // whole tiles inside the mapped pool, every time: staged_bytes is
        // unbounded there)
        const uint32_t in_stage =
            tb >= a.staged_bytes ? 0u : uint32_t(min(uint64_t(tile_bytes), a.staged_bytes - tb));
        const uint32_t pos0 = uint32_t(base & (a.chunk_elems - 1u));  // in-chunk position of element 0
        const uint8_t* st = ring + stage * kStageBytes;

        // Full-size tiles delivered whole take a copy of the body in which
        // every bounds test folds away at compile time; in the other copy each
        // thread handles only its `ne` elements of the tile.  The stores and
        // the record staging are written out here rather than through the
        // small-tensor encoder's helpers (store_streams, stage_records): this
        // loop is bound by its per-tile latency chain, and the helper-based
        // body measured 2.8 % slower on the BF16 cache.
        auto body = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            // elements of this thread in the tile (all TE of them in a full tile)
            const uint32_t ne = FULL ? TE : (len > my_elem ? min(len - my_elem, TE) : 0u);
            Out o;
            [[maybe_unused]] uint32_t p[8];  // E5M2 packed sign|mantissa groups
            if constexpr (DT == SPLITZIP_BF16) {
                o.mask = 0u;
            } else if constexpr (DT == SPLITZIP_FP16) {
                o.mask = 0u;
#pragma unroll
                for (int k = 0; k < 11; ++k) o.sm[k] = 0u;
            } else {
                o.mask[0] = o.mask[1] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 v;
                const uint32_t L = my_byte + 16u * i;
                if (FULL || L + 16u <= in_stage)
                    v = *reinterpret_cast<const uint4*>(st + piece_off[i]);
                else if (L < len * EB)  // past the tensor map's whole rows: read global memory
                    v = load_partial(in + tb + L, min(16u, len * EB - L));
                else
                    v = make_uint4(0u, 0u, 0u, 0u);
                if constexpr (DT == SPLITZIP_FP8_E5M2)
                    encode_piece(tab, v, i, o, p);
                else
                    encode_piece(tab, v, i, o);
            }

            // ---- nibble and sign|mantissa streams ----
            uint8_t* nb = nibbles + base / 2 + my_elem / 2;
            if constexpr (DT == SPLITZIP_BF16) {
                uint8_t* sb = signmant + base + my_elem;
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
                uint8_t* sb = signmant + (base + my_elem) / 8 * 11;
                if (FULL) {
                    // the warp's 1,408 contiguous bytes go through shared memory
                    // (a stride of 11 words is conflict-free) into 16-byte
                    // stores: eleven 4-byte stores at a 44-byte lane stride
                    // spread each warp request over ~44 sectors (FP16 cache
                    // encode 1.70 -> 1.52 ms, same-box timing)
                    __stcs(reinterpret_cast<uint4*>(nb), make_uint4(o.nib[0], o.nib[1], o.nib[2], o.nib[3]));
                    uint32_t* wb = fp16_run[warp];
#pragma unroll
                    for (int k = 0; k < 11; ++k) wb[11 * lane + k] = o.sm[k];
                    __syncwarp();
                    // the warp's run starts at byte 1,408 w of the tile's 11,264
                    uint4* dst = reinterpret_cast<uint4*>(signmant + (base + uint32_t(warp) * 32u * TE) / 8 * 11);
#pragma unroll
                    for (int i = 0; i < 3; ++i)
                        if (lane + 32 * i < 88)
                            __stcs(dst + lane + 32 * i, reinterpret_cast<const uint4*>(wb)[lane + 32 * i]);
                } else if (ne == TE) {
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
                uint8_t* sb = signmant + (base + my_elem) / 8 * 3;
                if (FULL || ne == TE) {
                    __stcs(reinterpret_cast<uint4*>(nb), make_uint4(o.nib[0], o.nib[1], o.nib[2], o.nib[3]));
                    __stcs(reinterpret_cast<uint4*>(nb) + 1, make_uint4(o.nib[4], o.nib[5], o.nib[6], o.nib[7]));
#pragma unroll
                    for (int k = 0; k < 3; ++k)
                        __stcs(reinterpret_cast<uint2*>(sb) + k, make_uint2(s3[2 * k], s3[2 * k + 1]));
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

            // ---- the warp's escapes, in element order, to its staging region ----
            uint32_t cnt;
            if constexpr (DT != SPLITZIP_FP8_E5M2)
                cnt = __popc(o.mask);
            else
                cnt = __popc(o.mask[0]) + __popc(o.mask[1]);
            uint32_t incl = cnt;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t y = __shfl_up_sync(kFull, incl, d);
                if (lane >= d) incl += y;
            }
            if (lane == 31) a.warp_counts[tile * kEncodeWarps + warp] = incl;
            // the bits of element b of this thread, and its staged record
            auto element_bits = [&](uint32_t b) -> uint32_t {
                const uint32_t e = my_elem + b;  // element of the tile
                const uint32_t B = e * EB;       // its first byte in the tile
                if (FULL || B + EB <= in_stage)
                    return EB == 2 ? uint32_t(*reinterpret_cast<const uint16_t*>(st + swizzled(B)))
                                   : uint32_t(st[swizzled(B)]);
                return EB == 2 ? uint32_t(reinterpret_cast<const uint16_t*>(in)[base + e]) : uint32_t(in[base + e]);
            };
            auto record = [&](uint32_t b, uint32_t x) -> uint32_t {
                const uint32_t exponent = DT == SPLITZIP_BF16   ? (x >> 7) & 0xFFu
                                          : DT == SPLITZIP_FP16 ? (x >> 10) & 0x1Fu
                                                                : (x >> 2) & 0x1Fu;
                return ((pos0 + my_elem + b) << 8) | exponent;
            };
            // the thread's escapes go contiguously into the warp's region of
            // the tile's slot, after the escapes of the warp's lower lanes
            if (cnt) {
                uint32_t* slot = a.staging + tile * a.tile_elems + uint32_t(warp) * (TE * 32u) + (incl - cnt);
#pragma unroll
                for (int h = 0; h < (DT == SPLITZIP_FP8_E5M2 ? 2 : 1); ++h) {
                    uint32_t m;
                    if constexpr (DT != SPLITZIP_FP8_E5M2)
                        m = o.mask;
                    else
                        m = o.mask[h];
                    // two escapes per round, so their two exponent reads overlap
                    while (m) {
                        const uint32_t b0 = 32u * h + uint32_t(__ffs(m) - 1);
                        m &= m - 1u;
                        const bool two = m != 0u;
                        const uint32_t b1 = two ? 32u * h + uint32_t(__ffs(m) - 1) : b0;
                        m &= two ? m - 1u : m;
                        const uint32_t x0 = element_bits(b0), x1 = element_bits(b1);
                        slot[0] = record(b0, x0);
                        if (two) slot[1] = record(b1, x1);
                        slot += two ? 2 : 1;
                    }
                }
            }
        };
        // (only a full-size tile gives every consumer thread its 64 bytes)
        if (in_stage == kTileBytes && len * EB == kTileBytes)
            body(std::true_type{});
        else
            body(std::false_type{});
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[stage]);  // the stage may be refilled
    }
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    return v;
}

// Escapes of one tile: the sum of its consumer warps' counts.
__device__ __forceinline__ uint32_t tile_count(const EncodeArgs& a, uint64_t t) {
    const uint4* wc = reinterpret_cast<const uint4*>(a.warp_counts + t * kEncodeWarps);
    const uint4 q0 = wc[0], q1 = wc[1];
    return q0.x + q0.y + q0.z + q0.w + q1.x + q1.y + q1.z + q1.w;
}

// One CTA per group of kGroupTiles tiles: the group's escape total (a plain
// store, so the streaming pass needs no atomics and the totals no clearing).
__global__ void __launch_bounds__(kFinishThreads) encode_group_kernel(const EncodeArgs a) {
    // launched early (programmatic dependent launch): wait for the previous
    // kernel of the call to complete and its writes to be visible, then let
    // the next one be scheduled (it waits for this one in turn)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ uint32_t warp_sum[kFinishThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint64_t t = uint64_t(blockIdx.x) * kGroupTiles + tid;
    uint32_t c = t < a.n_tiles ? tile_count(a, t) : 0u;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(kFull, c, d);
    if (lane == 0) warp_sum[warp] = c;
    __syncthreads();
    if (tid == 0) {
        uint32_t total = 0;
#pragma unroll
        for (int w = 0; w < kFinishThreads / 32; ++w) total += warp_sum[w];
        a.group_totals[blockIdx.x] = total;
    }
}

// One CTA per group of kGroupTiles tiles (groups are chunk-aligned: tiles per
// chunk is a power of two <= 8): the first record index of every tile of the
// group, the index entries of the group's chunks, and E from the last group.
__global__ void __launch_bounds__(kFinishThreads) encode_index_kernel(const EncodeArgs a) {
    // launched early (programmatic dependent launch): wait for the previous
    // kernel of the call to complete and its writes to be visible, then let
    // the next one be scheduled (it waits for this one in turn)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
    const uint32_t c = t < a.n_tiles ? tile_count(a, t) : 0u;
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
// kRecordTiles consecutive tiles: lane 8k + w holds the count and the
// exclusive prefix of consumer warp w of tile k, and every round moves one
// record of each tile per lane, so a lane keeps kRecordTiles independent
// loads in flight.
constexpr int kRecordTiles = 4;
constexpr int kRecordThreads = 256;
static_assert(kRecordTiles * kEncodeWarps == 32, "one lane per (tile, consumer warp)");

__global__ void __launch_bounds__(kRecordThreads) encode_records_kernel(const EncodeArgs a) {
    // launched early (programmatic dependent launch): wait for the previous
    // kernel of the call to complete and its writes to be visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31;
    const uint64_t t0 = (uint64_t(blockIdx.x) * (kRecordThreads / 32) + (threadIdx.x >> 5)) * kRecordTiles;
    if (t0 >= a.n_tiles) return;
    const int my_tile = lane >> 3, my_warp = lane & 7;
    const bool have = t0 + my_tile < a.n_tiles;
    const uint32_t c = have ? a.warp_counts[t0 * kEncodeWarps + lane] : 0u;
    uint32_t o = c;  // inclusive scan within each group of 8 lanes
#pragma unroll
    for (int d = 1; d < 8; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, o, d);
        if (my_warp >= d) o += y;
    }
    o -= c;  // first record of warp my_warp within its tile
    const uint64_t first = have && my_warp == 0 ? a.tile_first[t0 + my_tile] : 0u;
    uint64_t f[kRecordTiles];
    uint32_t tot[kRecordTiles], most = 0;
#pragma unroll
    for (int k = 0; k < kRecordTiles; ++k) {
        f[k] = __shfl_sync(kFull, first, 8 * k);
        tot[k] = __shfl_sync(kFull, o + c, 8 * k + 7);
        most = max(most, tot[k]);
    }
    const Layout L0 = layout_for(a.n, a.dtype, a.chunk_elems, 0);
    uint8_t* records = a.out + L0.escrec_off;
    const uint32_t region = 32u * kThreadBytes / elem_bytes(a.dtype);  // elements of a consumer warp's region
    // the staged record i of tile k (0 past the tile's count)
    auto staged = [&](int k, uint32_t i) -> uint32_t {
        // warp of record i: the last warp whose first record is <= i
        uint32_t w = 0;
#pragma unroll
        for (uint32_t step = 4; step > 0; step >>= 1) {
            const uint32_t first_w = __shfl_sync(kFull, o, 8 * k + int(w + step));
            if (i >= first_w) w += step;
        }
        const uint32_t first_w = __shfl_sync(kFull, o, 8 * k + int(w));
        // a plain load: neighbouring records are read by other lanes in other
        // rounds, so the sector must stay in L2 (an evict-first load re-read
        // it from DRAM each time)
        return i < tot[k] ? a.staging[(t0 + k) * a.tile_elems + w * region + (i - first_w)] : 0u;
    };
    auto put = [&](int k, uint32_t i, uint32_t v) {
        if (i < tot[k]) {
            uint8_t* d = records + 3 * (f[k] + i);
            d[0] = uint8_t(v >> 8);
            d[1] = uint8_t(v >> 16);
            d[2] = uint8_t(v);
        }
    };
    // two rounds at a time: eight independent loads in flight per lane
    for (uint32_t r0 = 0; r0 < most; r0 += 64u) {
        const uint32_t i0 = r0 + uint32_t(lane), i1 = i0 + 32u;
        uint32_t v[2 * kRecordTiles];
#pragma unroll
        for (int k = 0; k < kRecordTiles; ++k) {
            v[k] = staged(k, i0);
            v[kRecordTiles + k] = staged(k, i1);
        }
#pragma unroll
        for (int k = 0; k < kRecordTiles; ++k) {
            put(k, i0, v[k]);
            put(k, i1, v[kRecordTiles + k]);
        }
    }
}

// Launch with programmatic stream serialization: the kernel's CTAs may be
// scheduled while the previous kernel in the stream drains; each waits for it
// in griddepcontrol.wait before reading anything it wrote.
template <typename Kernel>
cudaError_t launch_dependent(Kernel kernel, unsigned grid, unsigned block, cudaStream_t s, const EncodeArgs& a) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

cudaError_t launch_encode(const EncodeArgs& a, const EncodeLut& lut, const CUtensorMap& map, int grid,
                          cudaStream_t s) {
    if (a.dtype == SPLITZIP_BF16)
        encode_kernel<SPLITZIP_BF16><<<grid, kBlock, kEncodeSmem<SPLITZIP_BF16>, s>>>(a, map, lut);
    else if (a.dtype == SPLITZIP_FP16)
        encode_kernel<SPLITZIP_FP16><<<grid, kBlock, kEncodeSmem<SPLITZIP_FP16>, s>>>(a, map, lut);
    else
        encode_kernel<SPLITZIP_FP8_E5M2><<<grid, kBlock, kEncodeSmem<SPLITZIP_FP8_E5M2>, s>>>(a, map, lut);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || a.n_groups == 0) return e;
    if ((e = launch_dependent(encode_group_kernel, unsigned(a.n_groups), kFinishThreads, s, a)) != cudaSuccess) return e;
    if ((e = launch_dependent(encode_index_kernel, unsigned(a.n_groups), kFinishThreads, s, a)) != cudaSuccess) return e;
    const uint64_t warps = (a.n_tiles + kRecordTiles - 1) / kRecordTiles;
    return launch_dependent(encode_records_kernel,
                            unsigned((warps + kRecordThreads / 32 - 1) / (kRecordThreads / 32)), kRecordThreads, s, a);
}

cudaError_t occupancy_encode(int* blocks_per_sm, int dtype) {
    auto k = dtype == SPLITZIP_BF16   ? encode_kernel<SPLITZIP_BF16>
             : dtype == SPLITZIP_FP16 ? encode_kernel<SPLITZIP_FP16>
                                      : encode_kernel<SPLITZIP_FP8_E5M2>;
    const int smem = int(dtype == SPLITZIP_BF16   ? kEncodeSmem<SPLITZIP_BF16>
                         : dtype == SPLITZIP_FP16 ? kEncodeSmem<SPLITZIP_FP16>
                                                  : kEncodeSmem<SPLITZIP_FP8_E5M2>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k, kBlock, smem);
}

}  // namespace splitzip
