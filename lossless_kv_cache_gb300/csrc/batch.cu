// Small tensors and batches of tensors (sm_103a).
//
// Method: "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", section "Method: SplitZip" (Encoding strategy, Decoding strategy);
// the page's transfers are per request and per layer (section "Results": the
// gains depend on sequence length and batch size), so a call often carries a
// few megabytes, or a list of such pieces.  At that size a call is set by its
// launches and dependent memory round trips, not by HBM bandwidth, so this
// path spends fewer of both:
//
// Encode, phase 1 (a tile: 16 KB of input): plain 16-byte loads (no
// staging ring), the same per-element arithmetic as the streaming encoder, a
// CTA-wide scan that puts the tile's escape records contiguously in its
// staging slot, and the tile's escape count and error code in the workspace.
// Phase 2 (a chunk): the escapes of the item's earlier tiles (read directly;
// items are bounded in size), the chunk's index entry, its records moved into
// the escape stream, and E and the size from the last chunk.
// Decode, per 8,192 elements: direct loads and the same recombination as the
// persistent decoder; per chunk: the index entry and every escape record
// checked, then the escapes patched.
//
// A single small tensor whose tiles all fit the GPU at once is encoded by ONE
// cooperative kernel (all CTAs resident; one grid-wide sync between the
// phases, which every CTA reaches exactly once; phase 2 is then per tile: the
// escapes of the earlier tiles, the tile's records, the index entry of the
// chunk it starts).  Block 0 clears the status word in phase 1; errors are
// reported only after the sync.  Otherwise (a batch: many tensors, any sizes
// up to the item limit) phase 1 and phase 2 are two kernels chained with
// programmatic dependent launch (the second grid is scheduled while the first
// drains and waits for it in griddepcontrol.wait).  The decoder is a
// one-thread status clear and one CTA per 8,192 elements that stages the
// escape records of the chunks it overlaps in shared memory while it decodes,
// checks them all and patches those inside its elements (no CTA depends on
// another).  (A cooperative decoder was measured and dropped: its grid-wide
// sync and serial spans cost more than the launch it saves.)  A batch's item
// table travels as a kernel parameter (no allocation, no copy).
#include <cstring>
#include <type_traits>
#include <utility>

#include <cooperative_groups.h>

#include "decode_core.cuh"
#include "encode_core.cuh"
#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
static_assert(kThreads * kThreadBytes == kTileBytes, "one tile = 64 bytes per thread");
constexpr uint32_t kDecodeSub = 8192;  // elements of a decode step

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

struct EncItem {
    const uint8_t* in;
    uint8_t* out;
    uint64_t* out_size;
    uint8_t* ws;       // the item's workspace (workspace_for layout)
    uint64_t n;
    uint64_t n_tiles;  // 0 for an empty item
    uint64_t cta0;     // first CTA of phase 1 (one per tile; one for an empty item)
    uint64_t chunk0;   // first CTA of phase 2 (one per chunk)
};

template <int MAXI>
struct EncBatch {
    uint32_t count;
    int dtype;
    uint32_t chunk_elems, tile_elems;
    int* status;
    const uint8_t* dev_codebook;  // a splitzip_codebook_t in device memory, or null
    uint8_t codebook[16];
    EncItem item[MAXI];
};

// The last item k whose range starts at or before x (ranges ascending; an
// item with an empty range is skipped by the next one starting at the same x).
template <int MAXI, typename First>
__device__ __forceinline__ uint32_t find_item(uint32_t count, uint64_t x, First first) {
    if constexpr (MAXI == 1) {
        return 0;
    } else {
        uint32_t lo = 0, hi = count;
        while (hi - lo > 1) {
            const uint32_t mid = (lo + hi) / 2;
            if (first(mid) <= x)
                lo = mid;
            else
                hi = mid;
        }
        return lo;
    }
}

// In the workspace of an item on this path: per tile its escape count (the
// first n_tiles words of the warp-count area) and its error code (the next
// n_tiles words); the staging slots as on the streaming path, each holding its
// tile's records contiguously.
struct SmallWs {
    uint32_t* count;
    uint32_t* err;
    uint32_t* staging;
};

__device__ __forceinline__ SmallWs small_ws(const EncItem& it, int dtype, uint32_t chunk) {
    const Workspace W = workspace_for(it.n, dtype, chunk);
    SmallWs s;
    s.count = reinterpret_cast<uint32_t*>(it.ws + W.warp_count_off);
    s.err = s.count + W.n_tiles;
    s.staging = reinterpret_cast<uint32_t*>(it.ws + W.staging_off);
    return s;
}

// Sum of v over the CTA (every thread gets it); scratch: kWarps words.
__device__ __forceinline__ uint64_t block_sum(uint64_t v, uint64_t* scratch) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(kFull, v, d);
    __syncthreads();  // scratch may still be read from a previous use
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    uint64_t s = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += scratch[w];
    return s;
}

// Shared-memory tables of a CTA: the code of every exponent (escape-flagged
// outside the codebook), the four position tables, and the codebook.  A
// device codebook is checked here (dtype, range, distinct); *err receives
// SPLITZIP_ERR_INVALID_ARG for a bad one.
struct EncShared {
    __align__(16) uint32_t tab[4 * 256];
    uint8_t code[256];
    uint8_t cb[16];
    uint32_t warp_total[kWarps];
    uint64_t scratch[kWarps];
    uint32_t pre[9];  // phase 2: escapes before each tile of the chunk
    int err;
};

template <int DT>
__device__ __forceinline__ void build_tables(EncShared& S, const uint8_t* dev_cb, const uint8_t* host_cb,
                                             const EncodeLut& lut, int dtype) {
    const int tid = threadIdx.x;
    if (tid == 0) S.err = SPLITZIP_OK;
    if (dev_cb) {
        for (int i = tid; i < 256; i += kThreads) S.code[i] = kEscapeFlag;
        if (tid < 16) S.cb[tid] = dev_cb[1 + tid];
        __syncthreads();
        if (tid == 0) {
            bool ok = dev_cb[0] == uint8_t(dtype);
            for (int c = 0; c < 16; ++c) {
                const uint32_t e = S.cb[c];
                ok &= e < (DT == SPLITZIP_BF16 ? 256u : 32u) && S.code[e] == kEscapeFlag;
                S.code[e] = uint8_t(c);
            }
            if (!ok) S.err = SPLITZIP_ERR_INVALID_ARG;
        }
    } else {
        for (int i = tid; i < 256; i += kThreads) S.code[i] = lut.code[i];
        if (tid < 16) S.cb[tid] = host_cb[tid];
    }
    __syncthreads();
    for (int i = tid; i < 4 * 256; i += kThreads) S.tab[i] = table_entry(DT, i >> 8, uint32_t(i & 255), S.code);
    __syncthreads();
}

// Phase 1 of tile t of an item: its streams stored, its escape records staged
// contiguously in element order, its count and error code in the workspace.
// Every thread of the CTA calls it (it holds a CTA barrier).
template <int DT>
__device__ __forceinline__ void encode_tile(EncShared& S, const EncItem& it, int dtype, uint32_t chunk_elems,
                                            uint32_t tile_elems, uint64_t t) {
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    using Out = ThreadOut<DT>;
    constexpr uint32_t TE = Out::kElems;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const Layout L0 = layout_for(it.n, dtype, chunk_elems, 0);
    const uint64_t base = t * tile_elems;
    const uint64_t rem = it.n - base;
    const uint32_t len = rem < tile_elems ? uint32_t(rem) : tile_elems;
    const uint32_t my_elem = kThreadBytes / EB * uint32_t(tid);
    const uint32_t ne = len > my_elem ? min(len - my_elem, TE) : 0u;
    const uint8_t* src = it.in + base * EB + kThreadBytes * uint32_t(tid);
    const uint32_t my_bytes = ne * EB;  // valid bytes of this thread's 64

    // compute and store: a copy for a thread with all TE elements, in which
    // every index is static (the results stay in registers), and one for the
    // thread that holds the end of the tensor
    uint32_t mask[2];
    auto body = [&](auto full_tag) {
        constexpr bool FULL = decltype(full_tag)::value;
        Out o;
        [[maybe_unused]] uint32_t p[8];
        clear_out<DT>(o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 v;
            if (FULL || 16u * (i + 1) <= my_bytes)
                v = __ldg(reinterpret_cast<const uint4*>(src) + i);
            else if (16u * i < my_bytes)
                v = load_partial(src + 16 * i, my_bytes - 16u * i);
            else
                v = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (DT == SPLITZIP_FP8_E5M2)
                encode_piece(S.tab, v, i, o, p);
            else
                encode_piece(S.tab, v, i, o);
        }
        store_streams<DT, FULL>(o, p, it.out + L0.nibble_off, it.out + L0.signmant_off, base + my_elem, ne);
        escape_masks<DT>(o, mask);
    };
    if (ne == TE)
        body(std::true_type{});
    else
        body(std::false_type{});

    // the tile's escapes, in element order and contiguous, to its staging slot
    const uint32_t cnt = __popc(mask[0]) + __popc(mask[1]);
    uint32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += y;
    }
    __syncthreads();  // warp_total may still be read for the previous tile
    if (lane == 31) S.warp_total[warp] = incl;
    __syncthreads();
    uint32_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        before += w < warp ? S.warp_total[w] : 0u;
        total += S.warp_total[w];
    }
    const SmallWs ws = small_ws(it, dtype, chunk_elems);
    if (cnt) {
        auto bits = [&](uint32_t b) -> uint32_t {
            const uint8_t* e = src + b * EB;
            return EB == 2 ? uint32_t(__ldg(reinterpret_cast<const uint16_t*>(e))) : uint32_t(__ldg(e));
        };
        const uint32_t pos0 = uint32_t(base & (chunk_elems - 1u)) + my_elem;
        stage_records_masked<DT>(mask, ws.staging + t * tile_elems + before + (incl - cnt), pos0, bits);
    }
    if (tid == 0) {
        ws.count[t] = total;
        ws.err[t] = uint32_t(S.err);
    }
}

// Phase 2 of chunk c of an item: the escapes of the item's earlier tiles, the
// chunk's index entry, its records moved from the staging slots of its tiles
// into the escape stream, E and the size from the last chunk, and the tiles'
// error codes to the status word.  Every thread of the CTA calls it.
__device__ __forceinline__ void finish_chunk(EncShared& S, const EncItem& it, int dtype, uint32_t chunk_elems,
                                             uint32_t tile_elems, uint64_t c, int* status) {
    const int tid = threadIdx.x;
    const SmallWs ws = small_ws(it, dtype, chunk_elems);
    const uint32_t tpc = chunk_elems / tile_elems;  // a power of two <= 8
    const uint64_t t0 = c * tpc;
    const uint32_t nt = uint32_t(min(uint64_t(tpc), it.n_tiles - t0));
    uint64_t b = 0;
    for (uint64_t q = uint64_t(tid); q < t0; q += kThreads) b += ws.count[q];
    const uint64_t before = block_sum(b, S.scratch);
    if (tid < 32) {
        // the chunk's tiles (at most 8): counts and errors in parallel, a scan
        const uint32_t cnt = uint32_t(tid) < nt ? ws.count[t0 + tid] : 0u;
        const int e = uint32_t(tid) < nt ? int(ws.err[t0 + tid]) : SPLITZIP_OK;
        if (e != SPLITZIP_OK) report(status, e);
        uint32_t incl = cnt;  // inclusive scan over lanes 0..8 (lane nt <= 8 has count 0: the total)
#pragma unroll
        for (int d = 1; d < 16; d <<= 1) {
            const uint32_t y = __shfl_up_sync(kFull, incl, d);
            if (tid >= d) incl += y;
        }
        if (uint32_t(tid) <= nt) S.pre[tid] = incl - cnt;
    }
    __syncthreads();
    const uint32_t run = S.pre[nt];
    if (tid == 0) {
        const Layout L0 = layout_for(it.n, dtype, chunk_elems, 0);
        reinterpret_cast<uint64_t*>(it.out + L0.index_off)[c] = before;
        reinterpret_cast<uint32_t*>(it.out + L0.counts_off)[c] = run;
        if (c + 1 == L0.n_chunks) {  // the last chunk knows E
            reinterpret_cast<uint64_t*>(it.out)[3] = before + run;
            *it.out_size = layout_for(it.n, dtype, chunk_elems, before + run).size;
        }
    }
    const uint32_t R = run;
    uint8_t* recs = it.out + layout_for(it.n, dtype, chunk_elems, 0).escrec_off + 3 * before;
    for (uint32_t r0 = 0; r0 < R; r0 += 4 * kThreads) {
        uint32_t v[4], at[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t r = r0 + uint32_t(k * kThreads + tid);
            v[k] = 0u;
            at[k] = r;
            if (r < R) {
                uint32_t i = 0;
                while (i + 1 < nt && S.pre[i + 1] <= r) ++i;  // the tile of record r
                v[k] = ws.staging[(t0 + i) * tile_elems + (r - S.pre[i])];
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (at[k] < R) {
                uint8_t* d = recs + 3 * at[k];
                d[0] = uint8_t(v[k] >> 8);
                d[1] = uint8_t(v[k] >> 16);
                d[2] = uint8_t(v[k]);
            }
        }
    }
    __syncthreads();  // S.pre is reused by the next chunk
}

// Phase 2 of tile t (every tile of the item resident in one grid, after a
// grid-wide sync): the escapes of the item's earlier tiles, the tile's records
// moved into the escape stream, the index entry of the chunk it starts, E and
// the size from the last tile, and the tile's error code to the status word.
// Every thread of the CTA calls it.
__device__ __forceinline__ void finish_tile(EncShared& S, const EncItem& it, int dtype, uint32_t chunk_elems,
                                            uint32_t tile_elems, uint64_t t, int* status) {
    const int tid = threadIdx.x;
    const SmallWs ws = small_ws(it, dtype, chunk_elems);
    uint64_t b = 0;
    for (uint64_t q = uint64_t(tid); q < t; q += kThreads) b += ws.count[q];
    const uint64_t before = block_sum(b, S.scratch);
    const uint32_t cnt = ws.count[t];
    const Layout L0 = layout_for(it.n, dtype, chunk_elems, 0);
    const uint32_t tpc = chunk_elems / tile_elems;  // a power of two <= 8
    if (tid < 32 && t % tpc == 0) {
        // the chunk this tile starts: its count is the sum over its tiles
        const uint64_t q = t + uint64_t(tid);
        uint32_t c = uint32_t(tid) < tpc && q < it.n_tiles ? ws.count[q] : 0u;
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) c += __shfl_xor_sync(kFull, c, d);
        if (tid == 0) {
            reinterpret_cast<uint64_t*>(it.out + L0.index_off)[t / tpc] = before;
            reinterpret_cast<uint32_t*>(it.out + L0.counts_off)[t / tpc] = c;
        }
    }
    if (tid == 0) {
        const int e = int(ws.err[t]);
        if (e != SPLITZIP_OK) report(status, e);
        if (t + 1 == it.n_tiles) {  // the last tile knows E
            reinterpret_cast<uint64_t*>(it.out)[3] = before + cnt;
            *it.out_size = layout_for(it.n, dtype, chunk_elems, before + cnt).size;
        }
    }
    uint8_t* recs = it.out + L0.escrec_off + 3 * before;
    const uint32_t* src = ws.staging + t * tile_elems;
    for (uint32_t r0 = 0; r0 < cnt; r0 += 4 * kThreads) {
        uint32_t v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t r = r0 + uint32_t(k * kThreads + tid);
            v[k] = r < cnt ? src[r] : 0u;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t r = r0 + uint32_t(k * kThreads + tid);
            if (r < cnt) {
                uint8_t* d = recs + 3 * r;
                d[0] = uint8_t(v[k] >> 8);
                d[1] = uint8_t(v[k] >> 16);
                d[2] = uint8_t(v[k]);
            }
        }
    }
}

template <int DT, int MAXI>
__global__ void __launch_bounds__(kThreads) small_encode_kernel(const __grid_constant__ EncBatch<MAXI> P,
                                                                const __grid_constant__ EncodeLut lut) {
    pdl_launch_dependents();  // phase 2 may be scheduled; it waits for this grid to finish
    __shared__ EncShared S;
    const uint32_t k = find_item<MAXI>(P.count, blockIdx.x, [&](uint32_t i) { return P.item[i].cta0; });
    const EncItem& it = P.item[k];
    const uint64_t t = blockIdx.x - it.cta0;  // tile of the item
    build_tables<DT>(S, P.dev_codebook, P.codebook, lut, P.dtype);
    if (blockIdx.x == 0 && threadIdx.x == 0) *P.status = SPLITZIP_OK;  // errors are reported by phase 2
    if (t == 0 && threadIdx.x == 0)
        write_header_and_padding(it.out, P.dtype, it.n, P.chunk_elems, (it.n + P.chunk_elems - 1) / P.chunk_elems,
                                 S.cb, it.out_size);
    if (it.n_tiles == 0) return;  // an empty item: its header is all there is
    encode_tile<DT>(S, it, P.dtype, P.chunk_elems, P.tile_elems, t);
}

template <int MAXI>
__global__ void __launch_bounds__(kThreads) small_finish_kernel(const __grid_constant__ EncBatch<MAXI> P) {
    pdl_wait();  // phase 1 has finished and its writes are visible
    __shared__ EncShared S;
    const uint32_t k = find_item<MAXI>(P.count, blockIdx.x, [&](uint32_t i) { return P.item[i].chunk0; });
    const EncItem& it = P.item[k];
    finish_chunk(S, it, P.dtype, P.chunk_elems, P.tile_elems, blockIdx.x - it.chunk0, P.status);
}

// A single small tensor: both phases in one cooperative grid (every CTA is
// resident; each reaches the grid-wide sync exactly once).
template <int DT>
__global__ void __launch_bounds__(kThreads) coop_encode_kernel(const __grid_constant__ EncBatch<1> P,
                                                               const __grid_constant__ EncodeLut lut) {
    __shared__ EncShared S;
    const EncItem& it = P.item[0];
    build_tables<DT>(S, P.dev_codebook, P.codebook, lut, P.dtype);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *P.status = SPLITZIP_OK;  // errors are reported after the sync
        write_header_and_padding(it.out, P.dtype, it.n, P.chunk_elems, (it.n + P.chunk_elems - 1) / P.chunk_elems,
                                 S.cb, it.out_size);
    }
    for (uint64_t t = blockIdx.x; t < it.n_tiles; t += gridDim.x)
        encode_tile<DT>(S, it, P.dtype, P.chunk_elems, P.tile_elems, t);
    cooperative_groups::this_grid().sync();
    for (uint64_t t = blockIdx.x; t < it.n_tiles; t += gridDim.x)
        finish_tile(S, it, P.dtype, P.chunk_elems, P.tile_elems, t, P.status);
}

// ------------------------------------------------------------------ decode

struct DecItem {
    const uint8_t* in;
    uint64_t in_bytes;
    uint8_t* out;
    uint64_t n;
    uint64_t unit0;  // first CTA of the item (one per 8,192 elements; one for an empty item)
};

template <int MAXI>
struct DecBatch {
    uint32_t count;
    int dtype;
    int* status;
    DecItem item[MAXI];
};

__global__ void clear_status_kernel(int* status) {
    pdl_launch_dependents();
    *status = SPLITZIP_OK;
}

constexpr uint32_t kRecRound = 2048;  // escape records staged in shared memory at a time

template <int DT>
struct DecShared {
    Header hdr;
    int header_ok;
    uint16_t lut2[256];
    uint32_t lut4[DT == SPLITZIP_FP16 ? 256 : 1];
    // the chunks that overlap an 8,192-element span (at most 8,192 / 64)
    uint64_t c_off[kDecodeSub / kMinChunk];
    uint32_t c_cnt[kDecodeSub / kMinChunk];
    // a window of the escape stream: up to kRecRound records and the one before
    uint32_t rbuf[(3 * (kRecRound + 1) + 3 + 3) / 4];
};

// Header of an item, checked (thread 0), and the nibble-byte tables; every
// thread of the CTA calls it; returns the verdict.
template <int DT>
__device__ __forceinline__ bool load_header(DecShared<DT>& S, const uint8_t* in, uint64_t in_bytes, uint64_t n,
                                            int dtype) {
    const int tid = threadIdx.x;
    if (tid == 0) {
        DecodeArgs a{};
        a.in = in;
        a.in_bytes = in_bytes;
        a.n = n;
        a.dtype = dtype;
        S.header_ok = read_header(a, S.hdr);
    }
    __syncthreads();
    if (!S.header_ok) return false;
    for (int b = tid; b < 256; b += kThreads) {
        if constexpr (DT == SPLITZIP_FP16)
            S.lut4[b] = (uint32_t(S.hdr.codebook[b & 15]) << 10) | (uint32_t(S.hdr.codebook[b >> 4]) << 26);
        else
            S.lut2[b] = uint16_t((S.hdr.codebook[b & 15] | (S.hdr.codebook[b >> 4] << 8)) << (DT == SPLITZIP_BF16 ? 0 : 2));
    }
    __syncthreads();
    return true;
}

// Dense decode of elements [g0, g0 + m) from the container in global memory:
// 16 output bytes per unit, loads straight from the streams.
template <int DT>
__device__ __forceinline__ void decode_span(const DecShared<DT>& S, const uint8_t* in, uint8_t* out, uint64_t g0,
                                            uint32_t m) {
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    constexpr uint32_t UE = DT == SPLITZIP_FP8_E5M2 ? 16u : 8u;
    const uint8_t* nibbles = in + S.hdr.L.nibble_off;
    const uint8_t* signmant = in + S.hdr.L.signmant_off;
    const uint8_t* end = in + S.hdr.L.size;
    const uint32_t units = (m + UE - 1u) / UE;
#pragma unroll 4
    for (uint32_t j = threadIdx.x; j < units; j += kThreads) {
        const uint64_t e = g0 + uint64_t(UE) * j;  // first element of the unit
        const uint32_t valid = min(UE, uint32_t(g0 + m - e));
        uint4 o;
        if constexpr (DT == SPLITZIP_BF16) {
            uint32_t nib;
            uint2 sm;
            if (valid == UE) {
                nib = __ldg(reinterpret_cast<const uint32_t*>(nibbles + e / 2));
                sm = __ldg(reinterpret_cast<const uint2*>(signmant + e));
            } else {
                uint64_t smw = 0;
                nib = 0;
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nib |= uint32_t(nibbles[e / 2 + b]) << (8u * b);
                for (uint32_t b = 0; b < valid; ++b) smw |= uint64_t(signmant[e + b]) << (8u * b);
                sm = make_uint2(uint32_t(smw), uint32_t(smw >> 32));
            }
            o = decode_unit_bf16(nib, sm, S.lut2);
        } else if constexpr (DT == SPLITZIP_FP16) {
            uint32_t nib = 0, f0, f1, f2;
            const uint8_t* s = signmant + e / 8 * 11;
            const uint8_t* s_aligned = reinterpret_cast<const uint8_t*>(reinterpret_cast<uintptr_t>(s) & ~uintptr_t(3));
            if (valid == UE && s_aligned + 16 <= end) {  // four whole words inside the container
                nib = __ldg(reinterpret_cast<const uint32_t*>(nibbles + e / 2));
                load96(s, f0, f1, f2);
            } else {
                uint32_t f[3] = {0u, 0u, 0u};
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nib |= uint32_t(nibbles[e / 2 + b]) << (8u * b);
                for (uint32_t b = 0; b < 11u * ((valid + 7u) / 8u); ++b) f[b >> 2] |= uint32_t(s[b]) << (8u * (b & 3u));
                f0 = f[0];
                f1 = f[1];
                f2 = f[2];
            }
            o = decode_unit_fp16(nib, f0, f1, f2, S.lut4);
        } else {
            uint2 nib;
            uint32_t s3lo, s3hi;
            const uint8_t* s = signmant + e / 8 * 3;  // 6 bytes, 2-byte aligned
            if (valid == UE) {
                nib = __ldg(reinterpret_cast<const uint2*>(nibbles + e / 2));
                const uint16_t* s16 = reinterpret_cast<const uint16_t*>(s);
                s3lo = uint32_t(__ldg(s16)) | (uint32_t(__ldg(s16 + 1)) << 16);
                s3hi = __ldg(s16 + 2);
            } else {
                uint64_t nw = 0, sw = 0;
                for (uint32_t b = 0; b < (valid + 1u) / 2u; ++b) nw |= uint64_t(nibbles[e / 2 + b]) << (8u * b);
                for (uint32_t b = 0; b < 3u * ((valid + 7u) / 8u); ++b) sw |= uint64_t(s[b]) << (8u * b);
                nib = make_uint2(uint32_t(nw), uint32_t(nw >> 32));
                s3lo = uint32_t(sw);
                s3hi = uint32_t(sw >> 32);
            }
            o = decode_unit_e5m2(nib, s3lo, s3hi, S.lut2);
        }
        uint8_t* dst = out + e * EB;
        if (valid == UE) {
            __stcs(reinterpret_cast<uint4*>(dst), o);
        } else {
            for (uint32_t b = 0; b < valid; ++b) {
                const uint32_t q = EB == 2 ? b >> 1 : b >> 2;
                const uint32_t w = q == 0 ? o.x : q == 1 ? o.y : q == 2 ? o.z : o.w;
                if constexpr (EB == 2)
                    reinterpret_cast<uint16_t*>(dst)[b] = uint16_t(w >> (16u * (b & 1u)));
                else
                    dst[b] = uint8_t(w >> (8u * (b & 3u)));
            }
        }
    }
}

// Index entry of chunk c, checked as the persistent decoder checks it.
__device__ __forceinline__ bool index_entry(const Header& h, const uint8_t* in, uint64_t n, uint64_t c,
                                           uint64_t* off_out, uint64_t* cnt_out) {
    const uint64_t* offsets = reinterpret_cast<const uint64_t*>(in + h.L.index_off);
    const uint32_t* counts = reinterpret_cast<const uint32_t*>(in + h.L.counts_off);
    const uint64_t off = offsets[c], cnt = counts[c];
    const uint64_t len = min(uint64_t(h.chunk), n - c * h.chunk);
    const uint64_t expect = c == 0 ? 0 : offsets[c - 1] + counts[c - 1];
    *off_out = off;
    *cnt_out = cnt;
    return off == expect && cnt <= len && off <= h.E && cnt <= h.E - off && (c + 1 < h.n_chunks || off + cnt == h.E);
}

// Index entries of the chunks that overlap [g0, g0 + m) into S.c_off /
// S.c_cnt (chunk c_lo + j at j < nc); returns the CTA-wide verdict.  Every
// thread calls it.
template <int DT>
__device__ __forceinline__ bool load_index(DecShared<DT>& S, const uint8_t* in, uint64_t n, uint64_t g0, uint32_t m,
                                           uint64_t* c_lo, uint32_t* nc) {
    const uint64_t chunk = S.hdr.chunk;
    *c_lo = g0 / chunk;
    *nc = uint32_t((g0 + m - 1) / chunk - *c_lo + 1);
    bool ok = true;
    for (uint32_t j = threadIdx.x; j < *nc; j += kThreads) {
        uint64_t off, cnt;
        ok = index_entry(S.hdr, in, n, *c_lo + j, &off, &cnt) && ok;
        S.c_off[j] = off;
        S.c_cnt[j] = uint32_t(cnt);
    }
    return __syncthreads_and(ok);
}

// A window of the escape stream in shared memory: records [wfirst, r_end)
// (wfirst = the first record of the run, or the one before it, for the order
// check), read with coalesced 4-byte loads (plain byte loads for the last
// word of the container).  No barrier: the caller syncs before reading.
struct Window {
    uint64_t wfirst;
    uint32_t shift;
};

template <int DT>
__device__ __forceinline__ Window load_window(DecShared<DT>& S, const uint8_t* in, uint64_t b, uint64_t r_end) {
    const uint8_t* stream = in + S.hdr.L.escrec_off;
    const uint8_t* end = in + S.hdr.L.size;
    Window w;
    w.wfirst = b > 0 ? b - 1 : 0;
    const uint8_t* p = stream + 3 * w.wfirst;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~uintptr_t(3);
    w.shift = uint32_t(reinterpret_cast<uintptr_t>(p) - a0);
    const uint32_t words = (w.shift + 3 * uint32_t(r_end - w.wfirst) + 3) / 4;
    for (uint32_t i = threadIdx.x; i < words; i += kThreads) {
        const uint8_t* q = reinterpret_cast<const uint8_t*>(a0 + 4 * i);
        uint32_t v = 0;
        if (q + 4 <= end) {
            v = __ldg(reinterpret_cast<const uint32_t*>(q));
        } else {
            for (int k = 0; k < 4; ++k)
                if (q + k < end) v |= uint32_t(q[k]) << (8 * k);
        }
        S.rbuf[i] = v;
    }
    return w;
}

// Records [b, e) held in the window w, which belong to the chunks c_lo + j
// (j < nc) of S.c_off (their index entries checked): with CHECK each record
// of a chunk at j >= j_check is checked (inside its chunk, after the chunk's
// previous record, exponent in range); with PATCH each record whose element
// lies in [lo, hi) is applied.  Returns false if a check failed (this thread).
template <int DT, bool CHECK, bool PATCH>
__device__ __forceinline__ bool window_records(const DecShared<DT>& S, const Window& w, uint8_t* out, uint64_t n,
                                               uint64_t c_lo, uint32_t nc, uint32_t j_check, uint64_t b, uint64_t e,
                                               uint64_t lo, uint64_t hi, int* status) {
    constexpr uint32_t EB = DT == SPLITZIP_FP8_E5M2 ? 1u : 2u;
    const uint64_t chunk = S.hdr.chunk;
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(S.rbuf) + w.shift;
    const OutMap<false> om{out, n * EB, nullptr, 0, 0, status};
    bool good = true;
    for (uint64_t r = b + threadIdx.x; r < e; r += kThreads) {
        const uint32_t k = uint32_t(r - w.wfirst);
        uint32_t jl = 0, jh = nc;  // the chunk of record r: the last j with c_off[j] <= r
        while (jh - jl > 1) {
            const uint32_t mid = (jl + jh) / 2;
            if (S.c_off[mid] <= r)
                jl = mid;
            else
                jh = mid;
        }
        const uint64_t c = c_lo + jl;
        const uint32_t len = uint32_t(min(chunk, n - c * chunk));
        const uint32_t pos = uint32_t(wb[3 * k]) | (uint32_t(wb[3 * k + 1]) << 8), ex = wb[3 * k + 2];
        const int64_t prev = r == S.c_off[jl] ? -1 : int64_t(uint32_t(wb[3 * k - 3]) | (uint32_t(wb[3 * k - 2]) << 8));
        const bool valid = pos < len && int64_t(pos) > prev && ex < (DT == SPLITZIP_BF16 ? 256u : 32u);
        if (CHECK && jl >= j_check && !valid) good = false;
        if (PATCH && valid) {
            const uint64_t g = c * chunk + pos;
            if (g >= lo && g < hi) patch_one<DT, false>(om, c * chunk, len, prev, pos, ex);
        }
    }
    return good;
}

// Records [r_begin, r_end) in rounds of the window (for runs longer than it);
// every thread calls it; returns the CTA-wide verdict of CHECK.
template <int DT, bool CHECK, bool PATCH>
__device__ __forceinline__ bool scan_records(DecShared<DT>& S, const uint8_t* in, uint8_t* out, uint64_t n,
                                             uint64_t c_lo, uint32_t nc, uint32_t j_check, uint64_t r_begin,
                                             uint64_t r_end, uint64_t lo, uint64_t hi, int* status) {
    bool good = true;
    for (uint64_t b = r_begin; b < r_end; b += kRecRound) {
        const uint64_t e = min(r_end, b + kRecRound);
        __syncthreads();  // the window may still be read from the previous round
        const Window w = load_window<DT>(S, in, b, e);
        __syncthreads();
        good = window_records<DT, CHECK, PATCH>(S, w, out, n, c_lo, nc, j_check, b, e, lo, hi, status) && good;
    }
    return __syncthreads_and(good);
}

template <int DT, int MAXI>
__global__ void __launch_bounds__(kThreads) small_decode_kernel(const __grid_constant__ DecBatch<MAXI> P) {
    __shared__ DecShared<DT> S;
    const int tid = threadIdx.x;
    const uint32_t k = find_item<MAXI>(P.count, blockIdx.x, [&](uint32_t i) { return P.item[i].unit0; });
    const DecItem& it = P.item[k];
    const uint64_t g0 = (blockIdx.x - it.unit0) * uint64_t(kDecodeSub);  // first element of the span
    pdl_wait();  // the status word has been cleared
    if (!load_header<DT>(S, it.in, it.in_bytes, it.n, P.dtype)) {
        if (tid == 0) report(P.status, SPLITZIP_ERR_CORRUPT);
        return;
    }
    if (it.n == 0) return;
    const uint32_t m = uint32_t(min(uint64_t(kDecodeSub), it.n - g0));
    uint64_t c_lo;
    uint32_t nc;
    const bool index_ok = load_index<DT>(S, it.in, it.n, g0, m, &c_lo, &nc);
    // the records of the overlapping chunks are one run of the stream (the
    // offsets are a prefix): staged while the span is decoded when they fit
    const uint64_t rb = S.c_off[0], re = S.c_off[nc - 1] + S.c_cnt[nc - 1];
    const bool fits = index_ok && re - rb <= kRecRound;
    Window w{};
    if (fits) w = load_window<DT>(S, it.in, rb, re);
    decode_span<DT>(S, it.in, it.out, g0, m);
    if (!index_ok) {
        if (tid == 0) report(P.status, SPLITZIP_ERR_CORRUPT);
        return;
    }
    // every record of the overlapping chunks checked (a chunk larger than the
    // span by every CTA it overlaps); the span's own elements patched, after
    // its dense stores (the barrier)
    bool ok;
    if (fits) {
        __syncthreads();
        ok = __syncthreads_and(
            window_records<DT, true, true>(S, w, it.out, it.n, c_lo, nc, 0, rb, re, g0, g0 + m, P.status));
    } else {
        ok = scan_records<DT, true, true>(S, it.in, it.out, it.n, c_lo, nc, 0, rb, re, g0, g0 + m, P.status);
    }
    if (!ok && tid == 0) report(P.status, SPLITZIP_ERR_CORRUPT);
}

// ------------------------------------------------------------------ launch

template <typename Kernel, typename... Args>
cudaError_t launch(Kernel kernel, uint64_t grid, int mode, cudaStream_t s, Args&&... args) {
    // mode 0: plain; 1: programmatic dependent launch; 2: cooperative
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (mode == 1) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    } else {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
    }
    cfg.attrs = mode ? attr : nullptr;
    cfg.numAttrs = mode ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <int MAXI>
void fill_encode(EncBatch<MAXI>& P, EncodeLut& lut, const SmallEncodeItem* items, uint32_t count, int dtype,
                 const uint8_t* codebook, const uint8_t* dev_codebook, uint32_t chunk, int* status, uint64_t* ctas,
                 uint64_t* chunks, uint64_t* tiles) {
    std::memset(&P, 0, sizeof(P));
    P.count = count;
    P.dtype = dtype;
    P.chunk_elems = chunk;
    P.tile_elems = tile_elems_for(dtype, chunk);
    P.status = status;
    P.dev_codebook = dev_codebook;
    std::memset(lut.code, kEscapeFlag, sizeof(lut.code));
    if (!dev_codebook) {
        std::memcpy(P.codebook, codebook, 16);
        for (int c = 0; c < 16; ++c) lut.code[codebook[c]] = uint8_t(c);
    }
    *ctas = *chunks = *tiles = 0;
    for (uint32_t i = 0; i < count; ++i) {
        EncItem& e = P.item[i];
        e.in = static_cast<const uint8_t*>(items[i].in);
        e.out = static_cast<uint8_t*>(items[i].out);
        e.out_size = items[i].out_size;
        e.ws = static_cast<uint8_t*>(items[i].ws);
        e.n = items[i].n;
        e.n_tiles = workspace_for(e.n, dtype, chunk).n_tiles;
        e.cta0 = *ctas;
        e.chunk0 = *chunks;
        *ctas += e.n_tiles > 0 ? e.n_tiles : 1;
        *chunks += (e.n + chunk - 1) / chunk;
        *tiles += e.n_tiles;
    }
}

template <int MAXI>
cudaError_t encode_batch_launch(const SmallEncodeItem* items, uint32_t count, int dtype, const uint8_t* codebook,
                                const uint8_t* dev_codebook, uint32_t chunk, int* status, cudaStream_t s) {
    EncBatch<MAXI> P;
    EncodeLut lut;
    uint64_t ctas, chunks, tiles;
    fill_encode(P, lut, items, count, dtype, codebook, dev_codebook, chunk, status, &ctas, &chunks, &tiles);
    cudaError_t err;
    if (dtype == SPLITZIP_BF16)
        err = launch(small_encode_kernel<SPLITZIP_BF16, MAXI>, ctas, 0, s, P, lut);
    else if (dtype == SPLITZIP_FP16)
        err = launch(small_encode_kernel<SPLITZIP_FP16, MAXI>, ctas, 0, s, P, lut);
    else
        err = launch(small_encode_kernel<SPLITZIP_FP8_E5M2, MAXI>, ctas, 0, s, P, lut);
    if (err != cudaSuccess || tiles == 0) return err;  // empty items: the headers are complete
    return launch(small_finish_kernel<MAXI>, chunks, 1, s, P);
}

template <int MAXI>
cudaError_t decode_batch_launch(const SmallDecodeItem* items, uint32_t count, int dtype, int* status,
                                cudaStream_t s) {
    DecBatch<MAXI> P;
    std::memset(&P, 0, sizeof(P));
    P.count = count;
    P.dtype = dtype;
    P.status = status;
    uint64_t units = 0;
    for (uint32_t i = 0; i < count; ++i) {
        DecItem& d = P.item[i];
        d.in = static_cast<const uint8_t*>(items[i].in);
        d.in_bytes = items[i].in_bytes;
        d.out = static_cast<uint8_t*>(items[i].out);
        d.n = items[i].n;
        d.unit0 = units;
        units += d.n > 0 ? (d.n + kDecodeSub - 1) / kDecodeSub : 1;  // an empty item still checks its header
    }
    cudaError_t err;
    if ((err = launch(clear_status_kernel, 1, 0, s, status)) != cudaSuccess) return err;
    if (dtype == SPLITZIP_BF16) return launch(small_decode_kernel<SPLITZIP_BF16, MAXI>, units, 1, s, P);
    if (dtype == SPLITZIP_FP16) return launch(small_decode_kernel<SPLITZIP_FP16, MAXI>, units, 1, s, P);
    return launch(small_decode_kernel<SPLITZIP_FP8_E5M2, MAXI>, units, 1, s, P);
}

}  // namespace

cudaError_t launch_small_encode(const SmallEncodeItem* items, uint32_t count, int dtype, const uint8_t* codebook,
                                const uint8_t* dev_codebook, uint32_t chunk, int* status, cudaStream_t s) {
    if (count == 1) return encode_batch_launch<1>(items, count, dtype, codebook, dev_codebook, chunk, status, s);
    return encode_batch_launch<kMaxBatch>(items, count, dtype, codebook, dev_codebook, chunk, status, s);
}

cudaError_t launch_small_decode(const SmallDecodeItem* items, uint32_t count, int dtype, int* status,
                                cudaStream_t s) {
    if (count == 1) return decode_batch_launch<1>(items, count, dtype, status, s);
    return decode_batch_launch<kMaxBatch>(items, count, dtype, status, s);
}

cudaError_t launch_coop_encode(const SmallEncodeItem& item, int dtype, const uint8_t* codebook,
                               const uint8_t* dev_codebook, uint32_t chunk, int* status, int grid, cudaStream_t s) {
    EncBatch<1> P;
    EncodeLut lut;
    uint64_t ctas, chunks, tiles;
    fill_encode(P, lut, &item, 1, dtype, codebook, dev_codebook, chunk, status, &ctas, &chunks, &tiles);
    if (dtype == SPLITZIP_BF16) return launch(coop_encode_kernel<SPLITZIP_BF16>, grid, 2, s, P, lut);
    if (dtype == SPLITZIP_FP16) return launch(coop_encode_kernel<SPLITZIP_FP16>, grid, 2, s, P, lut);
    return launch(coop_encode_kernel<SPLITZIP_FP8_E5M2>, grid, 2, s, P, lut);
}

cudaError_t occupancy_coop(int* encode_bpsm, int dtype) {
    if (dtype == SPLITZIP_BF16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(encode_bpsm, coop_encode_kernel<SPLITZIP_BF16>, kThreads,
                                                             0);
    if (dtype == SPLITZIP_FP16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(encode_bpsm, coop_encode_kernel<SPLITZIP_FP16>, kThreads,
                                                             0);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(encode_bpsm, coop_encode_kernel<SPLITZIP_FP8_E5M2>, kThreads,
                                                         0);
}

}  // namespace splitzip
