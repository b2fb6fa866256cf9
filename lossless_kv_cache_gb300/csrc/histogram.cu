// Exponent histogram and Top-16 codebook for calibration (sm_103a).
//
// "SplitZip: Ultra Fast Lossless KV Compression for Disaggregated LLM
// Serving", Results, "Ablations: Calibration": one codebook calibrated
// offline generalises across data and layers, so the histogram runs once,
// outside the encode path.  Per-warp shared-memory histograms, 16-byte
// loads, then one global 64-bit atomic add per non-empty bin per CTA.
// Integer counts, so the result does not depend on the order of the adds.
#include "splitzip_internal.cuh"

namespace splitzip {
namespace {

template <int DT>
__device__ __forceinline__ void count_word(uint32_t w, uint32_t* h) {
    if constexpr (DT == SPLITZIP_BF16) {
        atomicAdd(&h[(w >> 7) & 0xFFu], 1u);
        atomicAdd(&h[(w >> 23) & 0xFFu], 1u);
    } else if constexpr (DT == SPLITZIP_FP16) {
        atomicAdd(&h[(w >> 10) & 0x1Fu], 1u);
        atomicAdd(&h[(w >> 26) & 0x1Fu], 1u);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) atomicAdd(&h[(w >> (8 * k + 2)) & 0x1Fu], 1u);
    }
}

template <int DT>
__global__ void __launch_bounds__(kHistThreads)
histogram_kernel(const uint8_t* x, uint64_t n, unsigned long long* hist) {
    constexpr int kWarps = kHistThreads / 32;
    constexpr uint64_t kElemBytes = DT == SPLITZIP_FP8_E5M2 ? 1 : 2;
    __shared__ uint32_t h[kWarps][256];
    for (int i = threadIdx.x; i < kWarps * 256; i += kHistThreads) (&h[0][0])[i] = 0u;
    __syncthreads();
    uint32_t* mine = h[threadIdx.x >> 5];
    const uint64_t bytes = n * kElemBytes;
    const uint64_t vecs = bytes / 16;
    const uint64_t stride = uint64_t(gridDim.x) * kHistThreads;
    for (uint64_t v = uint64_t(blockIdx.x) * kHistThreads + threadIdx.x; v < vecs; v += stride) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(x) + v);
        count_word<DT>(q.x, mine);
        count_word<DT>(q.y, mine);
        count_word<DT>(q.z, mine);
        count_word<DT>(q.w, mine);
    }
    // tail elements (fewer than one vector), block 0 only
    if (blockIdx.x == 0) {
        for (uint64_t i = vecs * 16 / kElemBytes + threadIdx.x; i < n; i += kHistThreads) {
            uint32_t e;
            if constexpr (DT == SPLITZIP_BF16) {
                const uint32_t b = uint32_t(x[2 * i]) | (uint32_t(x[2 * i + 1]) << 8);
                e = (b >> 7) & 0xFFu;
            } else if constexpr (DT == SPLITZIP_FP16) {
                const uint32_t b = uint32_t(x[2 * i]) | (uint32_t(x[2 * i + 1]) << 8);
                e = (b >> 10) & 0x1Fu;
            } else {
                e = (uint32_t(x[i]) >> 2) & 0x1Fu;
            }
            atomicAdd(&mine[e], 1u);
        }
    }
    __syncthreads();
    for (int b = threadIdx.x; b < 256; b += kHistThreads) {
        unsigned long long s = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += h[w][b];
        if (s) atomicAdd(&hist[b], s);
    }
}

// Top-16 of the histogram (Method, "Top-16 exponent coding"): bin t's rank
// is the number of bins with a larger count, or an equal count and a smaller
// exponent -- the order of a stable sort by descending count -- and the bins
// of rank < 16 are the codebook, code = rank.  Exponents that never occur
// fill the remaining codes in ascending order.
__global__ void __launch_bounds__(256) codebook_kernel(const unsigned long long* hist, int dtype, uint8_t* cb) {
    __shared__ unsigned long long h[256];
    const int t = threadIdx.x;
    const int bins = dtype == SPLITZIP_BF16 ? 256 : 32;
    h[t] = t < bins ? hist[t] : 0ull;
    __syncthreads();
    if (t < bins) {
        int rank = 0;
        for (int j = 0; j < bins; ++j) rank += (h[j] > h[t]) || (h[j] == h[t] && j < t);
        if (rank < 16) cb[1 + rank] = uint8_t(t);
    }
    if (t == 0) cb[0] = uint8_t(dtype);
}

}  // namespace

cudaError_t launch_codebook(const unsigned long long* hist, int dtype, uint8_t* cb, cudaStream_t s) {
    codebook_kernel<<<1, 256, 0, s>>>(hist, dtype, cb);
    return cudaGetLastError();
}

cudaError_t launch_histogram(const void* x, uint64_t n, int dtype, unsigned long long* hist, int grid,
                             cudaStream_t s) {
    const uint8_t* p = static_cast<const uint8_t*>(x);
    if (dtype == SPLITZIP_BF16)
        histogram_kernel<SPLITZIP_BF16><<<grid, kHistThreads, 0, s>>>(p, n, hist);
    else if (dtype == SPLITZIP_FP16)
        histogram_kernel<SPLITZIP_FP16><<<grid, kHistThreads, 0, s>>>(p, n, hist);
    else
        histogram_kernel<SPLITZIP_FP8_E5M2><<<grid, kHistThreads, 0, s>>>(p, n, hist);
    return cudaGetLastError();
}

cudaError_t occupancy_histogram(int* blocks_per_sm, int dtype) {
    if (dtype == SPLITZIP_BF16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, histogram_kernel<SPLITZIP_BF16>,
                                                             kHistThreads, 0);
    if (dtype == SPLITZIP_FP16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, histogram_kernel<SPLITZIP_FP16>,
                                                             kHistThreads, 0);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm,
                                                         histogram_kernel<SPLITZIP_FP8_E5M2>, kHistThreads, 0);
}

}  // namespace splitzip
