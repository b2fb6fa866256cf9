// Self-test of the bounded device wait that the streaming kernels use.
//
// Every wait of the encode and decode kernels on a bulk-copy barrier gives up
// after a bounded number of SM cycles, records SPLITZIP_ERR_TIMEOUT in the
// status word and lets the CTA run to its end, so that no fault of the copy
// engine can hang the GPU.  In a healthy run that path never executes.  This
// kernel executes it on purpose, without any copy in flight: one warp waits,
// with a short limit, on an mbarrier that nothing ever arrives on, records the
// time-out exactly as the production kernels do, and returns.  A control wait
// on a barrier whose phase has completed must succeed.
#include "splitzip_internal.cuh"
#include "tma_pipeline.cuh"

namespace splitzip {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_kernel(int* status, long long limit, long long* cycles) {
    __shared__ __align__(8) uint64_t never;  // no thread arrives: its phase 0 never completes
    __shared__ __align__(8) uint64_t done;   // one arrival completes its phase 0
    if (threadIdx.x == 0) {
        mbar_init(&never, 1);
        mbar_init(&done, 1);
        mbar_init_fence();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_arrive(&done);
    __syncwarp();
    long long t0 = clock64();
    const bool control = mbar_wait_limit(&done, 0, limit);
    const long long control_cycles = clock64() - t0;
    t0 = clock64();
    const bool completed = mbar_wait_limit(&never, 0, limit);
    const long long wait_cycles = clock64() - t0;
    // the same report a streaming kernel makes when a wait runs out
    if (threadIdx.x == 0) {
        if (!completed || !control) atomicCAS(status, SPLITZIP_OK, SPLITZIP_ERR_TIMEOUT);
        if (cycles) {
            cycles[0] = wait_cycles;
            cycles[1] = control ? control_cycles : -1;
        }
    }
}

}  // namespace
}  // namespace splitzip

extern "C" int splitzip_selftest_bounded_wait(uint64_t limit_cycles, int* d_status, long long* d_cycles,
                                              cudaStream_t stream) {
    if (limit_cycles == 0 || limit_cycles > uint64_t(splitzip::kWaitLimitCycles)) return SPLITZIP_ERR_INVALID_ARG;
    if (!d_status || (reinterpret_cast<uintptr_t>(d_status) & 3u) != 0u) return SPLITZIP_ERR_INVALID_ARG;
    if (d_cycles && (reinterpret_cast<uintptr_t>(d_cycles) & 7u) != 0u) return SPLITZIP_ERR_INVALID_ARG;
    if (cudaMemsetAsync(d_status, 0, sizeof(int), stream) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    splitzip::bounded_wait_kernel<<<1, 32, 0, stream>>>(d_status, (long long)limit_cycles, d_cycles);
    return cudaGetLastError() == cudaSuccess ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
}
