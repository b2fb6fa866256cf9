// Allocation-free variant of splitzip_encode.
//
// splitzip_encode needs a device workspace from the caller (the per-tile
// escape staging area).  Some callers cannot allocate one: a serving engine
// that has already handed almost all device memory to its own KV-cache pool
// and allocator, or a code path that must not call cudaMalloc / cudaFree
// because those calls can synchronise the device and stall the other streams.
// This entry point runs the same encode with its scratch in a file-scope
// device array of fixed size, so it allocates nothing at call time.
//
// The array costs SPLITZIP_NOALLOC_SCRATCH_BYTES of device memory on every
// GPU that loads this library, for the life of the process.  All calls on a
// device share it: calls whose GPU work overlaps in time (different streams,
// or several host threads) race on it and must be serialised by the caller.
// splitzip_encode writes every word of its workspace before reading it, so
// the contents left by an earlier call do no harm.
#include <mutex>

#include "splitzip_internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[SPLITZIP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_address[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the symbol g_noalloc_scratch is only a host-side stand-in, so the address is
// asked from the runtime once per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SPLITZIP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_address[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SPLITZIP_ERR_CUDA;
        }
        g_scratch_address[dev] = p;
    }
    *out = g_scratch_address[dev];
    return SPLITZIP_OK;
}

}  // namespace

extern "C" int splitzip_encode_noalloc(const void* d_in, uint64_t n, int dtype, const splitzip_codebook_t* cb,
                                       uint32_t chunk_elems, void* d_out, uint64_t out_capacity,
                                       uint64_t* d_out_size, int* d_status, cudaStream_t stream) {
    uint64_t need = 0;
    int st = splitzip_encode_workspace_size(n, dtype, chunk_elems, &need);
    if (st != SPLITZIP_OK) return st;
    if (need > SPLITZIP_NOALLOC_SCRATCH_BYTES) return SPLITZIP_ERR_CAPACITY;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != SPLITZIP_OK) return st;
    return splitzip_encode(d_in, n, dtype, cb, chunk_elems, d_out, out_capacity, scratch,
                           SPLITZIP_NOALLOC_SCRATCH_BYTES, d_out_size, d_status, stream);
}
