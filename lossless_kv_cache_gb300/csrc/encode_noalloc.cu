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
#include "splitzip_internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[SPLITZIP_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array on the current device.  In host code
// the symbol g_noalloc_scratch is only a host-side stand-in, so the address is
// asked from the runtime, with the device current, on every call: once the
// module is loaded this is a table lookup, and an address taken before a
// device reset (after which the module can load at another address) is never
// reused.  The first call on a device loads the module, so it should come
// before any stream capture.
int scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    *out = p;
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
