// The transfer path around the codec: a tensor leaves this GPU, crosses a
// link and is rebuilt on the other side.  The SplitZip page measures exactly
// this (prefill-to-decode KV transfer in disaggregated serving, section
// "Results": KV transfer speedup and the codec's share of the transfer time);
// on one GPU the link is the GPU <-> host path: device -> pinned host memory
// (the send) and back (the receive).
//
// The tensor is cut into pieces of whole chunks.  Piece i is encoded into its
// own container, its exact bytes cross the link in both directions, and it is
// decoded into the destination.  Four internal streams (encode, D2H, H2D,
// decode) and per-slot events let the four stages of different pieces run at
// the same time; kRing slots of device and host buffers are reused in turn.
// The streams and events come from a per-device pool and are reused by later
// calls.
// Slots start on 2 MiB boundaries (64 KiB for slots under 2 MiB): with slots
// at the 16-byte-aligned stride of a container's maximum size, the link copies
// of every other slot ran ~30 % slower (BF16 cache, one-layer pieces: 23.2-27.5
// ms per transfer against 20.6-21.4 ms with aligned slots).
// The host learns each container's size from a record that a one-thread
// kernel behind its encode stores into the pinned staging memory (mapped into
// the device's address space), and enqueues that piece's copies while the
// next piece encodes, the way a sender must know a message's length before
// posting it.  (A copy of the record would queue on the copy engine behind
// the previous piece's link copy, so the size would arrive only after that
// copy drained and the link would idle while the host enqueued the next.)
#include <cstring>
#include <mutex>
#include <vector>

#include "splitzip.h"
#include "splitzip_internal.cuh"

using namespace splitzip;

namespace {

constexpr int kRing = 4;  // pieces in flight

uint64_t a16(uint64_t x) { return (x + 15u) & ~uint64_t(15); }
uint64_t align_up(uint64_t x, uint64_t a) { return (x + a - 1u) / a * a; }

// Slot alignment for slots of `bytes`.
uint64_t slot_align(uint64_t bytes) {
    constexpr uint64_t kLarge = uint64_t(2) << 20, kSmall = uint64_t(64) << 10;
    return bytes >= kLarge ? kLarge : kSmall;
}

// Per-piece record in device scratch and its copy in host staging: the
// container size written by the encode, the encode and decode status words.
struct PieceInfo {
    uint64_t size;
    int enc_status;
    int dec_status;
};
static_assert(sizeof(PieceInfo) == 16, "16-byte piece records");

// Piece record (size, encode status) -> pinned host memory, in stream order.
__global__ void publish_info_kernel(const PieceInfo* src, PieceInfo* host_dst) {
    volatile PieceInfo* d = host_dst;
    d->size = src->size;
    d->enc_status = src->enc_status;
    __threadfence_system();
}

struct Plan {
    uint64_t pieces, piece_elems, cap;        // cap: one slot (a piece's container capacity, aligned)
    uint64_t align;                           // slot alignment; scratch bases are rounded up to it
    uint64_t ws_bytes;                        // one encode workspace
    uint64_t send_off, recv_off, ws_off, info_off, device_bytes;
    uint64_t stage_off, hinfo_off, host_bytes;
};

int plan_for(uint64_t n, int dtype, uint32_t chunk, uint64_t piece_elems, int compress, Plan* p) {
    if (n == 0 || piece_elems == 0 || chunk == 0 || piece_elems % chunk != 0) return SPLITZIP_ERR_INVALID_ARG;
    uint64_t cap = 0, ws = 0;
    int st = splitzip_max_compressed_size(piece_elems, dtype, chunk, &cap);
    if (st != SPLITZIP_OK) return st;
    if ((st = splitzip_encode_workspace_size(piece_elems, dtype, chunk, &ws)) != SPLITZIP_OK) return st;
    const uint64_t eb = elem_bytes(dtype);
    p->piece_elems = piece_elems;
    p->pieces = (n + piece_elems - 1) / piece_elems;
    // raw pieces cross the link as they are
    const uint64_t slot = compress ? cap : piece_elems * eb;
    p->align = slot_align(slot);
    p->cap = align_up(slot, p->align);
    p->ws_bytes = compress ? a16(ws) : 0;
    const uint64_t ring = std::min<uint64_t>(kRing, p->pieces);
    p->send_off = 0;
    p->recv_off = compress ? ring * p->cap : 0;
    p->ws_off = p->recv_off + (compress ? ring * p->cap : 0);
    p->info_off = p->ws_off + p->ws_bytes;
    // + room to round a 16-byte-aligned base up to the slot alignment
    p->device_bytes = compress ? (p->align - 16u) + p->info_off + sizeof(PieceInfo) * p->pieces : 0;
    p->stage_off = 0;
    p->hinfo_off = ring * p->cap;
    p->host_bytes = (p->align - 16u) + p->hinfo_off + (compress ? sizeof(PieceInfo) * p->pieces : 0);
    return SPLITZIP_OK;
}

struct Streams {
    cudaStream_t s[4] = {nullptr, nullptr, nullptr, nullptr};  // encode, D2H, H2D, decode
    cudaEvent_t info[kRing], d2h[kRing], h2d[kRing], dec[kRing];
    cudaEvent_t t0 = nullptr, t1 = nullptr, entry = nullptr;
    cudaEvent_t join[4] = {nullptr, nullptr, nullptr, nullptr};  // each stream's last work, at the end
    bool ok = true;
    Streams() {
        for (auto& x : s) ok &= cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking) == cudaSuccess;
        for (auto& e : join) ok &= cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
        for (int k = 0; k < kRing; ++k) {
            info[k] = d2h[k] = h2d[k] = dec[k] = nullptr;
            ok &= cudaEventCreateWithFlags(&info[k], cudaEventDisableTiming) == cudaSuccess;
            ok &= cudaEventCreateWithFlags(&d2h[k], cudaEventDisableTiming) == cudaSuccess;
            ok &= cudaEventCreateWithFlags(&h2d[k], cudaEventDisableTiming) == cudaSuccess;
            ok &= cudaEventCreateWithFlags(&dec[k], cudaEventDisableTiming) == cudaSuccess;
        }
        ok &= cudaEventCreate(&t0) == cudaSuccess;
        ok &= cudaEventCreate(&t1) == cudaSuccess;
        ok &= cudaEventCreateWithFlags(&entry, cudaEventDisableTiming) == cudaSuccess;
    }
    ~Streams() {
        for (auto x : s)
            if (x) cudaStreamDestroy(x);
        for (int k = 0; k < kRing; ++k) {
            for (cudaEvent_t e : {info[k], d2h[k], h2d[k], dec[k]})
                if (e) cudaEventDestroy(e);
        }
        for (cudaEvent_t e : {t0, t1, entry, join[0], join[1], join[2], join[3]})
            if (e) cudaEventDestroy(e);
    }
};

// Stream sets are pooled per device: a call leases one (creating it only when
// every set is in use) and returns it, so repeated transfers (a request's
// layers one after another) create no streams or events, and concurrent calls
// each hold their own set.  Every wait a call issues is on an event that the
// same call recorded first, so a set carries nothing from one call to the
// next.  The sets live as long as the process: a static destructor could run
// after the CUDA runtime has shut down.
constexpr int kPoolDevices = 64;
std::mutex g_pool_mutex;
std::vector<Streams*> g_pool[kPoolDevices];

class StreamsLease {
  public:
    StreamsLease() {
        if (cudaGetDevice(&dev_) != cudaSuccess || dev_ < 0 || dev_ >= kPoolDevices) {
            dev_ = -1;
            return;
        }
        {
            std::lock_guard<std::mutex> lock(g_pool_mutex);
            if (!g_pool[dev_].empty()) {
                s_ = g_pool[dev_].back();
                g_pool[dev_].pop_back();
            }
        }
        if (!s_) {
            s_ = new Streams();
            if (!s_->ok) {
                delete s_;
                s_ = nullptr;
            }
        }
    }
    ~StreamsLease() {
        if (!s_) return;
        std::lock_guard<std::mutex> lock(g_pool_mutex);
        g_pool[dev_].push_back(s_);
    }
    StreamsLease(const StreamsLease&) = delete;
    StreamsLease& operator=(const StreamsLease&) = delete;
    Streams* get() const { return s_; }

  private:
    int dev_ = -1;
    Streams* s_ = nullptr;
};

// Page-locked host memory; *mapped = its address in the device's address
// space, or null if it has none.
bool is_pinned_host(const void* p, void** mapped) {
    cudaPointerAttributes attr;
    *mapped = nullptr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (attr.type != cudaMemoryTypeHost) return false;
    *mapped = attr.devicePointer;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int splitzip_transfer_scratch_size(uint64_t n, int dtype, uint32_t chunk_elems, uint64_t piece_elems,
                                              int compress, uint64_t* out_device_bytes, uint64_t* out_host_bytes) {
    if (!out_device_bytes || !out_host_bytes) return SPLITZIP_ERR_INVALID_ARG;
    Plan p;
    const int st = plan_for(n, dtype, chunk_elems, piece_elems, compress, &p);
    if (st != SPLITZIP_OK) return st;
    *out_device_bytes = p.device_bytes;
    *out_host_bytes = p.host_bytes;
    return SPLITZIP_OK;
}

extern "C" int splitzip_transfer(const void* d_src, void* d_dst, uint64_t n, int dtype,
                                 const splitzip_codebook_t* cb, uint32_t chunk_elems, uint64_t piece_elems,
                                 int compress, void* d_scratch, uint64_t d_scratch_bytes, void* h_stage,
                                 uint64_t h_stage_bytes, uint64_t* out_link_bytes, float* out_ms,
                                 cudaStream_t stream) {
    if (dtype != SPLITZIP_BF16 && dtype != SPLITZIP_FP8_E5M2 && dtype != SPLITZIP_FP16) return SPLITZIP_ERR_INVALID_ARG;
    if (compress != 0 && compress != 1) return SPLITZIP_ERR_INVALID_ARG;
    Plan p;
    int st = plan_for(n, dtype, chunk_elems, piece_elems, compress, &p);
    if (st != SPLITZIP_OK) return st;
    if (!d_src || !d_dst || !h_stage || !aligned16(d_src) || !aligned16(d_dst) || !aligned16(h_stage))
        return SPLITZIP_ERR_INVALID_ARG;
    if (compress && (!cb || !d_scratch || !aligned16(d_scratch))) return SPLITZIP_ERR_INVALID_ARG;
    if (d_scratch_bytes < p.device_bytes || h_stage_bytes < p.host_bytes) return SPLITZIP_ERR_CAPACITY;
    void* h_stage_mapped = nullptr;  // the link copies need page-locked memory
    if (!is_pinned_host(h_stage, &h_stage_mapped)) return SPLITZIP_ERR_INVALID_ARG;

    const StreamsLease lease;
    if (!lease.get()) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    Streams& S = *lease.get();
    const uint64_t eb = elem_bytes(dtype);
    const uint8_t* src = static_cast<const uint8_t*>(d_src);
    uint8_t* dst = static_cast<uint8_t*>(d_dst);
    // both scratch areas start at the slot alignment
    auto aligned_base = [&](void* b) {
        const uintptr_t u = reinterpret_cast<uintptr_t>(b);
        return reinterpret_cast<uint8_t*>(align_up(u, p.align));
    };
    uint8_t* dev = compress ? aligned_base(d_scratch) : nullptr;
    uint8_t* host = aligned_base(h_stage);
    const uint64_t host_pad = uint64_t(host - static_cast<uint8_t*>(h_stage));
    PieceInfo* dinfo = compress ? reinterpret_cast<PieceInfo*>(dev + p.info_off) : nullptr;
    PieceInfo* hinfo = compress ? reinterpret_cast<PieceInfo*>(host + p.hinfo_off) : nullptr;
    // the same records as the device sees them (null: copy them instead)
    PieceInfo* hinfo_mapped =
        compress && h_stage_mapped
            ? reinterpret_cast<PieceInfo*>(static_cast<uint8_t*>(h_stage_mapped) + host_pad + p.hinfo_off)
            : nullptr;
    cudaStream_t s_enc = S.s[0], s_d2h = S.s[1], s_h2d = S.s[2], s_dec = S.s[3];
    bool cuda_ok = true;
    auto ok = [&](cudaError_t e) { cuda_ok &= e == cudaSuccess; };

    // every internal stream starts after the caller's earlier work
    ok(cudaEventRecord(S.entry, stream));
    for (auto x : S.s) ok(cudaStreamWaitEvent(x, S.entry, 0));
    ok(cudaEventRecord(S.t0, s_enc));
    for (auto x : S.s) ok(cudaStreamWaitEvent(x, S.t0, 0));

    uint64_t link = 0;
    auto piece_len = [&](uint64_t i) { return std::min<uint64_t>(p.piece_elems, n - i * p.piece_elems); };

    if (!compress) {
        for (uint64_t i = 0; i < p.pieces && cuda_ok; ++i) {
            const int k = int(i % kRing);
            const uint64_t bytes = piece_len(i) * eb;
            if (i >= kRing) ok(cudaStreamWaitEvent(s_d2h, S.h2d[k], 0));  // staging slot free
            ok(cudaMemcpyAsync(host + k * p.cap, src + i * p.piece_elems * eb, bytes, cudaMemcpyDeviceToHost,
                               s_d2h));
            ok(cudaEventRecord(S.d2h[k], s_d2h));
            ok(cudaStreamWaitEvent(s_h2d, S.d2h[k], 0));
            ok(cudaMemcpyAsync(dst + i * p.piece_elems * eb, host + k * p.cap, bytes, cudaMemcpyHostToDevice,
                               s_h2d));
            ok(cudaEventRecord(S.h2d[k], s_h2d));
            link += bytes;
        }
    } else {
        // the link and decode stages of piece j, once its container size is known
        auto finish = [&](uint64_t j) -> int {
            const int k = int(j % kRing);
            if (cudaEventSynchronize(S.info[k]) != cudaSuccess) return SPLITZIP_ERR_CUDA;
            if (hinfo[j].enc_status != SPLITZIP_OK) return hinfo[j].enc_status;
            const uint64_t size = hinfo[j].size;
            if (size > p.cap) return SPLITZIP_ERR_CORRUPT;
            uint8_t* send = dev + p.send_off + k * p.cap;
            uint8_t* recv = dev + p.recv_off + k * p.cap;
            uint8_t* stage = host + p.stage_off + k * p.cap;
            if (j >= kRing) ok(cudaStreamWaitEvent(s_d2h, S.h2d[k], 0));  // staging slot free
            ok(cudaMemcpyAsync(stage, send, size, cudaMemcpyDeviceToHost, s_d2h));
            ok(cudaEventRecord(S.d2h[k], s_d2h));
            ok(cudaStreamWaitEvent(s_h2d, S.d2h[k], 0));
            if (j >= kRing) ok(cudaStreamWaitEvent(s_h2d, S.dec[k], 0));  // receive slot free
            ok(cudaMemcpyAsync(recv, stage, size, cudaMemcpyHostToDevice, s_h2d));
            ok(cudaEventRecord(S.h2d[k], s_h2d));
            ok(cudaStreamWaitEvent(s_dec, S.h2d[k], 0));
            const int d = splitzip_decode(recv, size, dst + j * p.piece_elems * eb, piece_len(j), dtype,
                                          &dinfo[j].dec_status, s_dec);
            if (d != SPLITZIP_OK) return d;
            ok(cudaEventRecord(S.dec[k], s_dec));
            link += size;
            return cuda_ok ? SPLITZIP_OK : SPLITZIP_ERR_CUDA;
        };
        for (uint64_t i = 0; i < p.pieces && st == SPLITZIP_OK; ++i) {
            const int k = int(i % kRing);
            if (i >= kRing) ok(cudaStreamWaitEvent(s_enc, S.d2h[k], 0));  // send slot free
            st = splitzip_encode(src + i * p.piece_elems * eb, piece_len(i), dtype, cb, chunk_elems,
                                 dev + p.send_off + k * p.cap, p.cap, dev + p.ws_off, p.ws_bytes, &dinfo[i].size,
                                 &dinfo[i].enc_status, s_enc);
            if (st != SPLITZIP_OK) break;
            if (hinfo_mapped) {
                publish_info_kernel<<<1, 1, 0, s_enc>>>(&dinfo[i], &hinfo_mapped[i]);
                ok(cudaGetLastError());
            } else {
                ok(cudaMemcpyAsync(&hinfo[i], &dinfo[i], 12, cudaMemcpyDeviceToHost, s_enc));  // size + status
            }
            ok(cudaEventRecord(S.info[k], s_enc));
            if (!cuda_ok) st = SPLITZIP_ERR_CUDA;
            // piece i encodes while the host places piece i - 1 on the link
            if (st == SPLITZIP_OK && i >= 1) st = finish(i - 1);
        }
        if (st == SPLITZIP_OK) st = finish(p.pieces - 1);
    }

    // join: the last operations of every stream before the end event
    for (int q = 0; q < 4; ++q) {
        ok(cudaEventRecord(S.join[q], S.s[q]));
        ok(cudaStreamWaitEvent(s_dec, S.join[q], 0));
    }
    ok(cudaEventRecord(S.t1, s_dec));
    ok(cudaStreamWaitEvent(stream, S.t1, 0));
    if (cudaEventSynchronize(S.t1) != cudaSuccess) cuda_ok = false;
    if (!cuda_ok) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    if (st != SPLITZIP_OK) return st;
    if (compress) {
        // every decode's status
        std::vector<PieceInfo> info(p.pieces);
        if (cudaMemcpy(info.data(), dinfo, sizeof(PieceInfo) * p.pieces, cudaMemcpyDeviceToHost) != cudaSuccess) {
            cudaGetLastError();
            return SPLITZIP_ERR_CUDA;
        }
        for (const PieceInfo& x : info)
            if (x.dec_status != SPLITZIP_OK) return x.dec_status;
    }
    if (out_ms && cudaEventElapsedTime(out_ms, S.t0, S.t1) != cudaSuccess) {
        cudaGetLastError();
        return SPLITZIP_ERR_CUDA;
    }
    if (out_link_bytes) *out_link_bytes = link;
    return SPLITZIP_OK;
}
