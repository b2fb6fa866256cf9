// Joining containers of consecutive chunk ranges into one container (host).
//
// Chunks are independent: a chunk's nibbles, sign|mantissa bytes and escape
// records depend on its own elements only, and the index holds one offset and
// one count per chunk.  So a tensor can be encoded in pieces of whole chunks
// (one piece per GPU, or per layer) and the piece containers joined later into
// exactly the container of the whole tensor.  The only quantity that crosses
// pieces is the escape offset: the merged offsets of piece i are its own plus
// the escapes of pieces 0..i-1 (an exclusive scan of the per-piece totals E).
// This file has no device code: it works on host copies of the containers.
#include <cstring>
#include <vector>

#include "splitzip_internal.cuh"

using namespace splitzip;

namespace {

uint64_t rd64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
    return v;
}
uint32_t rd32(const uint8_t* p) { return uint32_t(p[0]) | (uint32_t(p[1]) << 8) | (uint32_t(p[2]) << 16) | (uint32_t(p[3]) << 24); }
void wr64(uint8_t* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = uint8_t(v >> (8 * i));
}
void wr32(uint8_t* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = uint8_t(v >> (8 * i));
}

struct Part {
    const uint8_t* b;
    splitzip_header_t h;
};

// Parses and checks the pieces; fills the merged header fields.
int check_parts(const void* const* h_parts, const uint64_t* part_bytes, uint32_t count, std::vector<Part>* parts,
                uint64_t* n, uint64_t* E) {
    if (!h_parts || !part_bytes || count == 0) return SPLITZIP_ERR_INVALID_ARG;
    parts->resize(count);
    *n = 0;
    *E = 0;
    for (uint32_t i = 0; i < count; ++i) {
        Part& p = (*parts)[i];
        if (!h_parts[i]) return SPLITZIP_ERR_INVALID_ARG;
        p.b = static_cast<const uint8_t*>(h_parts[i]);
        const int st = splitzip_parse_header(p.b, part_bytes[i], &p.h);
        if (st != SPLITZIP_OK) return st;
        const splitzip_header_t& f = (*parts)[0].h;
        if (p.h.dtype != f.dtype || p.h.chunk_elems != f.chunk_elems || std::memcmp(p.h.codebook, f.codebook, 16) != 0)
            return SPLITZIP_ERR_INVALID_ARG;  // pieces of different encodings
        if (i + 1 < count && p.h.n_elems % p.h.chunk_elems != 0)
            return SPLITZIP_ERR_INVALID_ARG;  // only the last piece may end in a partial chunk
        // the piece's own index: offsets are the exclusive prefix of its counts
        uint64_t run = 0;
        for (uint32_t c = 0; c < p.h.n_chunks; ++c) {
            const uint32_t k = rd32(p.b + p.h.counts_off + 4ull * c);
            if (rd64(p.b + p.h.index_off + 8ull * c) != run || k > p.h.chunk_elems) return SPLITZIP_ERR_CORRUPT;
            run += k;
        }
        if (run != p.h.total_escapes) return SPLITZIP_ERR_CORRUPT;
        *n += p.h.n_elems;
        *E += p.h.total_escapes;
    }
    if (*n > (uint64_t(1) << 48) || (*n + (*parts)[0].h.chunk_elems - 1) / (*parts)[0].h.chunk_elems > 0xFFFFFFFFull)
        return SPLITZIP_ERR_UNSUPPORTED;
    return SPLITZIP_OK;
}

}  // namespace

extern "C" int splitzip_merge(const void* const* h_parts, const uint64_t* part_bytes, uint32_t count, void* h_out,
                              uint64_t out_capacity, uint64_t* out_bytes) {
    if (!out_bytes) return SPLITZIP_ERR_INVALID_ARG;
    std::vector<Part> parts;
    uint64_t n = 0, E = 0;
    int st = check_parts(h_parts, part_bytes, count, &parts, &n, &E);
    if (st != SPLITZIP_OK) return st;
    const splitzip_header_t& f = parts[0].h;
    const int dtype = f.dtype;
    const Layout L = layout_for(n, dtype, f.chunk_elems, E);
    *out_bytes = L.size;
    if (!h_out) return SPLITZIP_OK;  // size query
    if (out_capacity < L.size) return SPLITZIP_ERR_CAPACITY;

    uint8_t* o = static_cast<uint8_t*>(h_out);
    std::memset(o, 0, L.nibble_off);  // header, index and the padding after it
    wr32(o, kMagic);
    o[4] = uint8_t(kVersion);
    o[5] = uint8_t(kVersion >> 8);
    o[6] = uint8_t(dtype);
    wr64(o + 8, n);
    wr32(o + 16, f.chunk_elems);
    wr32(o + 20, uint32_t(L.n_chunks));
    wr64(o + 24, E);
    std::memcpy(o + 32, f.codebook, 16);

    uint64_t chunk0 = 0, elem0 = 0, esc0 = 0;
    for (const Part& p : parts) {
        const splitzip_header_t& h = p.h;
        // index: the piece's offsets moved by the escapes of the earlier pieces
        for (uint32_t c = 0; c < h.n_chunks; ++c) {
            wr64(o + L.index_off + 8 * (chunk0 + c), rd64(p.b + h.index_off + 8ull * c) + esc0);
            std::memcpy(o + L.counts_off + 4 * (chunk0 + c), p.b + h.counts_off + 4ull * c, 4);
        }
        // dense streams: every piece but the last holds whole chunks (a multiple
        // of 64 elements), so its bytes start on a byte boundary of the stream
        std::memcpy(o + L.nibble_off + elem0 / 2, p.b + h.nibble_off, (h.n_elems + 1) / 2);
        // (elem0 is a multiple of 8: the earlier pieces' streams end on whole bytes)
        std::memcpy(o + L.signmant_off + signmant_bytes(dtype, elem0), p.b + h.signmant_off,
                    signmant_bytes(dtype, h.n_elems));
        std::memcpy(o + L.escrec_off + 3 * esc0, p.b + h.escrec_off, 3 * h.total_escapes);
        chunk0 += h.n_chunks;
        elem0 += h.n_elems;
        esc0 += h.total_escapes;
    }
    // zero padding after the two dense streams
    std::memset(o + L.nibble_off + (n + 1) / 2, 0, L.signmant_off - (L.nibble_off + (n + 1) / 2));
    std::memset(o + L.signmant_off + signmant_bytes(dtype, n), 0,
                L.escrec_off - (L.signmant_off + signmant_bytes(dtype, n)));
    return SPLITZIP_OK;
}
