/*
 * SplitZip oracle: a plain, slow, scalar CPU implementation of the SplitZip
 * lossless KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this library.  The product path
 * (lossless_kv_cache_gb300/) never links, imports or calls it, and shares no
 * source, header, table or helper with it.
 *
 * Source of the method: "SplitZip: Ultra Fast Lossless KV Compression for
 * Disaggregated LLM Serving" (gist.science summary page), section "Method:
 * SplitZip".  Each function below names the part of that section it follows.
 * The page prints no code, no equations and no byte format; every point it
 * leaves open is taken with the plainest reading and marked READING below:
 *
 *   READING R1  Top-16 selection: exponent values ordered by (count desc,
 *               value asc); exponents with zero count fill remaining slots in
 *               ascending value order, so the codebook always holds 16
 *               distinct values (E5M2: drawn from 0..31).
 *   READING R2  code i = the i-th selected exponent (code 0 = most frequent).
 *   READING R3  BF16 sign|mantissa byte = (sign << 7) | mantissa7.
 *   READING R4  two codes per byte: even element in the low nibble, odd
 *               element in the high nibble; a missing final odd element
 *               leaves the high nibble 0.
 *   READING R5  an escaped element stores code 0 in the nibble stream.
 *   READING R6  escape exponent byte = the full original exponent (BF16 8-bit;
 *               E5M2 5-bit value zero-extended to 8 bits).
 *   READING R7  E5M2 sign|mantissa: s3 = (sign << 2) | mantissa2, packed as an
 *               LSB-first bitstream, element i at bits [3i, 3i+3); the stream
 *               is padded with zero bits to whole 3-byte groups of 8 elements.
 *   READING R8  container layout (little-endian, sections 16-byte aligned,
 *               padding zero):
 *                 0   u32 magic 0x50495A53      4  u16 version 1
 *                 6   u8  dtype (0 BF16, 1 E5M2) 7  u8  reserved 0
 *                 8   u64 n                     16  u32 chunk_elems
 *                 20  u32 n_chunks C            24  u64 total escapes E
 *                 32  u8  codebook[16]          48  16 reserved zero bytes
 *                 64  u64 esc_offset[C] (exclusive prefix of the counts)
 *                 64+8C u32 esc_count[C]
 *                 A16 nibble stream ceil(n/2) bytes
 *                 A16 sign|mantissa stream (BF16 n bytes, E5M2 3*ceil(n/8))
 *                 A16 escape records, E x 3 bytes (chunk-major, ascending
 *                     in-chunk position); the blob ends here.
 *   READING R9  one escape record = 3 bytes: the 16-bit in-chunk position
 *               (little-endian) then the 8-bit exponent, exactly the
 *               (position, exponent) pair the page describes.
 *   READING R10 fixed chunk_elems, a power of two in [64, 65536] (the 16-bit
 *               position field bounds it); the final chunk may be short.
 *   READING R11 the 16-bit position is the in-chunk index.
 *   READING R12 no value is special: NaN, inf, zero and subnormal exponents
 *               are ordinary exponent values; there is no float arithmetic.
 *   READING R16 FP16 (dtype 2; the page's "other formats", Significance): the
 *               5-bit exponent (bits 14..10) is coded through the Top-16
 *               codebook exactly as E5M2's; sign|mantissa s11 = (sign << 10) |
 *               mantissa10, packed as an LSB-first bitstream, element i at bits
 *               [11i, 11i+11), padded with zero bits to 11*ceil(n/8) bytes;
 *               the escape exponent byte is the 5-bit value zero-extended.
 *               4 + 11 = 15 bits per element bound the ratio by 16/15.
 */
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define OR_BF16 0
#define OR_E5M2 1
#define OR_FP16 2

#define OR_OK 0
#define OR_INVALID 1
#define OR_CAPACITY 2
#define OR_CORRUPT 3

#define OR_MAGIC 0x50495A53u
#define OR_VERSION 1u
#define OR_HEADER_BYTES 64u

/* ---------- little-endian byte helpers (no host-endianness assumption) ---- */

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static void put_u32(uint8_t* p, uint32_t v) { for (int i = 0; i < 4; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static void put_u64(uint8_t* p, uint64_t v) { for (int i = 0; i < 8; i++) p[i] = (uint8_t)(v >> (8 * i)); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static uint32_t get_u32(const uint8_t* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; i++) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const uint8_t* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; i++) v |= (uint64_t)p[i] << (8 * i);
    return v;
}
static uint64_t align16(uint64_t x) { return (x + 15u) & ~(uint64_t)15u; }

/* ---------- the per-element split (Method: "Key insight", "Sign/mantissa
 * preservation"): redundancy sits in the exponent field, sign and mantissa are
 * kept raw.  BF16 bit 15 = sign, bits 14..7 = exponent, bits 6..0 = mantissa.
 * E5M2 bit 7 = sign, bits 6..2 = exponent, bits 1..0 = mantissa. -------------- */

static int valid_dtype(int dtype) { return dtype == OR_BF16 || dtype == OR_E5M2 || dtype == OR_FP16; }

static unsigned exponent_bins(int dtype) { return dtype == OR_BF16 ? 256u : 32u; }

/* bits of one element's sign|mantissa field in the packed streams (E5M2,
 * FP16; BF16 stores it as one byte) */
static unsigned sm_bits(int dtype) { return dtype == OR_FP16 ? 11u : 3u; }

static unsigned read_element(const void* x, int dtype, uint64_t i) {
    if (dtype != OR_E5M2) {
        const uint8_t* p = (const uint8_t*)x + 2 * i;
        return (unsigned)p[0] | ((unsigned)p[1] << 8);
    }
    return ((const uint8_t*)x)[i];
}

static void write_element(void* out, int dtype, uint64_t i, unsigned v) {
    if (dtype != OR_E5M2) {
        uint8_t* p = (uint8_t*)out + 2 * i;
        p[0] = (uint8_t)v;
        p[1] = (uint8_t)(v >> 8);
    } else {
        ((uint8_t*)out)[i] = (uint8_t)v;
    }
}

static unsigned exponent_of(int dtype, unsigned v) {
    if (dtype == OR_BF16) return (v >> 7) & 0xFFu;
    if (dtype == OR_FP16) return (v >> 10) & 0x1Fu;
    return (v >> 2) & 0x1Fu;
}

/* sign|mantissa field: READING R3 (BF16), READING R7 (E5M2), READING R16
 * (FP16). */
static unsigned sign_mantissa_of(int dtype, unsigned v) {
    if (dtype == OR_BF16) return (((v >> 15) & 1u) << 7) | (v & 0x7Fu);
    if (dtype == OR_FP16) return (((v >> 15) & 1u) << 10) | (v & 0x3FFu);
    return (((v >> 7) & 1u) << 2) | (v & 0x3u);
}

/* inverse of the split: put sign, exponent and mantissa back in place. */
static unsigned join_fields(int dtype, unsigned sm, unsigned e) {
    if (dtype == OR_BF16) return (((sm >> 7) & 1u) << 15) | ((e & 0xFFu) << 7) | (sm & 0x7Fu);
    if (dtype == OR_FP16) return (((sm >> 10) & 1u) << 15) | ((e & 0x1Fu) << 10) | (sm & 0x3FFu);
    return (((sm >> 2) & 1u) << 7) | ((e & 0x1Fu) << 2) | (sm & 0x3u);
}

/* ---------- container geometry (READING R8) -------------------------------- */

static uint64_t sm_stream_bytes(int dtype, uint64_t n) {
    if (dtype == OR_BF16) return n;
    if (dtype == OR_FP16) return 11u * ((n + 7u) / 8u);
    return 3u * ((n + 7u) / 8u);
}

typedef struct {
    uint64_t n_chunks;
    uint64_t index_off, counts_off, nib_off, sm_off, rec_off, size;
} layout_t;

static layout_t layout_of(uint64_t n, int dtype, uint32_t chunk, uint64_t E) {
    layout_t L;
    L.n_chunks = (n + chunk - 1u) / chunk;
    L.index_off = OR_HEADER_BYTES;
    L.counts_off = L.index_off + 8u * L.n_chunks;
    L.nib_off = align16(L.counts_off + 4u * L.n_chunks);
    L.sm_off = L.nib_off + align16((n + 1u) / 2u);
    L.rec_off = L.sm_off + align16(sm_stream_bytes(dtype, n));
    L.size = L.rec_off + 3u * E;
    return L;
}

static int valid_chunk(uint32_t chunk) {
    return chunk >= 64u && chunk <= 65536u && (chunk & (chunk - 1u)) == 0u;
}

uint64_t oracle_container_size(uint64_t n, int dtype, uint32_t chunk, uint64_t total_escapes) {
    return layout_of(n, dtype, chunk, total_escapes).size;
}

/* ---------- histogram (calibration input; Results, "Ablations: Calibration":
 * one codebook calibrated offline) ------------------------------------------- */

int oracle_histogram(const void* x, uint64_t n, int dtype, uint64_t* hist256) {
    if (!hist256 || (n && !x) || !valid_dtype(dtype)) return OR_INVALID;
    for (int b = 0; b < 256; b++) hist256[b] = 0;
    for (uint64_t i = 0; i < n; i++) hist256[exponent_of(dtype, read_element(x, dtype, i))]++;
    return OR_OK;
}

/* ---------- Top-16 codebook (Method, "Fixed-length coding": the most frequent
 * exponent values, chosen offline, each get a 4-bit code).  READINGS R1, R2.
 * Plain selection: sixteen times, take the unchosen value with the largest
 * count, the smaller value on a tie. ------------------------------------------ */

int oracle_calibrate(const uint64_t* hist256, int dtype, uint8_t* cb16) {
    if (!hist256 || !cb16 || !valid_dtype(dtype)) return OR_INVALID;
    unsigned bins = exponent_bins(dtype);
    for (unsigned b = bins; b < 256; b++)
        if (hist256[b] != 0) return OR_INVALID;
    int chosen[256] = {0};
    for (int k = 0; k < 16; k++) {
        int best = -1;
        for (unsigned v = 0; v < bins; v++) {
            if (chosen[v]) continue;
            if (best < 0 || hist256[v] > hist256[best]) best = (int)v;
        }
        chosen[best] = 1;
        cb16[k] = (uint8_t)best;
    }
    return OR_OK;
}

/* code of exponent e: its index in the codebook, or -1 for an escape
 * (Method, "Escape stream": values outside the Top-16 set escape). */
static int code_of(const uint8_t* cb16, unsigned e) {
    for (int k = 0; k < 16; k++)
        if (cb16[k] == e) return k;
    return -1;
}

static int valid_codebook(const uint8_t* cb16, int dtype) {
    unsigned bins = exponent_bins(dtype);
    for (int a = 0; a < 16; a++) {
        if (cb16[a] >= bins) return 0;
        for (int b = a + 1; b < 16; b++)
            if (cb16[a] == cb16[b]) return 0;
    }
    return 1;
}

/* per-chunk escape counts: the number of elements of each chunk whose exponent
 * is outside the codebook. */
int oracle_chunk_escape_counts(const void* x, uint64_t n, int dtype, const uint8_t* cb16,
                               uint32_t chunk, uint32_t* counts) {
    if ((n && (!x || !counts)) || !cb16 || !valid_dtype(dtype) ||
        !valid_chunk(chunk) || !valid_codebook(cb16, dtype))
        return OR_INVALID;
    uint64_t C = (n + chunk - 1u) / chunk;
    for (uint64_t c = 0; c < C; c++) counts[c] = 0;
    for (uint64_t i = 0; i < n; i++)
        if (code_of(cb16, exponent_of(dtype, read_element(x, dtype, i))) < 0) counts[i / chunk]++;
    return OR_OK;
}

/* ---------- encode (Method, "Encoding strategy") -----------------------------
 * For every element in order: split off the exponent; map it through the
 * codebook to a 4-bit code, or, when it is not in the Top-16, record
 * (16-bit in-chunk position, 8-bit exponent) in the chunk's escape list and
 * store code 0 (R5); pack the codes two per byte (R4); store sign|mantissa raw
 * (R3, R7).  Then write the header and index (R8). */

int oracle_encode(const void* x, uint64_t n, int dtype, const uint8_t* cb16, uint32_t chunk,
                  uint8_t* out, uint64_t capacity, uint64_t* out_size) {
    if ((n && !x) || !cb16 || !out || !out_size || !valid_dtype(dtype) ||
        !valid_chunk(chunk) || !valid_codebook(cb16, dtype))
        return OR_INVALID;
    uint64_t C = (n + chunk - 1u) / chunk;
    if (C > 0xFFFFFFFFull) return OR_INVALID;

    /* pass 1: escape counts per chunk, so the sections can be placed */
    uint32_t* counts = (uint32_t*)calloc(C ? C : 1, sizeof(uint32_t));
    if (!counts) return OR_CAPACITY;
    oracle_chunk_escape_counts(x, n, dtype, cb16, chunk, counts);
    uint64_t E = 0;
    for (uint64_t c = 0; c < C; c++) E += counts[c];

    layout_t L = layout_of(n, dtype, chunk, E);
    if (L.size > capacity) {
        free(counts);
        return OR_CAPACITY;
    }
    memset(out, 0, L.size);

    /* header */
    put_u32(out + 0, OR_MAGIC);
    put_u16(out + 4, OR_VERSION);
    out[6] = (uint8_t)dtype;
    out[7] = 0;
    put_u64(out + 8, n);
    put_u32(out + 16, chunk);
    put_u32(out + 20, (uint32_t)C);
    put_u64(out + 24, E);
    for (int k = 0; k < 16; k++) out[32 + k] = cb16[k];

    /* index: exclusive prefix of the counts, then the counts */
    uint64_t running = 0;
    for (uint64_t c = 0; c < C; c++) {
        put_u64(out + L.index_off + 8u * c, running);
        put_u32(out + L.counts_off + 4u * c, counts[c]);
        running += counts[c];
    }

    /* pass 2: the element streams and the escape records */
    uint64_t next_escape = 0;
    for (uint64_t i = 0; i < n; i++) {
        unsigned v = read_element(x, dtype, i);
        unsigned e = exponent_of(dtype, v);
        unsigned sm = sign_mantissa_of(dtype, v);
        int code = code_of(cb16, e);
        if (code < 0) {
            uint64_t pos = i % chunk;
            put_u16(out + L.rec_off + 3u * next_escape, (uint16_t)pos);
            out[L.rec_off + 3u * next_escape + 2u] = (uint8_t)e;
            next_escape++;
            code = 0;
        }
        out[L.nib_off + i / 2] |= (uint8_t)((unsigned)code << (4u * (unsigned)(i % 2)));
        if (dtype == OR_BF16) {
            out[L.sm_off + i] = (uint8_t)sm;
        } else {
            unsigned w = sm_bits(dtype);
            for (unsigned b = 0; b < w; b++) {
                if ((sm >> b) & 1u) {
                    uint64_t bit = (uint64_t)w * i + b;
                    out[L.sm_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
                }
            }
        }
    }
    free(counts);
    *out_size = L.size;
    return OR_OK;
}

/* ---------- header parse and validation ------------------------------------ */

typedef struct {
    uint64_t n, total_escapes, size;
    uint32_t chunk_elems, n_chunks;
    uint8_t dtype;
    uint8_t codebook[16];
} oracle_header_t;

int oracle_parse_header(const uint8_t* blob, uint64_t bytes, oracle_header_t* h) {
    if (!blob || !h) return OR_INVALID;
    if (bytes < OR_HEADER_BYTES) return OR_CORRUPT;
    if (get_u32(blob) != OR_MAGIC || get_u16(blob + 4) != OR_VERSION) return OR_CORRUPT;
    if (!valid_dtype(blob[6])) return OR_CORRUPT;
    if (blob[7] != 0) return OR_CORRUPT;
    for (int k = 48; k < 64; k++)
        if (blob[k] != 0) return OR_CORRUPT;
    h->dtype = blob[6];
    h->n = get_u64(blob + 8);
    h->chunk_elems = get_u32(blob + 16);
    h->n_chunks = get_u32(blob + 20);
    h->total_escapes = get_u64(blob + 24);
    for (int k = 0; k < 16; k++) h->codebook[k] = blob[32 + k];
    if (!valid_chunk(h->chunk_elems)) return OR_CORRUPT;
    if ((h->n + h->chunk_elems - 1u) / h->chunk_elems != h->n_chunks) return OR_CORRUPT;
    if (h->total_escapes > h->n) return OR_CORRUPT;
    if (!valid_codebook(h->codebook, h->dtype)) return OR_CORRUPT;
    h->size = layout_of(h->n, h->dtype, h->chunk_elems, h->total_escapes).size;
    if (h->size > bytes) return OR_CORRUPT;
    return OR_OK;
}

/* ---------- decode (Method, "Decoding strategy") -----------------------------
 * Dense path ("Parallelism"): every nibble is unpacked and mapped through the
 * 16-entry table back to an exponent, then joined with its sign|mantissa.
 * Correction ("Correction"): the escape records then overwrite the exponents
 * of the escaped elements with their original values. */

int oracle_decode(const uint8_t* blob, uint64_t bytes, void* out, uint64_t n, int dtype) {
    if (!blob || (n && !out) || !valid_dtype(dtype)) return OR_INVALID;
    oracle_header_t h;
    int st = oracle_parse_header(blob, bytes, &h);
    if (st != OR_OK) return st;
    if (h.dtype != dtype || h.n != n) return OR_CORRUPT;
    layout_t L = layout_of(n, dtype, h.chunk_elems, h.total_escapes);
    uint64_t C = h.n_chunks, chunk = h.chunk_elems;

    /* index consistency: counts fit their chunk, offsets are the prefix */
    uint64_t running = 0;
    for (uint64_t c = 0; c < C; c++) {
        uint64_t off = get_u64(blob + L.index_off + 8u * c);
        uint64_t cnt = get_u32(blob + L.counts_off + 4u * c);
        uint64_t len = (c + 1 < C) ? chunk : n - c * chunk;
        if (off != running || cnt > len) return OR_CORRUPT;
        running += cnt;
    }
    if (running != h.total_escapes) return OR_CORRUPT;

    /* dense path */
    for (uint64_t i = 0; i < n; i++) {
        unsigned code = (blob[L.nib_off + i / 2] >> (4u * (unsigned)(i % 2))) & 0xFu;
        unsigned e = h.codebook[code];
        unsigned sm;
        if (dtype == OR_BF16) {
            sm = blob[L.sm_off + i];
        } else {
            unsigned w = sm_bits(dtype);
            sm = 0;
            for (unsigned b = 0; b < w; b++) {
                uint64_t bit = (uint64_t)w * i + b;
                sm |= ((blob[L.sm_off + bit / 8] >> (bit % 8)) & 1u) << b;
            }
        }
        write_element(out, dtype, i, join_fields(dtype, sm, e));
    }

    /* correction: positions strictly ascending within the chunk */
    for (uint64_t c = 0; c < C; c++) {
        uint64_t off = get_u64(blob + L.index_off + 8u * c);
        uint64_t cnt = get_u32(blob + L.counts_off + 4u * c);
        uint64_t len = (c + 1 < C) ? chunk : n - c * chunk;
        for (uint64_t j = 0; j < cnt; j++) {
            const uint8_t* rec = blob + L.rec_off + 3u * (off + j);
            uint64_t pos = get_u16(rec);
            unsigned e = rec[2];
            if (pos >= len) return OR_CORRUPT;
            if (j > 0 && pos <= get_u16(rec - 3)) return OR_CORRUPT;
            if (e >= exponent_bins(dtype)) return OR_CORRUPT;
            uint64_t i = c * chunk + pos;
            unsigned v = read_element(out, dtype, i);
            write_element(out, dtype, i, join_fields(dtype, sign_mantissa_of(dtype, v), e));
        }
    }
    return OR_OK;
}

/* ======================= ablation variants ==================================
 * Results, "Ablation Studies" (and Method, the design choice of Top-16 over
 * Top-15): the page compares Top-16 with Top-8 (fewer exponents, 3-bit codes:
 * lower coverage, more escapes, less efficient packing) and with Top-15 plus a
 * sentinel (one code marks an escape; escape positions are not stored but found
 * from the sentinels: less metadata, irregular decoding).  It gives no format
 * for either; the plainest forms of what it describes:
 *
 *   READING V1  both keep the main container's header, index and sign|mantissa
 *               stream; header byte 7 (reserved 0 in the main format) names the
 *               variant: 1 = Top-8, 2 = Top-15 + sentinel (0 = the main format).
 *   READING V2  Top-8: the 8 most frequent exponents (R1 order) get codes 0..7,
 *               packed 3 bits per element, LSB-first (as R7), 3 bytes per 8
 *               elements, zero-padded; escapes exactly as the main format (code
 *               0, 3-byte (position, exponent) records).  Codebook bytes 8..15
 *               are zero.
 *   READING V3  Top-15 + sentinel: the 15 most frequent exponents get codes
 *               0..14; an escaped element stores code 15 (the sentinel) in the
 *               nibble stream; the escape stream holds only the escaped
 *               elements' exponents, one byte each, chunk-major in element
 *               order (the index still gives each chunk's offset and count).
 *               Codebook byte 15 is zero.
 */

static unsigned variant_codes(int variant) { return variant == 1 ? 8u : variant == 2 ? 15u : 16u; }

static layout_t layout_variant(uint64_t n, int dtype, uint32_t chunk, int variant, uint64_t E) {
    layout_t L;
    L.n_chunks = (n + chunk - 1u) / chunk;
    L.index_off = OR_HEADER_BYTES;
    L.counts_off = L.index_off + 8u * L.n_chunks;
    L.nib_off = align16(L.counts_off + 4u * L.n_chunks);
    uint64_t code_bytes = variant == 1 ? 3u * ((n + 7u) / 8u) : (n + 1u) / 2u;
    L.sm_off = L.nib_off + align16(code_bytes);
    L.rec_off = L.sm_off + align16(sm_stream_bytes(dtype, n));
    L.size = L.rec_off + (variant == 2 ? 1u : 3u) * E;
    return L;
}

uint64_t oracle_variant_size(uint64_t n, int dtype, uint32_t chunk, int variant, uint64_t total_escapes) {
    return layout_variant(n, dtype, chunk, variant, total_escapes).size;
}

/* the first k entries distinct and in range, the rest zero */
static int valid_variant_codebook(const uint8_t* cb16, int dtype, int variant) {
    unsigned k = variant_codes(variant), bins = exponent_bins(dtype);
    for (unsigned a = 0; a < 16; a++) {
        if (a >= k) {
            if (cb16[a] != 0) return 0;
            continue;
        }
        if (cb16[a] >= bins) return 0;
        for (unsigned b = a + 1; b < k; b++)
            if (cb16[a] == cb16[b]) return 0;
    }
    return 1;
}

static int code_of_k(const uint8_t* cb16, unsigned k, unsigned e) {
    for (unsigned c = 0; c < k; c++)
        if (cb16[c] == e) return (int)c;
    return -1;
}

/* Encode with one of the variants (V1-V3); variant 0 is the main format.  Same
 * steps as oracle_encode: count the escapes per chunk, place the sections,
 * then per element the code (or the escape), the sign|mantissa bits and the
 * escape entry. */
int oracle_encode_variant(const void* x, uint64_t n, int dtype, const uint8_t* cb16, uint32_t chunk, int variant,
                          uint8_t* out, uint64_t capacity, uint64_t* out_size) {
    if ((n && !x) || !cb16 || !out || !out_size || (dtype != OR_BF16 && dtype != OR_E5M2) ||
        variant < 0 || variant > 2 || !valid_chunk(chunk) || !valid_variant_codebook(cb16, dtype, variant))
        return OR_INVALID;
    unsigned k = variant_codes(variant);
    uint64_t C = (n + chunk - 1u) / chunk;
    if (C > 0xFFFFFFFFull) return OR_INVALID;
    uint32_t* counts = (uint32_t*)calloc(C ? C : 1, sizeof(uint32_t));
    if (!counts) return OR_CAPACITY;
    for (uint64_t i = 0; i < n; i++)
        if (code_of_k(cb16, k, exponent_of(dtype, read_element(x, dtype, i))) < 0) counts[i / chunk]++;
    uint64_t E = 0;
    for (uint64_t c = 0; c < C; c++) E += counts[c];
    layout_t L = layout_variant(n, dtype, chunk, variant, E);
    if (L.size > capacity) {
        free(counts);
        return OR_CAPACITY;
    }
    memset(out, 0, L.size);
    put_u32(out + 0, OR_MAGIC);
    put_u16(out + 4, OR_VERSION);
    out[6] = (uint8_t)dtype;
    out[7] = (uint8_t)variant;
    put_u64(out + 8, n);
    put_u32(out + 16, chunk);
    put_u32(out + 20, (uint32_t)C);
    put_u64(out + 24, E);
    for (int c = 0; c < 16; c++) out[32 + c] = cb16[c];
    uint64_t running = 0;
    for (uint64_t c = 0; c < C; c++) {
        put_u64(out + L.index_off + 8u * c, running);
        put_u32(out + L.counts_off + 4u * c, counts[c]);
        running += counts[c];
    }
    uint64_t next_escape = 0;
    for (uint64_t i = 0; i < n; i++) {
        unsigned v = read_element(x, dtype, i);
        unsigned e = exponent_of(dtype, v);
        unsigned sm = sign_mantissa_of(dtype, v);
        int code = code_of_k(cb16, k, e);
        if (code < 0) {
            if (variant == 2) {
                out[L.rec_off + next_escape] = (uint8_t)e;  /* V3: the exponent only */
                code = 15;
            } else {
                put_u16(out + L.rec_off + 3u * next_escape, (uint16_t)(i % chunk));
                out[L.rec_off + 3u * next_escape + 2u] = (uint8_t)e;
                code = 0;
            }
            next_escape++;
        }
        if (variant == 1) {
            for (unsigned b = 0; b < 3; b++) {
                if (((unsigned)code >> b) & 1u) {
                    uint64_t bit = 3u * i + b;
                    out[L.nib_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
                }
            }
        } else {
            out[L.nib_off + i / 2] |= (uint8_t)((unsigned)code << (4u * (unsigned)(i % 2)));
        }
        if (dtype == OR_BF16) {
            out[L.sm_off + i] = (uint8_t)sm;
        } else {
            for (unsigned b = 0; b < 3; b++) {
                if ((sm >> b) & 1u) {
                    uint64_t bit = 3u * i + b;
                    out[L.sm_off + bit / 8] |= (uint8_t)(1u << (bit % 8));
                }
            }
        }
    }
    free(counts);
    *out_size = L.size;
    return OR_OK;
}

/* Decode a container of any variant (byte 7).  Header and index checks as
 * oracle_decode; dense path per element; then the correction: explicit records
 * (variants 0, 1) as oracle_decode, or, for the sentinel variant, each element
 * with code 15 takes the next exponent of its chunk's escape bytes, and the
 * chunk must hold exactly as many sentinels as its count says. */
int oracle_decode_variant(const uint8_t* blob, uint64_t bytes, void* out, uint64_t n, int dtype) {
    if (!blob || (n && !out) || (dtype != OR_BF16 && dtype != OR_E5M2)) return OR_INVALID;
    if (bytes < OR_HEADER_BYTES) return OR_CORRUPT;
    if (get_u32(blob) != OR_MAGIC || get_u16(blob + 4) != OR_VERSION) return OR_CORRUPT;
    if (blob[6] != (uint8_t)dtype || blob[7] > 2) return OR_CORRUPT;
    for (int b = 48; b < 64; b++)
        if (blob[b] != 0) return OR_CORRUPT;
    int variant = blob[7];
    uint64_t hn = get_u64(blob + 8), E = get_u64(blob + 24);
    uint32_t chunk = get_u32(blob + 16), C = get_u32(blob + 20);
    const uint8_t* cb = blob + 32;
    if (hn != n || !valid_chunk(chunk) || (n + chunk - 1u) / chunk != C || E > n) return OR_CORRUPT;
    if (!valid_variant_codebook(cb, dtype, variant)) return OR_CORRUPT;
    layout_t L = layout_variant(n, dtype, chunk, variant, E);
    if (L.size > bytes) return OR_CORRUPT;
    uint64_t running = 0;
    for (uint64_t c = 0; c < C; c++) {
        uint64_t off = get_u64(blob + L.index_off + 8u * c);
        uint64_t cnt = get_u32(blob + L.counts_off + 4u * c);
        uint64_t len = (c + 1 < C) ? chunk : n - c * chunk;
        if (off != running || cnt > len) return OR_CORRUPT;
        running += cnt;
    }
    if (running != E) return OR_CORRUPT;

    uint64_t sentinels = 0, chunk_start = 0;  /* variant 2: escapes of the current chunk so far */
    for (uint64_t i = 0; i < n; i++) {
        if (i % chunk == 0) {
            if (i > 0 && variant == 2 && sentinels != get_u32(blob + L.counts_off + 4u * (i / chunk - 1)))
                return OR_CORRUPT;
            sentinels = 0;
            chunk_start = get_u64(blob + L.index_off + 8u * (i / chunk));
        }
        unsigned code = 0;
        if (variant == 1) {
            for (unsigned b = 0; b < 3; b++) {
                uint64_t bit = 3u * i + b;
                code |= ((blob[L.nib_off + bit / 8] >> (bit % 8)) & 1u) << b;
            }
        } else {
            code = (blob[L.nib_off + i / 2] >> (4u * (unsigned)(i % 2))) & 0xFu;
        }
        unsigned e;
        if (variant == 2 && code == 15) {
            uint64_t cnt = get_u32(blob + L.counts_off + 4u * (i / chunk));
            if (sentinels >= cnt) return OR_CORRUPT;
            e = blob[L.rec_off + chunk_start + sentinels];
            if (e >= exponent_bins(dtype)) return OR_CORRUPT;
            sentinels++;
        } else {
            e = cb[code];
        }
        unsigned sm;
        if (dtype == OR_BF16) {
            sm = blob[L.sm_off + i];
        } else {
            sm = 0;
            for (unsigned b = 0; b < 3; b++) {
                uint64_t bit = 3u * i + b;
                sm |= ((blob[L.sm_off + bit / 8] >> (bit % 8)) & 1u) << b;
            }
        }
        write_element(out, dtype, i, join_fields(dtype, sm, e));
    }
    if (variant == 2) {
        if (n > 0 && sentinels != get_u32(blob + L.counts_off + 4u * (C - 1))) return OR_CORRUPT;
        return OR_OK;
    }
    for (uint64_t c = 0; c < C; c++) {
        uint64_t off = get_u64(blob + L.index_off + 8u * c);
        uint64_t cnt = get_u32(blob + L.counts_off + 4u * c);
        uint64_t len = (c + 1 < C) ? chunk : n - c * chunk;
        for (uint64_t j = 0; j < cnt; j++) {
            const uint8_t* rec = blob + L.rec_off + 3u * (off + j);
            uint64_t pos = get_u16(rec);
            unsigned e = rec[2];
            if (pos >= len) return OR_CORRUPT;
            if (j > 0 && pos <= get_u16(rec - 3)) return OR_CORRUPT;
            if (e >= exponent_bins(dtype)) return OR_CORRUPT;
            uint64_t i = c * chunk + pos;
            unsigned v = read_element(out, dtype, i);
            write_element(out, dtype, i, join_fields(dtype, sign_mantissa_of(dtype, v), e));
        }
    }
    return OR_OK;
}
