/*
 * GPULZ oracle: a plain, sequential CPU encoder and decoder of the GPULZ
 * chunked LZSS stream.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library. The product path
 * (the CUDA library) shares no code, header, table or constant with it.
 *
 * Every step follows the GPULZ stage documentation of FZGPUModules
 * ("fz::GPULZStage", stage_gpulz page) and the codebase note CN-GPULZ-1
 * ("match level and split mode"), in the order those pages give:
 *
 *   chunking into chunk_size-byte chunks of word_size-byte elements, one
 *   chunk coded on its own                  -> stage page, class summary
 *   zero padding of the tail chunk           -> stage page, "Alignment"
 *   all-zero chunk sentinel                  -> stage page, zero-chunk fast path
 *   exact longest match over the 32-element
 *   near window (omask + AND of successive
 *   masks), length capped at 255             -> stage page, match-search section
 *   (windows of 33..64 elements for the
 *   window-width study, same section)
 *   hashed two-word-key long-range candidates
 *   over 8 sub-blocks, offsets to 255,
 *   buckets keep max(pos+1)                  -> stage page, match-search section;
 *                                               CN-GPULZ-1 level table
 *   sequential literal/match parse           -> stage page, provenance paragraph
 *   literal = word_size bytes, match =
 *   2-byte [length, offset] token, per-chunk
 *   literal/match flag bitmap                -> stage page, class summary
 *   raw fallback with a high bit on the
 *   chunk's header entry                     -> stage page, raw-fallback paragraph
 *   per-chunk sizes + original size in the
 *   stream header                            -> stage page, graph-capture paragraph
 *
 * Where the pages are silent the oracle takes one documented reading (the
 * repository's design notes list them): minimum match length (a match is
 * taken only when it is shorter than the literal bytes it replaces), ties
 * broken toward the nearest offset, near candidate kept on equal length,
 * the hash function and table size, flag polarity (1 = match, LSB first),
 * and the exact byte layout of the header, size table and blocks.
 *
 * Parity: pinned by the tests under tests/ (brute-force longest match on
 * tiny inputs, closed forms for constant / periodic chunks at both levels,
 * stream invariants, round trip, hand-derived golden streams).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gpulz_oracle.h"

/* ---- stream-format constants (the repository's documented format v1) ---- */
#define ORC_MAGIC 0x5A4C5047u /* "GPLZ" little-endian */
#define ORC_VERSION 1u
#define ORC_HEADER_BYTES 32u
#define ORC_ENTRY_BYTES 8u
#define ORC_RAW_BIT 0x80000000u

/* ---- method constants from the pages ---- */
#define ORC_NEAR_WINDOW 32 /* default 32-element near window */
#define ORC_MAX_WINDOW 64  /* widest near window of the window-width study */
#define ORC_MAX_LEN 255    /* one-byte length field */
#define ORC_MAX_OFF 255    /* one-byte offset field, "offsets to 255" */
#define ORC_SUBBLOCKS 8    /* chunk walked in 8 sub-blocks */

/* Little-endian helpers. */
static void put_u16(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)(v & 0xFF);
    p[1] = (uint8_t)((v >> 8) & 0xFF);
}
static void put_u32(uint8_t* p, uint32_t v) {
    for (int k = 0; k < 4; ++k) p[k] = (uint8_t)((v >> (8 * k)) & 0xFF);
}
static void put_u64(uint8_t* p, uint64_t v) {
    for (int k = 0; k < 8; ++k) p[k] = (uint8_t)((v >> (8 * k)) & 0xFF);
}
static uint32_t get_u16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }
static uint32_t get_u32(const uint8_t* p) {
    uint32_t v = 0;
    for (int k = 0; k < 4; ++k) v |= (uint32_t)p[k] << (8 * k);
    return v;
}
static uint64_t get_u64(const uint8_t* p) {
    uint64_t v = 0;
    for (int k = 0; k < 8; ++k) v |= (uint64_t)p[k] << (8 * k);
    return v;
}

int orc_valid_geometry(int word_size, int chunk_size) {
    if (word_size != 1 && word_size != 2 && word_size != 4) return 0;
    if (chunk_size != 1024 && chunk_size != 2048 && chunk_size != 4096) return 0;
    return 1;
}

int orc_min_match_len(int word_size) {
    /* A match token costs 2 bytes; it is taken only if it replaces more than
     * 2 bytes of literals: len * word_size > 2. */
    int len = 1;
    while (len * word_size <= 2) ++len;
    return len;
}

uint32_t orc_hash_bits(int elems) {
    /* Table of 2*E buckets: bits = log2(2E). */
    uint32_t b = 0;
    while ((1u << b) < (uint32_t)(2 * elems)) ++b;
    return b;
}

uint32_t orc_hash(uint32_t k0, uint32_t k1, uint32_t bits) {
    uint32_t h = (k0 * 0x9E3779B1u) ^ (k1 * 0x85EBCA77u);
    return h >> (32u - bits);
}

uint64_t orc_compress_bound(uint64_t n_bytes, int word_size, int chunk_size) {
    (void)word_size;
    uint64_t chunks = (n_bytes + (uint64_t)chunk_size - 1) / (uint64_t)chunk_size;
    return ORC_HEADER_BYTES + ORC_ENTRY_BYTES * chunks + chunks * (uint64_t)chunk_size;
}

/* ------------------------------------------------------------------------ */
/* Level 0: exact longest match over the near window (32 elements; 33..64   */
/* for the window-width study of the match-search section).                 */
/* ------------------------------------------------------------------------ */
void orc_near_matches(const uint32_t* w, int elems, uint8_t* len_out, uint8_t* off_out) {
    orc_near_matches_w(w, elems, ORC_NEAR_WINDOW, len_out, off_out);
}

void orc_near_matches_w(const uint32_t* w, int elems, int window, uint8_t* len_out,
                        uint8_t* off_out) {
    uint64_t* omask = (uint64_t*)malloc(sizeof(uint64_t) * (size_t)elems);
    /* omask[i] bit (o-1) set iff w[i] == w[i-o], 1 <= o <= window, i-o >= 0. */
    for (int i = 0; i < elems; ++i) {
        uint64_t m = 0;
        for (int o = 1; o <= window; ++o) {
            if (i - o < 0) break;
            if (w[i] == w[i - o]) m |= 1ull << (o - 1);
        }
        omask[i] = m;
    }
    /* AND successive masks: the surviving offsets after k steps are exactly
     * those that match for k consecutive elements. */
    for (int i = 0; i < elems; ++i) {
        uint64_t m = omask[i];
        if (m == 0) {
            len_out[i] = 0;
            off_out[i] = 0;
            continue;
        }
        int cap = elems - i;
        if (cap > ORC_MAX_LEN) cap = ORC_MAX_LEN;
        int len = 1;
        while (len < cap) {
            uint64_t next = m & omask[i + len];
            if (next == 0) break;
            m = next;
            ++len;
        }
        /* nearest surviving offset */
        int off = 1;
        while (((m >> (off - 1)) & 1ull) == 0) ++off;
        len_out[i] = (uint8_t)len;
        off_out[i] = (uint8_t)off;
    }
    free(omask);
}

/* ------------------------------------------------------------------------ */
/* Level 1: hashed two-word-key long-range candidates, 8 sub-blocks.         */
/* Updates (len, off) in place where the hashed candidate is better.         */
/* ------------------------------------------------------------------------ */
void orc_level1_matches(const uint32_t* w, int elems, uint8_t* len_io, uint8_t* off_io) {
    uint32_t bits = orc_hash_bits(elems);
    uint32_t nbuckets = 1u << bits;
    uint32_t* table = (uint32_t*)calloc(nbuckets, sizeof(uint32_t)); /* pos+1, 0 = empty */
    int sub = elems / ORC_SUBBLOCKS;
    for (int s = 0; s < ORC_SUBBLOCKS; ++s) {
        int lo = s * sub, hi = (s + 1) * sub;
        /* lookup: the table holds only positions of earlier sub-blocks */
        for (int i = lo; i < hi; ++i) {
            if (i + 1 >= elems) continue;
            uint32_t slot = table[orc_hash(w[i], w[i + 1], bits)];
            if (slot == 0) continue;
            int p = (int)slot - 1;
            int dist = i - p;
            if (dist < 1 || dist > ORC_MAX_OFF) continue;
            int cap = elems - i;
            if (cap > ORC_MAX_LEN) cap = ORC_MAX_LEN;
            int len1 = 0;
            while (len1 < cap && w[i + len1] == w[p + len1]) ++len1;
            if (len1 == 0) continue;
            int len0 = len_io[i];
            int off0 = off_io[i];
            if (len1 > len0 || (len1 == len0 && dist < off0)) {
                len_io[i] = (uint8_t)len1;
                off_io[i] = (uint8_t)dist;
            }
        }
        /* insert after the lookups of this sub-block; keep the most recent */
        for (int p = lo; p < hi; ++p) {
            if (p + 1 >= elems) continue;
            uint32_t b = orc_hash(w[p], w[p + 1], bits);
            uint32_t v = (uint32_t)p + 1u;
            if (v > table[b]) table[b] = v;
        }
    }
    free(table);
}

/* ------------------------------------------------------------------------ */
/* One chunk: parse, pack, raw decision.                                     */
/* ------------------------------------------------------------------------ */
static uint32_t load_word(const uint8_t* p, int ws) {
    uint32_t v = 0;
    for (int k = 0; k < ws; ++k) v |= (uint32_t)p[k] << (8 * k);
    return v;
}

/* chunk: chunk_size bytes, already zero padded. Writes the block into
 * block_out (capacity >= chunk_size) and the two size-table words. Returns
 * the block's byte length. */
uint32_t orc_encode_chunk(const uint8_t* chunk, int word_size, int chunk_size, int match_level,
                          uint8_t* block_out, uint32_t* entry_items, uint32_t* entry_data) {
    return orc_encode_chunk_w(chunk, word_size, chunk_size, match_level, ORC_NEAR_WINDOW,
                              block_out, entry_items, entry_data);
}

uint32_t orc_encode_chunk_w(const uint8_t* chunk, int word_size, int chunk_size, int match_level,
                            int window, uint8_t* block_out, uint32_t* entry_items,
                            uint32_t* entry_data) {
    int elems = chunk_size / word_size;

    /* zero-chunk sentinel */
    int all_zero = 1;
    for (int k = 0; k < chunk_size; ++k) {
        if (chunk[k] != 0) {
            all_zero = 0;
            break;
        }
    }
    if (all_zero) {
        *entry_items = 0;
        *entry_data = 0;
        return 0;
    }

    uint32_t* w = (uint32_t*)calloc((size_t)elems, sizeof(uint32_t));
    for (int i = 0; i < elems; ++i) w[i] = load_word(chunk + (size_t)i * word_size, word_size);
    uint8_t* len = (uint8_t*)malloc((size_t)elems);
    uint8_t* off = (uint8_t*)malloc((size_t)elems);
    orc_near_matches_w(w, elems, window, len, off);
    if (match_level == 1) orc_level1_matches(w, elems, len, off);

    /* greedy sequential parse */
    int lmin = orc_min_match_len(word_size);
    uint32_t flag_words = ((uint32_t)elems + 31u) / 32u;
    uint32_t* flags = (uint32_t*)calloc(flag_words, sizeof(uint32_t));
    uint8_t* data = (uint8_t*)calloc((size_t)chunk_size * 2u + 8u, 1);
    uint32_t items = 0, dbytes = 0;
    int i = 0;
    while (i < elems) {
        if (len[i] >= lmin) {
            flags[items / 32u] |= 1u << (items % 32u);
            data[dbytes] = len[i];
            data[dbytes + 1] = off[i];
            dbytes += 2;
            i += len[i];
        } else {
            memcpy(data + dbytes, chunk + (size_t)i * word_size, (size_t)word_size);
            dbytes += (uint32_t)word_size;
            i += 1;
        }
        ++items;
    }

    uint32_t fbytes = 4u * ((items + 31u) / 32u);
    uint32_t padded = (dbytes + 3u) & ~3u;
    uint32_t blk = fbytes + padded;
    if (blk >= (uint32_t)chunk_size) {
        memcpy(block_out, chunk, (size_t)chunk_size);
        *entry_items = ORC_RAW_BIT;
        *entry_data = (uint32_t)chunk_size;
        blk = (uint32_t)chunk_size;
    } else {
        for (uint32_t k = 0; k < fbytes / 4u; ++k) put_u32(block_out + 4u * k, flags[k]);
        memcpy(block_out + fbytes, data, dbytes);
        memset(block_out + fbytes + dbytes, 0, padded - dbytes);
        *entry_items = items;
        *entry_data = dbytes;
    }
    free(w);
    free(len);
    free(off);
    free(flags);
    free(data);
    return blk;
}

/* ------------------------------------------------------------------------ */
/* Whole stream.                                                            */
/* ------------------------------------------------------------------------ */
int64_t orc_compress(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                     int match_level, uint8_t* out, uint64_t capacity) {
    return orc_compress_w(in, n_bytes, word_size, chunk_size, match_level, ORC_NEAR_WINDOW, out,
                          capacity);
}

int64_t orc_compress_w(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                       int match_level, int window, uint8_t* out, uint64_t capacity) {
    if (!orc_valid_geometry(word_size, chunk_size)) return ORC_ERR_INVALID_ARG;
    if (match_level != 0 && match_level != 1) return ORC_ERR_INVALID_ARG;
    if (window < 1 || window > ORC_MAX_WINDOW) return ORC_ERR_INVALID_ARG;
    if (n_bytes > 0 && in == NULL) return ORC_ERR_INVALID_ARG;
    uint64_t chunks = (n_bytes + (uint64_t)chunk_size - 1) / (uint64_t)chunk_size;
    if (chunks > 0xFFFFFFFFull) return ORC_ERR_INVALID_ARG;
    uint64_t bound = orc_compress_bound(n_bytes, word_size, chunk_size);
    if (capacity < bound) return ORC_ERR_CAPACITY; /* the oracle always writes whole streams */

    uint8_t* chunk = (uint8_t*)malloc((size_t)chunk_size);
    uint64_t table_at = ORC_HEADER_BYTES;
    uint64_t pos = ORC_HEADER_BYTES + ORC_ENTRY_BYTES * chunks;
    for (uint64_t c = 0; c < chunks; ++c) {
        uint64_t begin = c * (uint64_t)chunk_size;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)chunk_size) take = (uint64_t)chunk_size;
        memset(chunk, 0, (size_t)chunk_size);
        memcpy(chunk, in + begin, (size_t)take);
        uint32_t items = 0, dbytes = 0;
        uint32_t blk = orc_encode_chunk_w(chunk, word_size, chunk_size, match_level, window,
                                          out + pos, &items, &dbytes);
        put_u32(out + table_at + ORC_ENTRY_BYTES * c, items);
        put_u32(out + table_at + ORC_ENTRY_BYTES * c + 4, dbytes);
        pos += blk;
    }
    free(chunk);

    put_u32(out + 0, ORC_MAGIC);
    put_u16(out + 4, ORC_VERSION);
    out[6] = (uint8_t)word_size;
    out[7] = 0;
    put_u32(out + 8, (uint32_t)chunk_size);
    put_u32(out + 12, (uint32_t)chunks);
    put_u64(out + 16, n_bytes);
    put_u64(out + 24, pos);
    return (int64_t)pos;
}

int orc_parse_header(const uint8_t* in, uint64_t in_len, int* word_size, int* chunk_size,
                     uint64_t* n_chunks, uint64_t* orig_bytes, uint64_t* stream_bytes) {
    if (in_len < ORC_HEADER_BYTES) return ORC_ERR_CORRUPT;
    if (get_u32(in) != ORC_MAGIC || get_u16(in + 4) != ORC_VERSION || in[7] != 0)
        return ORC_ERR_CORRUPT;
    int ws = in[6];
    int cs = (int)get_u32(in + 8);
    if (!orc_valid_geometry(ws, cs)) return ORC_ERR_CORRUPT;
    uint64_t chunks = get_u32(in + 12);
    uint64_t orig = get_u64(in + 16);
    uint64_t total = get_u64(in + 24);
    if (chunks != (orig + (uint64_t)cs - 1) / (uint64_t)cs) return ORC_ERR_CORRUPT;
    if (total < ORC_HEADER_BYTES + ORC_ENTRY_BYTES * chunks) return ORC_ERR_CORRUPT;
    *word_size = ws;
    *chunk_size = cs;
    *n_chunks = chunks;
    *orig_bytes = orig;
    *stream_bytes = total;
    return 0;
}

/* Decode one normal chunk by sequential replay of its items: a literal
 * appends a word, a match copies `length` elements from `offset` elements
 * back, one element at a time so that overlapping copies repeat. */
static int decode_items(const uint8_t* block, uint32_t items, uint32_t dbytes, int word_size,
                        int chunk_size, uint8_t* chunk_out) {
    int elems = chunk_size / word_size;
    uint32_t fbytes = 4u * ((items + 31u) / 32u);
    const uint8_t* data = block + fbytes;
    uint32_t b = 0;
    int q = 0;
    for (uint32_t j = 0; j < items; ++j) {
        uint32_t fw = get_u32(block + 4u * (j / 32u));
        int is_match = (int)((fw >> (j % 32u)) & 1u);
        if (is_match) {
            if (b + 2u > dbytes) return ORC_ERR_CORRUPT;
            int L = data[b], O = data[b + 1];
            b += 2;
            if (L < 1 || O < 1 || O > q || q + L > elems) return ORC_ERR_CORRUPT;
            for (int k = 0; k < L; ++k) {
                memcpy(chunk_out + (size_t)(q + k) * word_size,
                       chunk_out + (size_t)(q + k - O) * word_size, (size_t)word_size);
            }
            q += L;
        } else {
            if (b + (uint32_t)word_size > dbytes) return ORC_ERR_CORRUPT;
            if (q + 1 > elems) return ORC_ERR_CORRUPT;
            memcpy(chunk_out + (size_t)q * word_size, data + b, (size_t)word_size);
            b += (uint32_t)word_size;
            q += 1;
        }
    }
    if (q != elems || b != dbytes) return ORC_ERR_CORRUPT;
    return 0;
}

int orc_decompress(const uint8_t* in, uint64_t in_len, uint8_t* out, uint64_t n_bytes) {
    int ws = 0, cs = 0;
    uint64_t chunks = 0, orig = 0, total = 0;
    int rc = orc_parse_header(in, in_len, &ws, &cs, &chunks, &orig, &total);
    if (rc != 0) return rc;
    if (orig != n_bytes) return ORC_ERR_CORRUPT;
    if (total > in_len) return ORC_ERR_CORRUPT;
    int elems = cs / ws;
    uint8_t* chunk = (uint8_t*)malloc((size_t)cs);
    uint64_t pos = ORC_HEADER_BYTES + ORC_ENTRY_BYTES * chunks;
    rc = 0;
    for (uint64_t c = 0; c < chunks && rc == 0; ++c) {
        const uint8_t* e = in + ORC_HEADER_BYTES + ORC_ENTRY_BYTES * c;
        uint32_t items = get_u32(e), dbytes = get_u32(e + 4);
        uint64_t blk;
        if (items == 0 && dbytes == 0) {
            memset(chunk, 0, (size_t)cs);
            blk = 0;
        } else if (items == ORC_RAW_BIT) {
            if (dbytes != (uint32_t)cs || pos + (uint64_t)cs > total) {
                rc = ORC_ERR_CORRUPT;
                break;
            }
            memcpy(chunk, in + pos, (size_t)cs);
            blk = (uint64_t)cs;
        } else {
            if (items & ORC_RAW_BIT || items > (uint32_t)elems || items == 0) {
                rc = ORC_ERR_CORRUPT;
                break;
            }
            blk = 4u * ((items + 31u) / 32u) + ((dbytes + 3u) & ~3u);
            if (dbytes > (uint32_t)cs || pos + blk > total) {
                rc = ORC_ERR_CORRUPT;
                break;
            }
            rc = decode_items(in + pos, items, dbytes, ws, cs, chunk);
            if (rc != 0) break;
        }
        uint64_t begin = c * (uint64_t)cs;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)cs) take = (uint64_t)cs;
        memcpy(out + begin, chunk, (size_t)take);
        pos += blk;
    }
    if (rc == 0 && pos != total) rc = ORC_ERR_CORRUPT;
    free(chunk);
    return rc;
}

/* Chunk-range entry used to spread the oracle over host threads: encodes
 * chunks [c0, c1) of `in` into per-chunk blocks at out_blocks + c*chunk_size
 * with sizes in block_bytes[c] and the size-table words in entries[2c..2c+1].
 * The caller concatenates in chunk order, which is byte-identical to
 * orc_compress. */
void orc_encode_chunk_range(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                            int match_level, uint64_t c0, uint64_t c1, uint8_t* out_blocks,
                            uint32_t* block_bytes, uint32_t* entries) {
    orc_encode_chunk_range_w(in, n_bytes, word_size, chunk_size, match_level, ORC_NEAR_WINDOW,
                             c0, c1, out_blocks, block_bytes, entries);
}

void orc_encode_chunk_range_w(const uint8_t* in, uint64_t n_bytes, int word_size,
                              int chunk_size, int match_level, int window, uint64_t c0,
                              uint64_t c1, uint8_t* out_blocks, uint32_t* block_bytes,
                              uint32_t* entries) {
    uint8_t* chunk = (uint8_t*)malloc((size_t)chunk_size);
    for (uint64_t c = c0; c < c1; ++c) {
        uint64_t begin = c * (uint64_t)chunk_size;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)chunk_size) take = (uint64_t)chunk_size;
        memset(chunk, 0, (size_t)chunk_size);
        memcpy(chunk, in + begin, (size_t)take);
        block_bytes[c] = orc_encode_chunk_w(chunk, word_size, chunk_size, match_level, window,
                                            out_blocks + c * (uint64_t)chunk_size,
                                            &entries[2 * c], &entries[2 * c + 1]);
    }
    free(chunk);
}

/* Chunk-range decode used to spread the oracle decoder over host threads:
 * decodes chunks [c0, c1) of a stream whose per-chunk block offsets (from the
 * start of the stream) are given in block_off[c]. Returns 0 or ORC_ERR_*. */
int orc_decode_chunk_range(const uint8_t* in, uint64_t in_len, const uint64_t* block_off,
                           uint8_t* out, uint64_t n_bytes, uint64_t c0, uint64_t c1) {
    int ws = 0, cs = 0;
    uint64_t chunks = 0, orig = 0, total = 0;
    int rc = orc_parse_header(in, in_len, &ws, &cs, &chunks, &orig, &total);
    if (rc != 0) return rc;
    if (orig != n_bytes || total > in_len || c1 > chunks) return ORC_ERR_CORRUPT;
    int elems = cs / ws;
    uint8_t* chunk = (uint8_t*)malloc((size_t)cs);
    for (uint64_t c = c0; c < c1 && rc == 0; ++c) {
        const uint8_t* e = in + ORC_HEADER_BYTES + ORC_ENTRY_BYTES * c;
        uint32_t items = get_u32(e), dbytes = get_u32(e + 4);
        uint64_t pos = block_off[c];
        if (items == 0 && dbytes == 0) {
            memset(chunk, 0, (size_t)cs);
        } else if (items == ORC_RAW_BIT) {
            if (dbytes != (uint32_t)cs || pos + (uint64_t)cs > total) rc = ORC_ERR_CORRUPT;
            else memcpy(chunk, in + pos, (size_t)cs);
        } else if ((items & ORC_RAW_BIT) || items > (uint32_t)elems || dbytes > (uint32_t)cs) {
            rc = ORC_ERR_CORRUPT;
        } else {
            uint64_t blk = 4u * ((items + 31u) / 32u) + ((dbytes + 3u) & ~3u);
            if (pos + blk > total) rc = ORC_ERR_CORRUPT;
            else rc = decode_items(in + pos, items, dbytes, ws, cs, chunk);
        }
        if (rc != 0) break;
        uint64_t begin = c * (uint64_t)cs;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)cs) take = (uint64_t)cs;
        memcpy(out + begin, chunk, (size_t)take);
    }
    free(chunk);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Split mode: the same items, laid out as four ports.                      */
/* ------------------------------------------------------------------------ */
/* Stage page, split-mode section (and CN-GPULZ-1): instead of one interleaved
 * stream the coder emits four ports -- literals (literal words back to back;
 * a raw-fallback chunk lands here whole), lengths (one byte per match token),
 * offsets (one byte per match token) and meta (stream header, per-chunk size
 * table and the flag bitmaps). The pages fix the ports' contents, not their
 * byte layout; the oracle takes this one (the repository's format notes):
 *
 *   meta: 48-byte header {u32 magic, u16 version 2, u8 word_size, u8 0,
 *         u32 chunk_size, u32 n_chunks, u64 orig_bytes, u64 meta_bytes,
 *         u64 literal_bytes, u64 n_matches}, then n_chunks entries
 *         {u32 n_items | RAW << 31, u32 n_matches} ({0,0} zero chunk,
 *         {RAW,0} raw chunk), then every coded chunk's flag words
 *         (ceil(n_items/32) u32, LSB first, 1 = match) in chunk order;
 *   literals, lengths, offsets: chunk order, back to back, no padding.
 *
 * The items are exactly those of the single-stream form (same parse, same
 * raw decision): split mode only moves bytes. */
#define ORC_SPLIT_VERSION 2u
#define ORC_SPLIT_HEADER_BYTES 48u

void orc_split_bounds(uint64_t n_bytes, int word_size, int chunk_size, uint64_t bounds[4]) {
    uint64_t chunks = (n_bytes + (uint64_t)chunk_size - 1) / (uint64_t)chunk_size;
    uint64_t elems = (uint64_t)(chunk_size / word_size);
    bounds[0] = ORC_SPLIT_HEADER_BYTES + ORC_ENTRY_BYTES * chunks + 4u * chunks * ((elems + 31u) / 32u);
    bounds[1] = chunks * (uint64_t)chunk_size;
    bounds[2] = chunks * elems;
    bounds[3] = chunks * elems;
}

int orc_compress_split(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                       int match_level, uint8_t* meta, uint8_t* lits, uint8_t* lens,
                       uint8_t* offs, uint64_t sizes[4]) {
    if (!orc_valid_geometry(word_size, chunk_size)) return ORC_ERR_INVALID_ARG;
    if (match_level != 0 && match_level != 1) return ORC_ERR_INVALID_ARG;
    if (n_bytes > 0 && in == NULL) return ORC_ERR_INVALID_ARG;
    uint64_t chunks = (n_bytes + (uint64_t)chunk_size - 1) / (uint64_t)chunk_size;
    if (chunks > 0xFFFFFFFFull) return ORC_ERR_INVALID_ARG;
    uint8_t* chunk = (uint8_t*)malloc((size_t)chunk_size);
    uint8_t* block = (uint8_t*)malloc((size_t)chunk_size);
    uint64_t flag_at = ORC_SPLIT_HEADER_BYTES + ORC_ENTRY_BYTES * chunks;
    uint64_t nl = 0, nm = 0;
    for (uint64_t c = 0; c < chunks; ++c) {
        uint64_t begin = c * (uint64_t)chunk_size;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)chunk_size) take = (uint64_t)chunk_size;
        memset(chunk, 0, (size_t)chunk_size);
        memcpy(chunk, in + begin, (size_t)take);
        uint32_t items = 0, dbytes = 0;
        orc_encode_chunk(chunk, word_size, chunk_size, match_level, block, &items, &dbytes);
        uint8_t* e = meta + ORC_SPLIT_HEADER_BYTES + ORC_ENTRY_BYTES * c;
        if (items == ORC_RAW_BIT) {
            memcpy(lits + nl, block, (size_t)chunk_size);
            nl += (uint64_t)chunk_size;
            put_u32(e, ORC_RAW_BIT);
            put_u32(e + 4, 0);
            continue;
        }
        uint32_t fwords = (items + 31u) / 32u;
        memcpy(meta + flag_at, block, 4u * (size_t)fwords);
        flag_at += 4u * (uint64_t)fwords;
        const uint8_t* data = block + 4u * fwords;
        uint32_t b = 0, m = 0;
        for (uint32_t j = 0; j < items; ++j) {
            if ((get_u32(block + 4u * (j / 32u)) >> (j % 32u)) & 1u) {
                lens[nm + m] = data[b];
                offs[nm + m] = data[b + 1];
                b += 2;
                ++m;
            } else {
                memcpy(lits + nl, data + b, (size_t)word_size);
                nl += (uint64_t)word_size;
                b += (uint32_t)word_size;
            }
        }
        nm += m;
        put_u32(e, items);
        put_u32(e + 4, m);
    }
    free(chunk);
    free(block);
    put_u32(meta + 0, ORC_MAGIC);
    put_u16(meta + 4, ORC_SPLIT_VERSION);
    meta[6] = (uint8_t)word_size;
    meta[7] = 0;
    put_u32(meta + 8, (uint32_t)chunk_size);
    put_u32(meta + 12, (uint32_t)chunks);
    put_u64(meta + 16, n_bytes);
    put_u64(meta + 24, flag_at);
    put_u64(meta + 32, nl);
    put_u64(meta + 40, nm);
    sizes[0] = flag_at;
    sizes[1] = nl;
    sizes[2] = nm;
    sizes[3] = nm;
    return 0;
}

/* Sequential replay out of the four ports. port_len[k] are the bytes
 * available in each port. Returns 0, or a negative ORC_ERR_* code. */
int orc_decompress_split(const uint8_t* meta, const uint8_t* lits, const uint8_t* lens,
                         const uint8_t* offs, const uint64_t port_len[4], uint8_t* out,
                         uint64_t n_bytes) {
    if (port_len[0] < ORC_SPLIT_HEADER_BYTES) return ORC_ERR_CORRUPT;
    if (get_u32(meta) != ORC_MAGIC || get_u16(meta + 4) != ORC_SPLIT_VERSION || meta[7] != 0)
        return ORC_ERR_CORRUPT;
    int ws = meta[6];
    int cs = (int)get_u32(meta + 8);
    if (!orc_valid_geometry(ws, cs)) return ORC_ERR_CORRUPT;
    uint64_t chunks = get_u32(meta + 12), orig = get_u64(meta + 16);
    uint64_t meta_bytes = get_u64(meta + 24), nlit = get_u64(meta + 32), nmat = get_u64(meta + 40);
    if (orig != n_bytes || chunks != (orig + (uint64_t)cs - 1) / (uint64_t)cs) return ORC_ERR_CORRUPT;
    uint64_t flag_at = ORC_SPLIT_HEADER_BYTES + ORC_ENTRY_BYTES * chunks;
    if (meta_bytes < flag_at || meta_bytes > port_len[0] || nlit > port_len[1] ||
        nmat > port_len[2] || nmat > port_len[3])
        return ORC_ERR_CORRUPT;
    int elems = cs / ws;
    uint8_t* chunk = (uint8_t*)malloc((size_t)cs);
    uint64_t li = 0, mi = 0;
    int rc = 0;
    for (uint64_t c = 0; c < chunks && rc == 0; ++c) {
        const uint8_t* e = meta + ORC_SPLIT_HEADER_BYTES + ORC_ENTRY_BYTES * c;
        uint32_t items = get_u32(e), m = get_u32(e + 4);
        if (items == 0 && m == 0) {
            memset(chunk, 0, (size_t)cs);
        } else if (items == ORC_RAW_BIT && m == 0) {
            if (li + (uint64_t)cs > nlit) {
                rc = ORC_ERR_CORRUPT;
                break;
            }
            memcpy(chunk, lits + li, (size_t)cs);
            li += (uint64_t)cs;
        } else if ((items & ORC_RAW_BIT) || items == 0 || items > (uint32_t)elems) {
            rc = ORC_ERR_CORRUPT;
            break;
        } else {
            uint32_t fwords = (items + 31u) / 32u;
            if (flag_at + 4u * (uint64_t)fwords > meta_bytes) {
                rc = ORC_ERR_CORRUPT;
                break;
            }
            const uint8_t* fl = meta + flag_at;
            flag_at += 4u * (uint64_t)fwords;
            int q = 0;
            uint32_t seen = 0;
            for (uint32_t j = 0; j < items && rc == 0; ++j) {
                if ((get_u32(fl + 4u * (j / 32u)) >> (j % 32u)) & 1u) {
                    if (mi >= nmat || seen >= m) {
                        rc = ORC_ERR_CORRUPT;
                        break;
                    }
                    int L = lens[mi], O = offs[mi];
                    ++mi;
                    ++seen;
                    if (L < 1 || O < 1 || O > q || q + L > elems) {
                        rc = ORC_ERR_CORRUPT;
                        break;
                    }
                    for (int k = 0; k < L; ++k)
                        memcpy(chunk + (size_t)(q + k) * ws, chunk + (size_t)(q + k - O) * ws, (size_t)ws);
                    q += L;
                } else {
                    if (li + (uint64_t)ws > nlit || q + 1 > elems) {
                        rc = ORC_ERR_CORRUPT;
                        break;
                    }
                    memcpy(chunk + (size_t)q * ws, lits + li, (size_t)ws);
                    li += (uint64_t)ws;
                    q += 1;
                }
            }
            if (rc == 0 && (q != elems || seen != m)) rc = ORC_ERR_CORRUPT;
        }
        if (rc != 0) break;
        uint64_t begin = c * (uint64_t)cs;
        uint64_t take = n_bytes - begin;
        if (take > (uint64_t)cs) take = (uint64_t)cs;
        memcpy(out + begin, chunk, (size_t)take);
    }
    if (rc == 0 && (li != nlit || mi != nmat || flag_at != meta_bytes)) rc = ORC_ERR_CORRUPT;
    free(chunk);
    return rc;
}
