/*
 * GPULZ oracle (test infrastructure only): plain sequential CPU encoder and
 * decoder of the GPULZ chunked LZSS stream. See gpulz_oracle.c for the
 * passages each step follows. Not included by, and not linked into, the
 * CUDA library.
 */
#ifndef GPULZ_ORACLE_H
#define GPULZ_ORACLE_H

#include <stdint.h>

#define ORC_ERR_INVALID_ARG (-1)
#define ORC_ERR_CAPACITY (-2)
#define ORC_ERR_CORRUPT (-3)

#ifdef __cplusplus
extern "C" {
#endif

int orc_valid_geometry(int word_size, int chunk_size);
int orc_min_match_len(int word_size);
uint32_t orc_hash_bits(int elems);
uint32_t orc_hash(uint32_t k0, uint32_t k1, uint32_t bits);
uint64_t orc_compress_bound(uint64_t n_bytes, int word_size, int chunk_size);

/* Per-position longest match of one chunk of `elems` words (zero-extended to
 * 32 bits). len = 0 means no candidate; off is in elements. */
void orc_near_matches(const uint32_t* w, int elems, uint8_t* len_out, uint8_t* off_out);
/* Same with a near window of `window` elements (1..64); the default is 32.
 * The window-width study of the match-search section compares 32, 48, 64. */
void orc_near_matches_w(const uint32_t* w, int elems, int window, uint8_t* len_out,
                        uint8_t* off_out);
void orc_level1_matches(const uint32_t* w, int elems, uint8_t* len_io, uint8_t* off_io);

uint32_t orc_encode_chunk(const uint8_t* chunk, int word_size, int chunk_size, int match_level,
                          uint8_t* block_out, uint32_t* entry_items, uint32_t* entry_data);
uint32_t orc_encode_chunk_w(const uint8_t* chunk, int word_size, int chunk_size, int match_level,
                            int window, uint8_t* block_out, uint32_t* entry_items,
                            uint32_t* entry_data);

/* Returns the stream length, or a negative ORC_ERR_* code. `capacity` must be
 * at least orc_compress_bound(). */
int64_t orc_compress(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                     int match_level, uint8_t* out, uint64_t capacity);
int64_t orc_compress_w(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                       int match_level, int window, uint8_t* out, uint64_t capacity);
int orc_parse_header(const uint8_t* in, uint64_t in_len, int* word_size, int* chunk_size,
                     uint64_t* n_chunks, uint64_t* orig_bytes, uint64_t* stream_bytes);
/* Returns 0, or a negative ORC_ERR_* code. */
int orc_decompress(const uint8_t* in, uint64_t in_len, uint8_t* out, uint64_t n_bytes);

void orc_encode_chunk_range(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                            int match_level, uint64_t c0, uint64_t c1, uint8_t* out_blocks,
                            uint32_t* block_bytes, uint32_t* entries);
void orc_encode_chunk_range_w(const uint8_t* in, uint64_t n_bytes, int word_size,
                              int chunk_size, int match_level, int window, uint64_t c0,
                              uint64_t c1, uint8_t* out_blocks, uint32_t* block_bytes,
                              uint32_t* entries);

int orc_decode_chunk_range(const uint8_t* in, uint64_t in_len, const uint64_t* block_off,
                           uint8_t* out, uint64_t n_bytes, uint64_t c0, uint64_t c1);

/* Split mode: four ports (meta, literals, lengths, offsets) holding the same
 * items. bounds[k] is an upper bound on port k's bytes; sizes[k] receives
 * each port's length. */
void orc_split_bounds(uint64_t n_bytes, int word_size, int chunk_size, uint64_t bounds[4]);
int orc_compress_split(const uint8_t* in, uint64_t n_bytes, int word_size, int chunk_size,
                       int match_level, uint8_t* meta, uint8_t* lits, uint8_t* lens,
                       uint8_t* offs, uint64_t sizes[4]);
int orc_decompress_split(const uint8_t* meta, const uint8_t* lits, const uint8_t* lens,
                         const uint8_t* offs, const uint64_t port_len[4], uint8_t* out,
                         uint64_t n_bytes);

#ifdef __cplusplus
}
#endif
#endif
