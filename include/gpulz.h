/*
 * gpulz.h -- C ABI of the GB300 (sm_103a) GPULZ chunked LZSS coder.
 *
 * The coder is the one described by the FZGPUModules GPULZ stage
 * documentation ("fz::GPULZStage", stage_gpulz page) and its codebase note
 * CN-GPULZ-1: the input is split into fixed chunk_size-byte chunks of
 * word_size-byte elements; each chunk is coded on its own into literal words
 * and 2-byte [length, offset] match tokens plus a literal/match flag bitmap
 * (class summary); level 0 searches the 32-element near window exactly with
 * ANDed equality masks, level 1 adds hashed two-word-key candidates with
 * offsets up to 255 over 8 sub-blocks (match-search section); a chunk whose
 * coded form is not smaller is stored raw (raw-fallback paragraph); an all-zero
 * chunk costs only its size-table entry (zero-chunk paragraph); decode is
 * block-parallel (scan of item sizes, pointer jumping over back-references).
 *
 * Stream format v1 (little-endian, every padding byte zero):
 *   header, 32 bytes : u32 magic 0x5A4C5047 ("GPLZ"), u16 version = 1,
 *                      u8 word_size, u8 reserved = 0, u32 chunk_size,
 *                      u32 n_chunks, u64 orig_bytes, u64 stream_bytes
 *   size table       : n_chunks x { u32 n_items | RAW << 31, u32 data_bytes }
 *                      zero chunk = {0, 0}; raw chunk = {RAW, chunk_size}
 *   blocks, in chunk order, each a multiple of 4 bytes:
 *     normal : u32 flags[ceil(n_items/32)] (bit j of word j/32, 1 = match),
 *              then the items (literal = word_size bytes as in the input,
 *              match = u8 length, u8 offset, both in elements), zero padded
 *     raw    : chunk_size bytes of the zero-padded chunk
 *     zero   : nothing
 * The match level is not recorded: streams from either level decode alike.
 *
 * Supported geometry: word_size in {1, 2, 4}, chunk_size in {1024, 2048,
 * 4096} (elements per chunk = chunk_size / word_size, a power of two >= 256).
 *
 * Memory: every d_* pointer is device memory owned by the caller. The library
 * owns one scratch area per (device, stream): a status word, ticket counters,
 * 12 bytes per chunk (block sizes and offsets) and, for gpulz_compress, one
 * chunk_size slot per chunk in which each chunk's block is staged before it
 * is placed (so about n_bytes of scratch for an n_bytes input). The first
 * call on a stream, or a call needing more room than any earlier call on it,
 * allocates that scratch stream-ordered (cudaMallocAsync); later calls
 * allocate nothing. The scratch lives until gpulz_release_scratch(stream) is
 * called (or the process exits): a caller that makes short-lived streams
 * releases each one's scratch before destroying the stream.
 * gpulz_compress_noalloc never allocates.
 *
 * Errors: argument errors a host can check are returned synchronously and
 * nothing is launched. Conditions found on the device (corrupt stream, size
 * mismatch, output capacity exceeded, look-back wait timeout) are recorded in
 * the stream's device status word, read and cleared by gpulz_device_status().
 * The kernels never trap.
 */
#ifndef GPULZ_H
#define GPULZ_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gpulz_status {
    GPULZ_OK = 0,
    GPULZ_ERR_INVALID_ARG = 1,   /* bad pointer / geometry / level; nothing launched */
    GPULZ_ERR_CAPACITY = 2,      /* compressed stream did not fit in `capacity` */
    GPULZ_ERR_CORRUPT = 3,       /* stream fails validation while decoding */
    GPULZ_ERR_TIMEOUT = 4,       /* a bounded device-side wait gave up */
    GPULZ_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    GPULZ_ERR_SIZE_MISMATCH = 6  /* n_bytes differs from the stream's original size */
} gpulz_status;

/*
 * gpulz_compress -- encode n_bytes at d_in into one GPULZ stream at d_out.
 * (GPULZ stage page: class summary, match-search section, raw-fallback and
 * zero-chunk paragraphs; graph-capture paragraph for the deferred size.)
 *
 *   d_in        device, n_bytes bytes, any alignment (16-byte alignment takes
 *               the vector-load path). May be NULL only if n_bytes == 0.
 *   word_size   1, 2 or 4: element width in bytes.
 *   chunk_size  1024, 2048 or 4096: bytes per independently coded chunk. The
 *               last chunk is zero padded (the padding is coded like data).
 *   match_level 0 = exact near window only; 1 = plus hashed candidates.
 *   d_out       device buffer of `capacity` bytes. Nothing is written at or
 *               past d_out + capacity. capacity >= gpulz_compress_bound()
 *               always suffices.
 *   d_out_bytes device pointer to one size_t that receives the stream length
 *               (the length needed, if it exceeds capacity; then the device
 *               status also records GPULZ_ERR_CAPACITY).
 *   stream      CUDA stream; the call only enqueues work on it.
 * Returns GPULZ_OK once the work is enqueued.
 */
gpulz_status gpulz_compress(const void* d_in, size_t n_bytes, int word_size, int chunk_size,
                            int match_level, void* d_out, size_t capacity, size_t* d_out_bytes,
                            cudaStream_t stream);

/*
 * gpulz_compress_window -- gpulz_compress with a wider exact near window.
 * (GPULZ stage page, match-search section: the window-width measurement,
 * ratio at 32, 48 and 64 elements.)
 *
 *   window      32..64: the level-0 search finds the longest run over offsets
 *               1..window (nearest offset on ties), lengths capped at 255 and
 *               at the chunk end. 32 is gpulz_compress exactly. Above 32,
 *               match_level must be 0. Offsets still fit the token's byte, so
 *               the stream format and gpulz_decompress are unchanged.
 *   Other arguments, ownership and errors as gpulz_compress; a window outside
 *   32..64, or above 32 with match_level 1, returns GPULZ_ERR_INVALID_ARG and
 *   launches nothing. A wider window costs a second mask-and-chain pass per
 *   chunk (about twice the match-search work).
 */
gpulz_status gpulz_compress_window(const void* d_in, size_t n_bytes, int word_size,
                                   int chunk_size, int match_level, int window, void* d_out,
                                   size_t capacity, size_t* d_out_bytes, cudaStream_t stream);

/*
 * gpulz_decompress -- decode the GPULZ stream at d_in into n_bytes at d_out.
 * (GPULZ stage page: decode paragraph -- one scan recovers every item's
 * offset, each element points back to q - offset, pointer jumping for
 * log2(elements) rounds; zero-chunk and raw-fallback paragraphs.)
 *
 *   d_in    device, the whole stream. The header's stream_bytes bytes must be
 *           readable; use gpulz_decompress_bounded() when the buffer length
 *           is known and the stream is untrusted.
 *   d_out   device, n_bytes bytes, written only in [d_out, d_out + n_bytes).
 *   n_bytes the original length; a header that disagrees records
 *           GPULZ_ERR_SIZE_MISMATCH and nothing is written.
 * The header is parsed on the device: the call does not synchronise with the
 * host, and it can be captured into a CUDA graph.
 *
 * CUDA graphs (this call, gpulz_decompress_bounded, gpulz_compress,
 * gpulz_compress_window and the split calls): a call made while its stream
 * is being captured records, around its kernels, the reset of the ticket
 * counters and look-back descriptors it uses, so the graph can be launched
 * any number of times, with new input contents each time (sizes and
 * pointers are those captured). Capture allocates nothing: the stream needs
 * its scratch from an earlier direct call of at least the same size on it,
 * else the call returns GPULZ_ERR_INVALID_ARG during capture.
 */
gpulz_status gpulz_decompress(const void* d_in, void* d_out, size_t n_bytes, cudaStream_t stream);

/* As gpulz_decompress, but no byte at or past d_in + in_bytes is read: a
 * header or size table that points further records GPULZ_ERR_CORRUPT. */
gpulz_status gpulz_decompress_bounded(const void* d_in, size_t in_bytes, void* d_out,
                                      size_t n_bytes, cudaStream_t stream);

/* Worst-case stream length: 32 + n_chunks * (8 + chunk_size) (every chunk
 * raw). Host only; returns 0 for an unsupported geometry. */
size_t gpulz_compress_bound(size_t n_bytes, int word_size, int chunk_size);

/* Parse a stream header copied to host memory (h_len >= 32). Host only. Any
 * output pointer may be NULL. */
gpulz_status gpulz_stream_info(const void* h_header, size_t h_len, size_t* orig_bytes,
                               size_t* stream_bytes, int* word_size, int* chunk_size);

/* Synchronise `stream`, return the first error recorded by the device since
 * the last call (GPULZ_OK if none) and clear it. */
gpulz_status gpulz_device_status(cudaStream_t stream);

/*
 * gpulz_release_scratch -- give back the scratch the library holds for
 * `stream` on the current device (no counterpart in the paper: the lifetime
 * of this library's own scratch).
 *
 * The memory is freed stream-ordered (cudaFreeAsync on `stream`), so work
 * already enqueued on the stream finishes first; the stream must still be
 * valid. A status the device recorded on this stream and not yet read by
 * gpulz_device_status() is dropped with it. The next call on the stream
 * allocates afresh. Returns GPULZ_OK if the stream holds no scratch, and
 * GPULZ_ERR_INVALID_ARG (nothing freed) while the stream is being captured.
 */
gpulz_status gpulz_release_scratch(cudaStream_t stream);

/*
 * gpulz_compress_noalloc -- gpulz_compress for callers that cannot allocate.
 * (No counterpart in the paper: the GPULZ pages have no such entry point.)
 *
 * Some callers cannot let a library call cudaMalloc: code running while a
 * framework's caching allocator already holds the device memory, code on a
 * latency-critical path that cannot take cudaMalloc's implicit device-wide
 * synchronisation, and plug-ins whose host forbids allocations it does not
 * make. This entry point never allocates and calls no allocating routine. Its
 * scratch (look-back descriptors, ticket counter, status word) is one fixed
 * device array of about 512 KiB inside the library, which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments, output and stream format are exactly those of gpulz_compress.
 * Limit: at most 65536 chunks per call (256 MiB of input at chunk_size 4096,
 * 128 MiB at 2048, 64 MiB at 1024); larger inputs return
 * GPULZ_ERR_INVALID_ARG and launch nothing.
 * Set-up: the first call on a device looks up the array's device address,
 * with that device current.
 * Sharing: all calls on a device share the one array, which keeps the last
 * call's contents; each call first clears, on its stream, the part it uses
 * (status word, ticket, one look-back entry per chunk). Calls that overlap on
 * the GPU (other streams, other host threads) race and must not be issued.
 * A device-side wait that gives up sets *d_out_bytes to SIZE_MAX; capacity
 * overflow shows as *d_out_bytes > capacity. gpulz_device_status() does not
 * see this path.
 */
gpulz_status gpulz_compress_noalloc(const void* d_in, size_t n_bytes, int word_size,
                                    int chunk_size, int match_level, void* d_out,
                                    size_t capacity, size_t* d_out_bytes, cudaStream_t stream);

/*
 * Split mode (stage page, split-mode section; codebase note CN-GPULZ-1):
 * the same items as gpulz_compress, emitted as four ports instead of one
 * interleaved stream, so that a downstream entropy coder sees each kind of
 * symbol on its own:
 *   meta     -- 48-byte header {u32 magic "GPLZ", u16 version 2, u8 word_size,
 *               u8 0, u32 chunk_size, u32 n_chunks, u64 orig_bytes,
 *               u64 meta_bytes, u64 literal_bytes, u64 n_matches}, then
 *               n_chunks entries {u32 n_items | RAW << 31, u32 n_matches}
 *               ({0,0} zero chunk, {RAW,0} raw chunk), then every coded
 *               chunk's flag words (ceil(n_items/32) u32, 1 = match, LSB
 *               first), in chunk order;
 *   literals -- every literal word (word_size bytes, as in the input) in
 *               item order, chunk after chunk; a raw chunk's chunk_size
 *               bytes (zero padded) land here whole;
 *   lengths  -- one byte per match token, item order, chunk after chunk;
 *   offsets  -- one byte per match token, likewise.
 * Ports are back to back, without padding. The pages fix the ports' contents,
 * not this byte layout, which is this library's.
 */

/* Upper bounds on the four ports' bytes, in the order meta, literals,
 * lengths, offsets. */
gpulz_status gpulz_split_bounds(size_t n_bytes, int word_size, int chunk_size, size_t bounds[4]);

/* Split-mode encode. d_meta must be 4-byte aligned; the other ports have no
 * alignment rule. capacity[4] (host) bounds each port in the same order;
 * nothing is written at or past a port's capacity. The four port lengths are
 * written on the device to d_port_bytes[0..3] (8-byte aligned); a port that
 * did not fit is recorded as GPULZ_ERR_CAPACITY for gpulz_device_status().
 * Other arguments and errors as gpulz_compress. */
gpulz_status gpulz_compress_split(const void* d_in, size_t n_bytes, int word_size, int chunk_size,
                                  int match_level, void* d_meta, void* d_literals,
                                  void* d_lengths, void* d_offsets, const size_t capacity[4],
                                  size_t* d_port_bytes, cudaStream_t stream);

/* Split-mode decode straight out of the four ports (no rebuilt single
 * stream): port_bytes[4] (host) gives each port's available bytes in the
 * order meta, literals, lengths, offsets; d_meta must be 4-byte aligned; an
 * empty port may be null. Output, n_bytes and errors as
 * gpulz_decompress_bounded. */
gpulz_status gpulz_decompress_split(const void* d_meta, const void* d_literals,
                                    const void* d_lengths, const void* d_offsets,
                                    const size_t port_bytes[4], void* d_out, size_t n_bytes,
                                    cudaStream_t stream);

/*
 * gpulz_set_kernel_events -- measurement hook (no counterpart in the paper).
 *
 * gpulz_compress runs three kernels (encode, tile scan of block sizes, copy to
 * the stream) and gpulz_decompress two (offset scan, decode). To time the
 * main one alone, pass two CUDA events (created by the caller, which keeps
 * ownership): while they are set, every following gpulz_compress and
 * gpulz_decompress issued from this host thread records `start` on its stream
 * right before its encode or decode kernel and `stop` right after it. Passing
 * two nulls clears the hook. Returns GPULZ_ERR_INVALID_ARG if exactly one of
 * the two is null. The events add no synchronisation.
 */
gpulz_status gpulz_set_kernel_events(cudaEvent_t start, cudaEvent_t stop);

/* Static, human-readable name of a status code. */
const char* gpulz_status_string(gpulz_status status);

#ifdef __cplusplus
}
#endif

#endif /* GPULZ_H */
