// C ABI of the GPULZ coder: argument checks, per-(device, stream) scratch,
// launches and the device status word. The kernels live in gpulz_encode.cu and
// gpulz_decode.cu.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/gpulz.h"
#include "../../include/gpulz_testing.h"
#include "gpulz_internal.cuh"

namespace {

using namespace gpulz;

// Scratch of one (device, stream): status word, two ticket counters per
// epoch, tile descriptors, one word per chunk (block sizes or offsets) and,
// for the two-pass encode, one chunk_size slot per chunk. A call takes the
// next epoch; descriptors and tickets of other epochs never match, so nothing
// is cleared between calls. When the 16-bit epoch wraps, the whole area is
// cleared once on the stream.
struct Scratch {
    int device;
    cudaStream_t stream;
    uint8_t* base;
    uint64_t cap_chunks;
    uint64_t slot_bytes;
    uint32_t epoch;  // last epoch used
};

std::mutex g_mu;
std::vector<Scratch*> g_scratch;

size_t scratch_bytes(uint64_t cap_chunks, uint64_t slot_bytes) {
    return kStateOffset + scratch_regions(cap_chunks, slot_bytes).end;
}

// Returns the scratch for (current device, stream) with room for `chunks`
// per-chunk words and `slot_bytes` of slots, and advances its epoch. While the
// stream is being captured into a graph nothing may be allocated (the graph
// would own the area): the scratch must already be large enough.
cudaError_t acquire_scratch(cudaStream_t stream, uint64_t chunks, uint64_t slot_bytes,
                            bool capturing, Scratch** out, uint32_t* epoch_out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_mu);
    Scratch* s = nullptr;
    for (Scratch* t : g_scratch)
        if (t->device == dev && t->stream == stream) s = t;
    if (s == nullptr) {
        s = new Scratch{dev, stream, nullptr, 0, 0, 0};
        g_scratch.push_back(s);
    }
    if (s->base == nullptr || s->cap_chunks < chunks || s->slot_bytes < slot_bytes) {
        if (capturing) return cudaErrorStreamCaptureUnsupported;
        const uint64_t cap = chunks < 4096 ? 4096 : (chunks > s->cap_chunks ? chunks : s->cap_chunks);
        const uint64_t sb = slot_bytes > s->slot_bytes ? slot_bytes : s->slot_bytes;
        void* p = nullptr;
        if ((err = cudaMallocAsync(&p, scratch_bytes(cap, sb), stream)) != cudaSuccess) return err;
        // slots need no clearing: every byte read from a slot was written by the same call
        if ((err = cudaMemsetAsync(p, 0, kStateOffset + scratch_regions(cap, sb).slots, stream)) !=
            cudaSuccess)
            return err;
        if (s->base != nullptr) {
            // keep recorded errors; earlier work on this stream still owns the old area,
            // so it is released in stream order
            if ((err = cudaMemcpyAsync(p, s->base, sizeof(uint32_t), cudaMemcpyDeviceToDevice,
                                       stream)) != cudaSuccess)
                return err;
            if ((err = cudaFreeAsync(s->base, stream)) != cudaSuccess) return err;
            s->base = nullptr;
        }
        s->base = static_cast<uint8_t*>(p);
        s->cap_chunks = cap;
        s->slot_bytes = sb;
        s->epoch = 0;
    }
    s->epoch += 1;
    if (s->epoch >= kEpochs) {
        // clear tickets and descriptors (keep the status word)
        if ((err = cudaMemsetAsync(s->base + kTicketOffset, 0,
                                   kStateOffset - kTicketOffset +
                                       scratch_regions(s->cap_chunks, s->slot_bytes).slots,
                                   stream)) != cudaSuccess)
            return err;
        s->epoch = 1;
    }
    *out = s;
    *epoch_out = s->epoch;
    return cudaSuccess;
}

// A graph captured from a call launches it again and again with the epoch it
// took at capture. Each launch starts and ends by putting that epoch's two
// ticket counters and the tile descriptors back to the clean state (zero: no
// descriptor carries epoch 0), so every launch, and a direct call that later
// takes the same epoch, finds them as a fresh epoch.
cudaError_t clear_epoch_state(const Scratch* s, uint32_t epoch, cudaStream_t stream) {
    cudaError_t err = cudaMemsetAsync(s->base + kTicketOffset + 2 * sizeof(uint32_t) * epoch, 0,
                                      2 * sizeof(uint32_t), stream);
    if (err != cudaSuccess) return err;
    const ScratchRegions r = scratch_regions(s->cap_chunks, s->slot_bytes);
    return cudaMemsetAsync(s->base + kStateOffset + r.tdesc, 0, r.offsets - r.tdesc, stream);
}

// Whether `stream` is being captured into a graph.
cudaError_t is_capturing(cudaStream_t stream, bool* capturing) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaError_t err = cudaStreamIsCapturing(stream, &st);
    *capturing = st != cudaStreamCaptureStatusNone;
    return err;
}

// Removes and returns the scratch entry of (current device, stream), or null.
Scratch* take_scratch(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    for (size_t k = 0; k < g_scratch.size(); ++k) {
        Scratch* t = g_scratch[k];
        if (t->device == dev && t->stream == stream) {
            g_scratch.erase(g_scratch.begin() + (long)k);
            return t;
        }
    }
    return nullptr;
}

// Test hook: one warp runs the library's look-back over a caller-made
// descriptor array with the given wait limit; a wait that gives up records
// the timeout in the stream's status word, as the coder's kernels do.
__global__ void lookback_probe(uint64_t* desc, uint32_t idx, uint64_t value, uint32_t epoch,
                               uint64_t limit_ns, unsigned long long* prefix_out,
                               uint32_t* status) {
    const int lane = threadIdx.x & 31;
    bool to = false;
    const uint64_t prefix = lookback(desc, idx, value, epoch, lane, &to, limit_ns);
    if (lane == 0) {
        *prefix_out = prefix;
        if (to) atomicOr(status, kStatTimeout);
    }
}

Scratch* find_scratch(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    for (Scratch* t : g_scratch)
        if (t->device == dev && t->stream == stream && t->base) return t;
    return nullptr;
}

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

namespace gpulz {
KernelEvents& kernel_events() {
    static thread_local KernelEvents ev{nullptr, nullptr};
    return ev;
}
}  // namespace gpulz

extern "C" {

size_t gpulz_compress_bound(size_t n_bytes, int word_size, int chunk_size) {
    if (!valid_geometry(word_size, chunk_size)) return 0;
    uint64_t chunks = ((uint64_t)n_bytes + (uint64_t)chunk_size - 1) / (uint64_t)chunk_size;
    return (size_t)(kHeaderBytes + chunks * ((uint64_t)kEntryBytes + (uint64_t)chunk_size));
}

namespace {
// Shared by the single-stream and split encoders: argument checks, scratch,
// and the launch. ports/port_cap are null for the single-stream form.
gpulz_status compress_impl(const void* d_in, size_t n_bytes, int word_size, int chunk_size,
                           int match_level, int window, void* d_out, size_t capacity,
                           size_t* d_out_bytes, uint8_t* const* ports, const size_t* port_cap,
                           cudaStream_t stream) {
    if (!valid_geometry(word_size, chunk_size)) return GPULZ_ERR_INVALID_ARG;
    if (match_level != 0 && match_level != 1) return GPULZ_ERR_INVALID_ARG;
    if (window < 32 || window > 64 || (window > 32 && match_level != 0)) return GPULZ_ERR_INVALID_ARG;
    if ((n_bytes > 0 && d_in == nullptr) || d_out == nullptr || d_out_bytes == nullptr)
        return GPULZ_ERR_INVALID_ARG;
    if (!aligned(d_out, 4) || !aligned(d_out_bytes, 8)) return GPULZ_ERR_INVALID_ARG;
    const uint64_t chunks = ((uint64_t)n_bytes + chunk_size - 1) / (uint64_t)chunk_size;
    if (chunks > 0xFFFFFFFFull) return GPULZ_ERR_INVALID_ARG;
    bool capturing = false;
    if (is_capturing(stream, &capturing) != cudaSuccess) return GPULZ_ERR_CUDA;
    Scratch* s = nullptr;
    uint32_t epoch = 0;
    cudaError_t err = acquire_scratch(stream, chunks, chunks * (uint64_t)chunk_size, capturing,
                                      &s, &epoch);
    if (err == cudaErrorStreamCaptureUnsupported) return GPULZ_ERR_INVALID_ARG;
    if (err != cudaSuccess) return GPULZ_ERR_CUDA;
    if (capturing && clear_epoch_state(s, epoch, stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    const ScratchRegions r = scratch_regions(s->cap_chunks, s->slot_bytes);
    uint8_t* st = s->base + kStateOffset;
    uint32_t* tickets = reinterpret_cast<uint32_t*>(s->base + kTicketOffset);
    EncodeArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.n_bytes = n_bytes;
    a.out = static_cast<uint8_t*>(d_out);
    a.capacity = capacity;
    a.out_bytes = reinterpret_cast<unsigned long long*>(d_out_bytes);
    a.desc = nullptr;
    a.slots = st + r.slots;
    a.sizes = reinterpret_cast<uint32_t*>(st + r.sizes);
    a.msizes = a.sizes + s->cap_chunks;
    a.offsets = reinterpret_cast<uint64_t*>(st + r.offsets);
    a.tdesc = reinterpret_cast<uint64_t*>(st + r.tdesc);
    a.tdesc_stride = tdesc_len(s->cap_chunks);
    a.ticket = tickets + 2 * epoch;
    a.ticket2 = tickets + 2 * epoch + 1;
    a.status = reinterpret_cast<uint32_t*>(s->base);
    a.epoch = epoch;
    a.chunk_size = (uint32_t)chunk_size;
    a.elems = (uint32_t)(chunk_size / word_size);
    a.n_chunks = (uint32_t)chunks;
    a.hash_bits = log2_exact(2u * a.elems);
    a.far_mask = window == 32 ? 0u : (window == 64 ? 0xFFFFFFFFu : (1u << (window - 32)) - 1u);
    a.split = ports != nullptr;
    for (int k = 0; k < 3; ++k) {
        a.port[k] = ports ? ports[k] : nullptr;
        a.port_cap[k] = ports ? port_cap[k] : 0;
    }
    if (launch_encode(a, word_size, match_level, false, stream) != cudaSuccess)
        return GPULZ_ERR_CUDA;
    if (capturing && clear_epoch_state(s, epoch, stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    return GPULZ_OK;
}
}  // namespace

gpulz_status gpulz_compress(const void* d_in, size_t n_bytes, int word_size, int chunk_size,
                            int match_level, void* d_out, size_t capacity, size_t* d_out_bytes,
                            cudaStream_t stream) {
    return compress_impl(d_in, n_bytes, word_size, chunk_size, match_level, 32, d_out, capacity,
                         d_out_bytes, nullptr, nullptr, stream);
}

gpulz_status gpulz_compress_window(const void* d_in, size_t n_bytes, int word_size,
                                   int chunk_size, int match_level, int window, void* d_out,
                                   size_t capacity, size_t* d_out_bytes, cudaStream_t stream) {
    return compress_impl(d_in, n_bytes, word_size, chunk_size, match_level, window, d_out,
                         capacity, d_out_bytes, nullptr, nullptr, stream);
}

gpulz_status gpulz_split_bounds(size_t n_bytes, int word_size, int chunk_size, size_t bounds[4]) {
    if (!valid_geometry(word_size, chunk_size) || bounds == nullptr) return GPULZ_ERR_INVALID_ARG;
    const uint64_t chunks = ((uint64_t)n_bytes + chunk_size - 1) / (uint64_t)chunk_size;
    const uint64_t elems = (uint64_t)(chunk_size / word_size);
    bounds[0] = (size_t)(kSplitHeaderBytes + kEntryBytes * chunks + 4u * chunks * ((elems + 31u) / 32u));
    bounds[1] = (size_t)(chunks * (uint64_t)chunk_size);
    bounds[2] = (size_t)(chunks * elems);
    bounds[3] = (size_t)(chunks * elems);
    return GPULZ_OK;
}

gpulz_status gpulz_compress_split(const void* d_in, size_t n_bytes, int word_size, int chunk_size,
                                  int match_level, void* d_meta, void* d_literals,
                                  void* d_lengths, void* d_offsets, const size_t capacity[4],
                                  size_t* d_port_bytes, cudaStream_t stream) {
    if (capacity == nullptr || d_literals == nullptr || d_lengths == nullptr || d_offsets == nullptr)
        return GPULZ_ERR_INVALID_ARG;
    uint8_t* const ports[3] = {static_cast<uint8_t*>(d_literals), static_cast<uint8_t*>(d_lengths),
                               static_cast<uint8_t*>(d_offsets)};
    return compress_impl(d_in, n_bytes, word_size, chunk_size, match_level, 32, d_meta,
                         capacity[0], d_port_bytes, ports, capacity + 1, stream);
}

namespace {
gpulz_status decompress_impl(const void* d_in, size_t in_bytes, void* d_out, size_t n_bytes,
                             const uint8_t* const* ports, const size_t* port_len,
                             cudaStream_t stream) {
    if (d_in == nullptr || (n_bytes > 0 && d_out == nullptr)) return GPULZ_ERR_INVALID_ARG;
    if (!aligned(d_in, 4)) return GPULZ_ERR_INVALID_ARG;
    const uint64_t max_chunks = ((uint64_t)n_bytes + 1023u) / 1024u;
    bool capturing = false;
    if (is_capturing(stream, &capturing) != cudaSuccess) return GPULZ_ERR_CUDA;
    Scratch* s = nullptr;
    uint32_t epoch = 0;
    const cudaError_t err = acquire_scratch(stream, max_chunks, 0, capturing, &s, &epoch);
    if (err == cudaErrorStreamCaptureUnsupported) return GPULZ_ERR_INVALID_ARG;
    if (err != cudaSuccess) return GPULZ_ERR_CUDA;
    if (capturing && clear_epoch_state(s, epoch, stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    const ScratchRegions r = scratch_regions(s->cap_chunks, s->slot_bytes);
    uint8_t* st = s->base + kStateOffset;
    uint32_t* tickets = reinterpret_cast<uint32_t*>(s->base + kTicketOffset);
    DecodeArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.in_bytes = in_bytes;
    a.out = static_cast<uint8_t*>(d_out);
    a.n_bytes = n_bytes;
    a.offsets = reinterpret_cast<uint64_t*>(st + r.offsets);
    a.tdesc = reinterpret_cast<uint64_t*>(st + r.tdesc);
    a.tdesc_stride = tdesc_len(s->cap_chunks);
    a.ticket = tickets + 2 * epoch;
    a.ticket2 = tickets + 2 * epoch + 1;
    a.status = reinterpret_cast<uint32_t*>(s->base);
    a.epoch = epoch;
    a.split = ports != nullptr;
    for (int k = 0; k < 3; ++k) {
        a.port[k] = ports ? ports[k] : nullptr;
        a.port_len[k] = ports ? port_len[k] : 0;
    }
    if (launch_decode(a, stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    if (capturing && clear_epoch_state(s, epoch, stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    return GPULZ_OK;
}
}  // namespace

gpulz_status gpulz_decompress_bounded(const void* d_in, size_t in_bytes, void* d_out,
                                      size_t n_bytes, cudaStream_t stream) {
    return decompress_impl(d_in, in_bytes, d_out, n_bytes, nullptr, nullptr, stream);
}

gpulz_status gpulz_decompress_split(const void* d_meta, const void* d_literals,
                                    const void* d_lengths, const void* d_offsets,
                                    const size_t port_bytes[4], void* d_out, size_t n_bytes,
                                    cudaStream_t stream) {
    if (port_bytes == nullptr) return GPULZ_ERR_INVALID_ARG;
    // a null port counts as empty: every read of a port is bounded by its length
    const uint8_t* const ports[3] = {static_cast<const uint8_t*>(d_literals),
                                     static_cast<const uint8_t*>(d_lengths),
                                     static_cast<const uint8_t*>(d_offsets)};
    const size_t lens[3] = {d_literals ? port_bytes[1] : 0, d_lengths ? port_bytes[2] : 0,
                            d_offsets ? port_bytes[3] : 0};
    return decompress_impl(d_meta, port_bytes[0], d_out, n_bytes, ports, lens, stream);
}

gpulz_status gpulz_decompress(const void* d_in, void* d_out, size_t n_bytes, cudaStream_t stream) {
    return gpulz_decompress_bounded(d_in, SIZE_MAX, d_out, n_bytes, stream);
}

gpulz_status gpulz_stream_info(const void* h_header, size_t h_len, size_t* orig_bytes,
                               size_t* stream_bytes, int* word_size, int* chunk_size) {
    if (h_header == nullptr || h_len < kHeaderBytes) return GPULZ_ERR_INVALID_ARG;
    const uint8_t* h = static_cast<const uint8_t*>(h_header);
    uint32_t w[8];
    for (int k = 0; k < 8; ++k)
        w[k] = (uint32_t)h[4 * k] | ((uint32_t)h[4 * k + 1] << 8) | ((uint32_t)h[4 * k + 2] << 16) |
               ((uint32_t)h[4 * k + 3] << 24);
    const int ws = (int)((w[1] >> 16) & 0xFFu);
    const int cs = (int)w[2];
    const uint64_t orig = (uint64_t)w[4] | ((uint64_t)w[5] << 32);
    const uint64_t total = (uint64_t)w[6] | ((uint64_t)w[7] << 32);
    if (w[0] != kMagic || (w[1] & 0xFFFFu) != kVersion || (w[1] >> 24) != 0 ||
        !valid_geometry(ws, cs))
        return GPULZ_ERR_CORRUPT;
    const uint64_t chunks = (orig + (uint64_t)cs - 1) / (uint64_t)cs;
    if (chunks != w[3] || total < kHeaderBytes + kEntryBytes * chunks) return GPULZ_ERR_CORRUPT;
    if (orig_bytes) *orig_bytes = (size_t)orig;
    if (stream_bytes) *stream_bytes = (size_t)total;
    if (word_size) *word_size = ws;
    if (chunk_size) *chunk_size = cs;
    return GPULZ_OK;
}

gpulz_status gpulz_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GPULZ_ERR_CUDA;
    Scratch* s = find_scratch(stream);
    if (s == nullptr) return GPULZ_OK;
    uint32_t bits = 0;
    if (cudaMemcpy(&bits, s->base, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GPULZ_ERR_CUDA;
    if (bits != 0 && cudaMemset(s->base, 0, sizeof(bits)) != cudaSuccess) return GPULZ_ERR_CUDA;
    if (bits & kStatCorrupt) return GPULZ_ERR_CORRUPT;
    if (bits & kStatSizeMismatch) return GPULZ_ERR_SIZE_MISMATCH;
    if (bits & kStatTimeout) return GPULZ_ERR_TIMEOUT;
    if (bits & kStatCapacity) return GPULZ_ERR_CAPACITY;
    return GPULZ_OK;
}

gpulz_status gpulz_release_scratch(cudaStream_t stream) {
    if (find_scratch(stream) == nullptr) {
        // nothing held (an entry whose allocation failed holds no memory)
        delete take_scratch(stream);
        return GPULZ_OK;
    }
    bool capturing = false;
    if (is_capturing(stream, &capturing) != cudaSuccess) return GPULZ_ERR_CUDA;
    if (capturing) return GPULZ_ERR_INVALID_ARG;
    Scratch* s = take_scratch(stream);
    if (s == nullptr) return GPULZ_OK;
    const cudaError_t err = s->base ? cudaFreeAsync(s->base, stream) : cudaSuccess;
    delete s;
    return err == cudaSuccess ? GPULZ_OK : GPULZ_ERR_CUDA;
}

gpulz_status gpulz_test_lookback(uint64_t* d_desc, uint32_t idx, uint64_t value, uint32_t epoch,
                                 uint64_t limit_ns, size_t* d_prefix, cudaStream_t stream) {
    if (d_desc == nullptr || d_prefix == nullptr || epoch == 0 || epoch >= kEpochs ||
        limit_ns > kWaitLimitNs || !aligned(d_desc, 8) || !aligned(d_prefix, 8))
        return GPULZ_ERR_INVALID_ARG;
    bool capturing = false;
    if (is_capturing(stream, &capturing) != cudaSuccess) return GPULZ_ERR_CUDA;
    Scratch* s = nullptr;
    uint32_t scratch_epoch = 0;
    const cudaError_t err = acquire_scratch(stream, 0, 0, capturing, &s, &scratch_epoch);
    if (err == cudaErrorStreamCaptureUnsupported) return GPULZ_ERR_INVALID_ARG;
    if (err != cudaSuccess) return GPULZ_ERR_CUDA;
    lookback_probe<<<1, 32, 0, stream>>>(d_desc, idx, value, epoch, limit_ns,
                                         reinterpret_cast<unsigned long long*>(d_prefix),
                                         reinterpret_cast<uint32_t*>(s->base));
    return cudaGetLastError() == cudaSuccess ? GPULZ_OK : GPULZ_ERR_CUDA;
}

gpulz_status gpulz_set_kernel_events(cudaEvent_t start, cudaEvent_t stop) {
    if ((start == nullptr) != (stop == nullptr)) return GPULZ_ERR_INVALID_ARG;
    kernel_events() = KernelEvents{start, stop};
    return GPULZ_OK;
}

const char* gpulz_status_string(gpulz_status status) {
    switch (status) {
        case GPULZ_OK: return "ok";
        case GPULZ_ERR_INVALID_ARG: return "invalid argument";
        case GPULZ_ERR_CAPACITY: return "output capacity exceeded";
        case GPULZ_ERR_CORRUPT: return "corrupt stream";
        case GPULZ_ERR_TIMEOUT: return "device wait timed out";
        case GPULZ_ERR_CUDA: return "CUDA error";
        case GPULZ_ERR_SIZE_MISMATCH: return "n_bytes differs from the stream's original size";
    }
    return "unknown status";
}

}  // extern "C"
