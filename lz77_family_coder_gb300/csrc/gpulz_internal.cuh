// Internal definitions shared by the GPULZ encode/decode kernels and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gpulz {

// ---- stream format v1 (see include/gpulz.h) ----
constexpr uint32_t kMagic = 0x5A4C5047u;  // "GPLZ"
constexpr uint32_t kVersion = 1u;
constexpr uint32_t kHeaderBytes = 32u;
constexpr uint32_t kEntryBytes = 8u;
constexpr uint32_t kRawBit = 0x80000000u;
// split mode (four ports): meta = 48-byte header {u32 magic, u16 version 2,
// u8 word_size, u8 0, u32 chunk_size, u32 n_chunks, u64 orig_bytes,
// u64 meta_bytes, u64 literal_bytes, u64 n_matches}, the size table
// {u32 n_items | RAW << 31, u32 n_matches} per chunk, then every coded
// chunk's flag words; literals, lengths and offsets back to back
constexpr uint32_t kSplitVersion = 2u;
constexpr uint32_t kSplitHeaderBytes = 48u;

// ---- method constants (GPULZ stage page, match-search section) ----
constexpr int kWindow = 32;     // near window, elements
constexpr int kMaxLen = 255;    // one-byte length field
constexpr int kMaxOff = 255;    // one-byte offset field
constexpr int kSubBlocks = 8;   // level-1 sub-blocks per chunk

// Shortest match worth a 2-byte token: its literal bytes must exceed 2.
__host__ __device__ constexpr int min_match_len(int ws) { return ws == 1 ? 3 : (ws == 2 ? 2 : 1); }

__host__ __device__ inline bool valid_geometry(int ws, int cs) {
    return (ws == 1 || ws == 2 || ws == 4) && (cs == 1024 || cs == 2048 || cs == 4096);
}

// ---- device status bits ----
constexpr uint32_t kStatCorrupt = 1u;
constexpr uint32_t kStatTimeout = 2u;
constexpr uint32_t kStatCapacity = 4u;
constexpr uint32_t kStatSizeMismatch = 8u;

// ---- per-(device, stream) scratch layout ----
// [0, 256)                    status word (u32 at 0)
// [256, 256 + 8*65536)        two ticket counters per epoch (epoch in [1, 65535])
// [kStateOffset, ...)         scratch_regions(): tile descriptors, per-chunk words,
//                             block slots
constexpr uint32_t kEpochs = 65536u;
constexpr size_t kTicketOffset = 256;
constexpr size_t kStateOffset = kTicketOffset + 2 * sizeof(uint32_t) * kEpochs;

// Scan tiles: one CTA of kScanThreads threads covers kTile chunks.
constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 4;
constexpr uint32_t kTile = kScanThreads * kScanPerThread;

struct ScratchRegions {
    size_t tdesc, offsets, sizes, slots, end;  // byte offsets from the state base
};
// cap_chunks: chunks the per-chunk arrays can hold; slot_bytes: bytes of block
// slots (chunks x chunk_size for the two-pass encode, 0 otherwise). Three
// tile-descriptor arrays, three u64 offsets and two u32 sizes per chunk (the
// single-stream form uses the first of each; split mode all three).
__host__ __device__ constexpr uint64_t tdesc_len(uint64_t cap_chunks) { return cap_chunks / kTile + 2; }
__host__ __device__ constexpr ScratchRegions scratch_regions(uint64_t cap_chunks,
                                                            uint64_t slot_bytes) {
    ScratchRegions r{};
    r.tdesc = 0;
    r.offsets = 3 * 8 * tdesc_len(cap_chunks);        // 3 x u64 per chunk
    r.sizes = r.offsets + 3 * 8 * cap_chunks;         // 2 x u32 per chunk
    r.slots = (r.sizes + 2 * 4 * cap_chunks + 255) & ~(size_t)255;
    r.end = r.slots + slot_bytes;
    return r;
}

// Descriptor: [63:48] epoch, [47:46] kind, [45:0] value (bytes).
constexpr uint64_t kDescAggregate = 1ull;
constexpr uint64_t kDescInclusive = 2ull;
__host__ __device__ inline uint64_t make_desc(uint32_t epoch, uint64_t kind, uint64_t value) {
    return ((uint64_t)epoch << 48) | (kind << 46) | (value & ((1ull << 46) - 1));
}
__device__ inline uint32_t desc_epoch(uint64_t d) { return (uint32_t)(d >> 48); }
__device__ inline uint64_t desc_kind(uint64_t d) { return (d >> 46) & 3ull; }
__device__ inline uint64_t desc_value(uint64_t d) { return d & ((1ull << 46) - 1); }

// Bounded waits: give up after this many nanoseconds of device time.
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;

__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Level-1 bucket of a two-word key; `bits` = log2(2 * elements per chunk).
__device__ __forceinline__ uint32_t key_hash(uint32_t k0, uint32_t k1, uint32_t bits) {
    return ((k0 * 0x9E3779B1u) ^ (k1 * 0x85EBCA77u)) >> (32u - bits);
}

__host__ __device__ inline uint32_t log2_exact(uint32_t v) {
    uint32_t b = 0;
    while ((1u << b) < v) ++b;
    return b;
}

// ---- decoupled look-back over an array of descriptors (one warp) ----
constexpr int kLBPerLane = 8;  // 32 lanes x 8 descriptors per step
constexpr uint32_t kLBWidth = 32u * kLBPerLane;

struct LBStep {
    uint64_t sum;
    bool found;
    bool wait;
    uint32_t first_bad;  // smallest distance not yet published (when wait)
};

// One step over arr[top - dist], dist in [0, count) (count <= kLBWidth); an
// index below 0 reads as an inclusive prefix of 0. Sums the values back to
// (and including) the nearest inclusive prefix, or all `count` if none.
__device__ __forceinline__ LBStep lb_step(const uint64_t* arr, int64_t top, uint32_t count,
                                          uint32_t epoch, int lane) {
    uint64_t d[kLBPerLane];
#pragma unroll
    for (int k = 0; k < kLBPerLane; ++k) {
        const uint32_t dist = (uint32_t)(k * 32 + lane);
        const int64_t idx = top - (int64_t)dist;
        d[k] = dist >= count ? 0ull
                             : (idx >= 0 ? ld_relaxed_u64(arr + idx)
                                         : make_desc(epoch, kDescInclusive, 0));
    }
    uint32_t my_min = 0xFFFFFFFFu;
#pragma unroll
    for (int k = kLBPerLane - 1; k >= 0; --k) {
        const uint32_t dist = (uint32_t)(k * 32 + lane);
        if (dist < count && desc_epoch(d[k]) == epoch && desc_kind(d[k]) == kDescInclusive)
            my_min = dist;
    }
    const uint32_t dmin = __reduce_min_sync(0xFFFFFFFFu, my_min);
    const uint32_t lim = dmin == 0xFFFFFFFFu ? count : dmin + 1u;
    uint32_t my_bad = 0xFFFFFFFFu;
    uint64_t v = 0;
#pragma unroll
    for (int k = kLBPerLane - 1; k >= 0; --k) {
        const uint32_t dist = (uint32_t)(k * 32 + lane);
        if (dist < lim) {
            if (!(desc_epoch(d[k]) == epoch && desc_kind(d[k]) != 0)) my_bad = dist;
            v += desc_value(d[k]);
        }
    }
    LBStep r;
    r.first_bad = __reduce_min_sync(0xFFFFFFFFu, my_bad);
    r.wait = r.first_bad != 0xFFFFFFFFu;
    r.found = dmin != 0xFFFFFFFFu;
    r.sum = warp_sum_u64(v);
    return r;
}

// Lane 0 polls one descriptor, backing off, until it carries this call's
// epoch. Returns false if the wait gave up after limit_ns (measured from *t0,
// set on the first wait).
__device__ __forceinline__ bool wait_published(const uint64_t* arr, int64_t idx, uint32_t epoch,
                                               int lane, uint64_t* t0, uint64_t limit_ns) {
    bool ok = true;
    if (lane == 0) {
        uint32_t ns = 32;
        for (;;) {
            const uint64_t d = ld_relaxed_u64(arr + idx);
            if (desc_epoch(d) == epoch && desc_kind(d) != 0) break;
            const uint64_t now = globaltimer_ns();
            if (*t0 == 0) *t0 = now;
            if (now - *t0 > limit_ns) {
                ok = false;
                break;
            }
            __nanosleep(ns);
            if (ns < 1024) ns <<= 1;
        }
    }
    return __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
}

// Exclusive prefix of `value` over entries [0, idx) of arr (one warp). The
// caller has published arr[idx] (aggregate). Publishes arr[idx]'s inclusive
// prefix. Every wait is on entries with smaller tickets, which publish their
// aggregates without waiting. A wait that gives up (limit_ns) sets
// *timed_out; arr[idx] is then still published, with the partial sum, so that
// later entries do not wait as well (the caller records the timeout, which
// marks the whole result invalid).
__device__ __forceinline__ uint64_t lookback(uint64_t* arr, uint32_t idx, uint64_t value,
                                             uint32_t epoch, int lane, bool* timed_out,
                                             uint64_t limit_ns = kWaitLimitNs) {
    *timed_out = false;
    uint64_t prefix = 0;
    int64_t top = (int64_t)idx - 1;
    uint64_t t0 = 0;
    while (top >= 0) {
        const LBStep r = lb_step(arr, top, kLBWidth, epoch, lane);
        if (r.wait) {
            if (!wait_published(arr, top - (int64_t)r.first_bad, epoch, lane, &t0, limit_ns)) {
                *timed_out = true;
                break;
            }
            continue;
        }
        prefix += r.sum;
        if (r.found) break;
        top -= kLBWidth;
    }
    if (lane == 0) st_relaxed_u64(&arr[idx], make_desc(epoch, kDescInclusive, prefix + value));
    return prefix;
}

// Per-tile scan used by the encode pack pass and the decode offset pass: the
// CTA (kScanThreads threads) takes the next tile ticket, computes the
// exclusive offsets of its chunks' sizes (s_off, relative to the tile) and
// the tile's exclusive prefix over earlier tiles (returned), by decoupled
// look-back over tile descriptors. size_of(c) gives chunk c's block size.
struct TileSmem {
    uint32_t off[kTile];
    uint32_t size[kTile];
    uint32_t warp_sum[kScanThreads / 32];
    uint32_t tile;
    uint32_t total;
    unsigned long long prefix;
    uint32_t flags;
};

template <typename SizeFn>
__device__ __forceinline__ uint64_t tile_scan(TileSmem& sm, uint32_t t, uint32_t n_chunks,
                                              uint64_t* tdesc, uint32_t epoch, uint32_t* status,
                                              SizeFn size_of) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t c0 = t * kTile;
    uint32_t v[kScanPerThread];
    uint32_t sum = 0;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        const uint32_t c = c0 + (uint32_t)(tid * kScanPerThread + k);
        v[k] = c < n_chunks ? size_of(c) : 0u;
        sum += v[k];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += x;
    }
    if (lane == 31) sm.warp_sum[warp] = incl;
    __syncthreads();
    uint32_t wbase = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kScanThreads / 32; ++w) {
        const uint32_t x = sm.warp_sum[w];
        if (w < warp) wbase += x;
        total += x;
    }
    uint32_t excl = wbase + incl - sum;
#pragma unroll
    for (int k = 0; k < kScanPerThread; ++k) {
        sm.off[tid * kScanPerThread + k] = excl;
        sm.size[tid * kScanPerThread + k] = v[k];
        excl += v[k];
    }
    if (warp == 0) {
        if (lane == 0)
            st_relaxed_u64(&tdesc[t], make_desc(epoch, t == 0 ? kDescInclusive : kDescAggregate,
                                                total));
        uint64_t prefix = 0;
        if (t > 0) {
            bool to = false;
            prefix = lookback(tdesc, t, total, epoch, lane, &to);
            if (to && lane == 0) atomicOr(status, kStatTimeout);
        }
        if (lane == 0) {
            sm.prefix = prefix;
            sm.total = total;
        }
    }
    __syncthreads();
    return sm.prefix;
}

struct EncodeArgs {
    const uint8_t* in;
    uint64_t n_bytes;
    uint8_t* out;
    uint64_t capacity;
    unsigned long long* out_bytes;
    uint64_t* desc;     // single pass: per chunk aggregate, then inclusive prefix
    uint8_t* slots;     // two pass: chunk c's block at slots + c * chunk_size
    uint32_t* sizes;    // two pass: chunk c's block size (split: its literal bytes)
    uint32_t* msizes;   // split: chunk c's matches | flag words << 16
    uint64_t* offsets;  // two pass: chunk c's block offset (split: 3 per chunk,
                        // flag bytes / literal bytes / matches before it)
    uint64_t* tdesc;    // two pass: tile descriptors of the pack pass (split: 3 arrays)
    uint64_t tdesc_stride;  // split: distance between the descriptor arrays
    uint32_t* ticket2;  // two pass: tile ticket of the pack pass
    // split mode: out/capacity is the meta port; three more ports, and
    // out_bytes points at 4 u64 (meta, literals, lengths, offsets)
    uint32_t split;
    uint8_t* port[3];
    uint64_t port_cap[3];
    uint32_t* ticket;
    uint32_t* status;
    uint32_t epoch;
    uint32_t chunk_size;
    uint32_t elems;
    uint32_t n_chunks;
    uint32_t hash_bits;
    uint32_t far_mask;  // near window 33..64: offsets 33..window as bits 0..window-33; 0 = 32
};

struct DecodeArgs {
    const uint8_t* in;
    uint64_t in_bytes;
    uint8_t* out;
    uint64_t n_bytes;
    uint64_t* offsets;  // per chunk: stream offset of its block (written by the offset pass)
    uint64_t* tdesc;    // tile descriptors of the offset pass
    uint32_t* ticket;   // tile ticket of the offset pass
    uint32_t* ticket2;  // chunk ticket of the decode pass
    uint32_t* status;
    uint32_t epoch;
    // split mode: `in` is the meta port; three more ports with their lengths;
    // offsets then holds 3 per chunk (flag words, literal bytes, matches before
    // it) and tdesc 3 arrays tdesc_stride apart
    uint32_t split;
    const uint8_t* port[3];
    uint64_t port_len[3];
    uint64_t tdesc_stride;
};

// Programmatic dependent launch: a kernel launched with pdl_launch() may be
// scheduled before the previous kernel in the stream has finished; it calls
// pdl_wait() before it reads anything that kernel writes (the wait returns
// once that kernel has completed and its memory is visible). pdl_trigger()
// lets the next kernel be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Events a caller asked to bracket the main kernel with (see
// gpulz_set_kernel_events); both null when unset. Per host thread.
struct KernelEvents {
    cudaEvent_t start, stop;
};
KernelEvents& kernel_events();

// Host launchers (gpulz_encode.cu / gpulz_decode.cu). Return a CUDA error.
// single_pass: one kernel, blocks placed by look-back over chunk descriptors
// (needs only `desc`); otherwise encode into slots, then the pack pass.
cudaError_t launch_encode(const EncodeArgs& a, int word_size, int match_level, bool single_pass,
                          cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace gpulz
