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
// [0, 256)                 status word (u32 at 0)
// [256, 256 + 4*65536)     one ticket counter per epoch (epoch in [1, 65535])
// [kDescOffset, ...)       look-back descriptors, u64 per chunk
constexpr uint32_t kEpochs = 65536u;
constexpr size_t kTicketOffset = 256;
constexpr size_t kDescOffset = kTicketOffset + sizeof(uint32_t) * kEpochs;

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

struct EncodeArgs {
    const uint8_t* in;
    uint64_t n_bytes;
    uint8_t* out;
    uint64_t capacity;
    unsigned long long* out_bytes;
    uint64_t* desc;
    uint32_t* ticket;
    uint32_t* status;
    uint32_t epoch;
    uint32_t chunk_size;
    uint32_t elems;
    uint32_t n_chunks;
    uint32_t hash_bits;
};

struct DecodeArgs {
    const uint8_t* in;
    uint64_t in_bytes;
    uint8_t* out;
    uint64_t n_bytes;
    uint64_t* desc;
    uint32_t* ticket;
    uint32_t* status;
    uint32_t epoch;
};

// Host launchers (gpulz_encode.cu / gpulz_decode.cu). Return a CUDA error.
cudaError_t launch_encode(const EncodeArgs& a, int word_size, int match_level,
                          cudaStream_t stream);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

}  // namespace gpulz
