// gpulz_compress_noalloc: the encode path with its scratch in a fixed,
// file-scope device array instead of memory the library allocates.
//
// Some callers cannot let a library call cudaMalloc: code that runs while a
// framework's caching allocator has already reserved the device memory, code
// on a latency-critical path where cudaMalloc's implicit device-wide
// synchronisation is not acceptable, and plug-ins whose host forbids
// allocations behind its back. This entry point serves them: it allocates
// nothing, ever. Its look-back descriptors, ticket counter and status word live
// in g_noalloc_scratch below, which every GPU that loads the library holds
// until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/gpulz.h"
#include "gpulz_internal.cuh"

namespace {

using namespace gpulz;

// Largest input the fixed scratch can serve: one 8-byte look-back descriptor
// per chunk.
constexpr uint64_t kNoAllocMaxChunks = 65536;
constexpr size_t kNoAllocHead = 256;  // u32 status at 0, u32 ticket at 4
constexpr size_t kNoAllocBytes = kNoAllocHead + sizeof(uint64_t) * kNoAllocMaxChunks;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint8_t* g_scratch_dev[kMaxDevices] = {};
uint32_t g_epoch[kMaxDevices] = {};  // last epoch used on each device

// Device address of g_noalloc_scratch on the current device, looked up once
// per device with that device current, and the next epoch for this call.
// Look-back entries carry the epoch of the call that wrote them, and every
// call also clears, on its stream, the status word, the ticket and the entries
// of the chunks it codes, so no entry left by an earlier call (whatever its
// epoch) can be taken for one of this call's; on first use the whole array is
// cleared (*clear_all).
cudaError_t scratch_address(uint8_t** out, uint32_t* epoch, bool* clear_all) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    *clear_all = false;
    if (g_scratch_dev[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_dev[dev] = static_cast<uint8_t*>(p);
        *clear_all = true;
        g_epoch[dev] = 0;
    }
    g_epoch[dev] += 1;
    if (g_epoch[dev] >= kEpochs) g_epoch[dev] = 1;
    *out = g_scratch_dev[dev];
    *epoch = g_epoch[dev];
    return cudaSuccess;
}

// A bounded look-back wait that gave up is reported through the length:
// *d_out_bytes = SIZE_MAX.
__global__ void noalloc_report(const uint32_t* status, unsigned long long* out_bytes) {
    if (threadIdx.x == 0 && (*status & kStatTimeout)) *out_bytes = ~0ull;
}

}  // namespace

extern "C" gpulz_status gpulz_compress_noalloc(const void* d_in, size_t n_bytes, int word_size,
                                               int chunk_size, int match_level, void* d_out,
                                               size_t capacity, size_t* d_out_bytes,
                                               cudaStream_t stream) {
    if (!valid_geometry(word_size, chunk_size)) return GPULZ_ERR_INVALID_ARG;
    if (match_level != 0 && match_level != 1) return GPULZ_ERR_INVALID_ARG;
    if ((n_bytes > 0 && d_in == nullptr) || d_out == nullptr || d_out_bytes == nullptr)
        return GPULZ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_out) & 3u) || (reinterpret_cast<uintptr_t>(d_out_bytes) & 7u))
        return GPULZ_ERR_INVALID_ARG;
    const uint64_t chunks = ((uint64_t)n_bytes + chunk_size - 1) / (uint64_t)chunk_size;
    if (chunks > kNoAllocMaxChunks) return GPULZ_ERR_INVALID_ARG;
    uint8_t* base = nullptr;
    uint32_t epoch = 0;
    bool clear_all = false;
    if (scratch_address(&base, &epoch, &clear_all) != cudaSuccess) return GPULZ_ERR_CUDA;
    // The array keeps the previous call's contents: clear the status word, the
    // ticket and this call's look-back entries (all of it on first use), in
    // stream order.
    const size_t used = kNoAllocHead + sizeof(uint64_t) * (size_t)chunks;
    if (cudaMemsetAsync(base, 0, clear_all ? kNoAllocBytes : used, stream) != cudaSuccess)
        return GPULZ_ERR_CUDA;
    EncodeArgs a;
    a.in = static_cast<const uint8_t*>(d_in);
    a.n_bytes = n_bytes;
    a.out = static_cast<uint8_t*>(d_out);
    a.capacity = capacity;
    a.out_bytes = reinterpret_cast<unsigned long long*>(d_out_bytes);
    a.desc = reinterpret_cast<uint64_t*>(base + kNoAllocHead);
    a.slots = nullptr;
    a.sizes = nullptr;
    a.msizes = nullptr;
    a.offsets = nullptr;
    a.tdesc_stride = 0;
    a.split = 0;
    for (int k = 0; k < 3; ++k) {
        a.port[k] = nullptr;
        a.port_cap[k] = 0;
    }
    a.tdesc = nullptr;
    a.ticket2 = nullptr;
    a.ticket = reinterpret_cast<uint32_t*>(base + 4);
    a.status = reinterpret_cast<uint32_t*>(base);
    a.epoch = epoch;
    a.chunk_size = (uint32_t)chunk_size;
    a.elems = (uint32_t)(chunk_size / word_size);
    a.n_chunks = (uint32_t)chunks;
    a.hash_bits = log2_exact(2u * a.elems);
    a.far_mask = 0u;
    if (launch_encode(a, word_size, match_level, true, stream) != cudaSuccess)
        return GPULZ_ERR_CUDA;
    noalloc_report<<<1, 32, 0, stream>>>(a.status, a.out_bytes);
    if (cudaGetLastError() != cudaSuccess) return GPULZ_ERR_CUDA;
    return GPULZ_OK;
}
