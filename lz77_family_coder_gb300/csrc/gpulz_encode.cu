// GPULZ encode kernel for sm_103a.
//
// One CTA ("team" of 1..8 warps) codes one chunk at a time and loops over
// chunks by ticket (persistent grid); every thread owns a segment of 8
// consecutive positions (16 for 4096-element chunks). Per chunk, following
// the GPULZ stage page of FZGPUModules:
//   E1 load + zero pad         (class summary; "Alignment" paragraph)
//   E2 zero test -> {0,0}      (zero-chunk paragraph)
//   E3 near equality masks     (match-search section: bit o-1 of omask[i])
//   E4 AND-chain longest match (match-search section; cap 255)
//   E5 level-1 hashed lookups  (match-search section: 8 sub-blocks, barrier
//                               between lookup and insert, atomicMax(pos+1))
//   E6 greedy parse            (provenance paragraph: sequential parse)
//   E7 flag bitmap + packing   (class summary: scan of item sizes, staging
//                               buffer, coalesced 32-bit stores)
//   E8 raw fallback            (raw-fallback paragraph)
//   E9 cross-chunk offsets     (two pass: tile scan of the block sizes;
//                               single pass: bounded decoupled look-back)
//   E10 store-out, size table, header and the stream length
//
// The greedy parse is computed in parallel: each thread walks its own
// segment from the segment start, then every thread whose true entry (the
// previous segment's exit) differs re-walks from it until its path meets the
// old one (paths that meet coincide afterwards); this repeats until a round
// changes no exit, when every entry equals the exit before it: exactly the
// sequential parse.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gpulz_internal.cuh"

namespace gpulz {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;

struct EncLayout {
    uint32_t el, om, lo, sa, tab, fl, data, misc, total;
};

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline EncLayout enc_layout(uint32_t cs, uint32_t E, int level) {
    EncLayout L;
    uint32_t o = 0;
    L.el = o;   o = align16(o + cs + E);                 // elements, 16 B pad per 16 elements
    L.om = o;   o = align16(o + 4u * (E + E / 4u));      // omask, 4 pad words per 16 masks
    L.lo = o;   o = align16(o + 2u * E);                 // (len | off << 8) per position
    L.sa = o;   o = align16(o + E / 2u);                 // AND of each segment's masks (<= E/8 u32)
    L.tab = o;  o = align16(o + (level ? 8u * E : 0u));  // level-1 table, 2E buckets of u32
    L.fl = o;   o = align16(o + E / 8u);                 // flag staging
    L.data = o; o = align16(o + cs + 16u);               // block staging
    L.misc = o; o = align16(o + 256u);
    L.total = o;
    return L;
}

// Warps per chunk: 8-position segments (16 for 4096-element chunks, which
// would need 16 warps). Short segments keep the register AND-chain triangle
// small, and more warps per chunk shorten the time a chunk takes, which is
// what the tail of the persistent grid waits for.
__host__ __device__ inline int team_warps(uint32_t E) { return E <= 256u ? 1 : (E >= 2048u ? 8 : (int)(E / 256u)); }

// Byte address of element i in the padded element array.
template <int WS>
__device__ __forceinline__ uint32_t el_addr(uint32_t i) {
    return i * WS + ((i >> 4) << 4);
}
template <int WS>
__device__ __forceinline__ uint32_t el_get(const uint8_t* el, uint32_t i) {
    const uint8_t* p = el + el_addr<WS>(i);
    if (WS == 4) return *reinterpret_cast<const uint32_t*>(p);
    if (WS == 2) return *reinterpret_cast<const uint16_t*>(p);
    return *p;
}
// Element i of an unpadded element array (level 1 keeps one in the staging
// buffer while the match search runs).
template <int WS>
__device__ __forceinline__ uint32_t lin_get(const uint8_t* lin, uint32_t i) {
    if (WS == 4) return reinterpret_cast<const uint32_t*>(lin)[i];
    if (WS == 2) return reinterpret_cast<const uint16_t*>(lin)[i];
    return lin[i];
}
template <int WS>
__device__ __forceinline__ uint32_t lin_at(const uint8_t* p, uint32_t k) {
    return lin_get<WS>(p, k);
}

// Word index of omask[i] in the padded omask array.
__device__ __forceinline__ uint32_t om_idx(uint32_t i) { return i + ((i >> 4) << 2); }

// Position of chunk byte b inside the padded element array.
template <int WS>
__device__ __forceinline__ uint32_t chunk_byte_addr(uint32_t b) {
    return b + ((b / (16u * WS)) << 4);
}

// ---------------------------------------------------------------------------
// Parse helpers.
// ---------------------------------------------------------------------------
// Step byte of relative position p (< 16) from four packed words.
__device__ __forceinline__ uint32_t seg_step(const uint32_t (&T)[4], uint32_t p) {
    const uint32_t lo = (p & 8u) ? T[2] : T[0];
    const uint32_t hi = (p & 8u) ? T[3] : T[1];
    return __byte_perm(lo, hi, p & 7u) & 0xFFu;
}

// OR `bits` (relative to bit position `start`) into a bitmask in shared memory.
__device__ __forceinline__ void or_bits(uint32_t* words, uint32_t start, uint32_t bits) {
    if (!bits) return;
    const uint32_t w = start >> 5, sh = start & 31u;
    atomicOr(&words[w], bits << sh);
    if (sh && (bits >> (32u - sh))) atomicOr(&words[w + 1], bits >> (32u - sh));
}

// ---------------------------------------------------------------------------
// Single-pass placement (used by the allocation-free entry point): chunk c
// publishes its block size, and its offset is the exclusive prefix over the
// chunk descriptors by decoupled look-back (lookback() in gpulz_internal.cuh).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void publish_size(const EncodeArgs& a, uint32_t c, uint32_t blk) {
    st_relaxed_u64(&a.desc[c], make_desc(a.epoch, c == 0 ? kDescInclusive : kDescAggregate, blk));
}

__device__ void store_u32_capped(uint8_t* out, uint64_t off, uint32_t v, uint64_t cap) {
    if (off + 4 <= cap) *reinterpret_cast<uint32_t*>(out + off) = v;
}

__device__ void write_header(const EncodeArgs& a, uint32_t ws, uint64_t total) {
    const uint32_t h[8] = {kMagic,
                           kVersion | (ws << 16),  // u16 version, u8 word_size, u8 reserved
                           a.chunk_size,
                           a.n_chunks,
                           (uint32_t)a.n_bytes,
                           (uint32_t)(a.n_bytes >> 32),
                           (uint32_t)total,
                           (uint32_t)(total >> 32)};
#pragma unroll
    for (int k = 0; k < 8; ++k) store_u32_capped(a.out, 4ull * k, h[k], a.capacity);
    *a.out_bytes = (unsigned long long)total;
    if (total > a.capacity) atomicOr(a.status, kStatCapacity);
}

// Split mode: the meta port's 48-byte header and the four port lengths.
__device__ void write_header_split(const EncodeArgs& a, uint32_t ws, uint64_t meta_bytes,
                                   uint64_t lit_bytes, uint64_t matches) {
    const uint32_t h[12] = {kMagic, kSplitVersion | (ws << 16), a.chunk_size, a.n_chunks,
                            (uint32_t)a.n_bytes, (uint32_t)(a.n_bytes >> 32),
                            (uint32_t)meta_bytes, (uint32_t)(meta_bytes >> 32),
                            (uint32_t)lit_bytes, (uint32_t)(lit_bytes >> 32),
                            (uint32_t)matches, (uint32_t)(matches >> 32)};
#pragma unroll
    for (int k = 0; k < 12; ++k) store_u32_capped(a.out, 4ull * k, h[k], a.capacity);
    a.out_bytes[0] = meta_bytes;
    a.out_bytes[1] = lit_bytes;
    a.out_bytes[2] = matches;
    a.out_bytes[3] = matches;
    if (meta_bytes > a.capacity || lit_bytes > a.port_cap[0] || matches > a.port_cap[1] ||
        matches > a.port_cap[2])
        atomicOr(a.status, kStatCapacity);
}

// The steps below are written as predicated PTX because the plain C forms
// (`mm |= (a == b) ? bit : 0`, and a select of the chain's new mask) compile
// to a compare, a select and an OR on the integer pipe, which bounds this
// kernel; the near masks alone are 32 compares per element. Measured, all
// streams unchanged: near masks +8-18 % encode on every workload, chain steps
// and verification compares a further +3-10 %, and chains that hold 0 once
// dead (no liveness test per step) +3-10 % more.
//
// mm |= bit where a == b: one compare and one predicated OR.
__device__ __forceinline__ void or_if_equal(uint32_t& mm, uint32_t a, uint32_t b, uint32_t bit) {
    asm("{\n\t.reg .pred q;\n\tsetp.eq.u32 q, %1, %2;\n\t@q or.b32 %0, %0, %3;\n\t}"
        : "+r"(mm)
        : "r"(a), "r"(b), "r"(bit));
}

// One AND-chain step for chains that hold 0 once dead: c &= m; where the
// result is nonzero, keep = c and an |= bit.
__device__ __forceinline__ void chain_step(uint32_t& c, uint32_t& keep, uint32_t& an, uint32_t m, uint32_t bit) {
    asm("{\n\t.reg .pred q;\n\tand.b32 %0, %0, %3;\n\tsetp.ne.u32 q, %0, 0;\n\t"
        "@q mov.b32 %1, %0;\n\t@q or.b32 %2, %2, %4;\n\t}"
        : "+r"(c), "+r"(keep), "+r"(an)
        : "r"(m), "r"(bit));
}

// an |= bit where x != 0: one test and one predicated OR.
__device__ __forceinline__ void or_if_nonzero(uint32_t& an, uint32_t x, uint32_t bit) {
    asm("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q or.b32 %0, %0, %2;\n\t}"
        : "+r"(an)
        : "r"(x), "r"(bit));
}

// Shared-memory byte store under a predicate (the byte staging pass).
__device__ __forceinline__ void st8_if(uint32_t on, uint8_t* p, uint32_t v) {
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.shared.u8 [%1], %2;\n\t}"
                 ::"r"(on), "r"((uint32_t)__cvta_generic_to_shared(p)), "h"((uint16_t)(v & 0xFFu))
                 : "memory");
}

// ---------------------------------------------------------------------------
// Per-segment near masks (E3): m[p] bit o-1 set iff element (base+p) equals
// element (base+p-o), 1 <= o <= 32, base+p-o >= 0.
// ---------------------------------------------------------------------------
template <int WS, int SEGP>
__device__ __forceinline__ void near_masks(const uint8_t* s_el, uint32_t base, uint32_t (&m)[SEGP]) {
    // Eight positions at a time: their 32-element window and themselves are
    // 40 elements, loaded as ten aligned 4-element vectors.
#pragma unroll
    for (int h = 0; h < SEGP / 8; ++h) {
        const int first = (int)base + 8 * h - 32;  // a multiple of 4
        uint32_t v[40];
#pragma unroll
        for (int q = 0; q < 10; ++q) {
            // a window element before the chunk is read from element 0 instead:
            // it only meets offsets past the position, whose bits the head
            // masking below clears
            const int i0 = max(first + 4 * q, 0);
            uint32_t w[4];
            const uint8_t* p = s_el + el_addr<WS>((uint32_t)i0);
            if (WS == 4) {
                const uint4 t = *reinterpret_cast<const uint4*>(p);
                w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
            } else if (WS == 2) {
                const uint2 t = *reinterpret_cast<const uint2*>(p);
                w[0] = t.x & 0xFFFFu; w[1] = t.x >> 16; w[2] = t.y & 0xFFFFu; w[3] = t.y >> 16;
            } else {
                const uint32_t t = *reinterpret_cast<const uint32_t*>(p);
                w[0] = t & 0xFFu; w[1] = (t >> 8) & 0xFFu; w[2] = (t >> 16) & 0xFFu; w[3] = t >> 24;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) v[4 * q + r] = w[r];
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint32_t x = v[32 + p];
            uint32_t mm = 0;
#pragma unroll
            for (int o = 1; o <= 32; ++o) or_if_equal(mm, v[32 + p - o], x, 1u << (o - 1));
            m[8 * h + p] = mm;
        }
    }
    if (base < 32u) {  // positions whose window starts before the chunk (the first threads only)
#pragma unroll
        for (int p = 0; p < SEGP; ++p) {
            const uint32_t i = base + (uint32_t)p;
            if (i < 32u) m[p] &= (1u << i) - 1u;
        }
    }
}

// True when every live chain (bit p of `live`) keeps an offset after AND-ing
// with `sa`, the AND of the masks of the positions to be skipped.
template <int SEGP>
__device__ __forceinline__ bool chains_live(const uint32_t (&cc)[SEGP], uint32_t live, uint32_t sa) {
    bool all = true;
#pragma unroll
    for (int p = 0; p < SEGP; ++p) all = all && (((live >> p) & 1u) == 0u || (cc[p] & sa) != 0u);
    return all;
}

// 4 bits -> 4 bytes of 0/1.
__device__ __forceinline__ uint32_t expand4(uint32_t bits) { return (bits * 0x00204081u) & 0x01010101u; }

// ---------------------------------------------------------------------------
// Wider near windows (the window-width study of the match-search section:
// 48 and 64 elements). Offsets 33..64 get a second set of masks over the same
// positions: m[p] bit o-1 set iff element (base+p) equals element
// (base+p-32-o), 1 <= o <= 32, base+p-32-o >= 0, then ANDed with `far_mask`
// (the offsets 33..window). The longest run over 1..window is the longer of
// the two passes' runs, the first pass winning ties (its offsets are nearer).
// ---------------------------------------------------------------------------
template <int WS>
__device__ __forceinline__ void load4(const uint8_t* s_el, int i0, uint32_t (&w)[4]) {
    w[0] = w[1] = w[2] = w[3] = 0u;
    if (i0 < 0) return;
    const uint8_t* p = s_el + el_addr<WS>((uint32_t)i0);
    if (WS == 4) {
        const uint4 t = *reinterpret_cast<const uint4*>(p);
        w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
    } else if (WS == 2) {
        const uint2 t = *reinterpret_cast<const uint2*>(p);
        w[0] = t.x & 0xFFFFu; w[1] = t.x >> 16; w[2] = t.y & 0xFFFFu; w[3] = t.y >> 16;
    } else {
        const uint32_t t = *reinterpret_cast<const uint32_t*>(p);
        w[0] = t & 0xFFu; w[1] = (t >> 8) & 0xFFu; w[2] = (t >> 16) & 0xFFu; w[3] = t >> 24;
    }
}

template <int WS, int SEGP>
__device__ __forceinline__ void near_masks_far(const uint8_t* s_el, uint32_t base, uint32_t far_mask,
                                               uint32_t (&m)[SEGP]) {
#pragma unroll
    for (int h = 0; h < SEGP / 8; ++h) {
        // elements base+8h-64 .. base+8h-25: the far windows of eight positions
        const int first = (int)base + 8 * h - 64;  // a multiple of 4
        uint32_t v[40];
#pragma unroll
        for (int q = 0; q < 10; ++q) {
            uint32_t w[4];
            load4<WS>(s_el, first + 4 * q, w);
#pragma unroll
            for (int r = 0; r < 4; ++r) v[4 * q + r] = w[r];
        }
#pragma unroll
        for (int p = 0; p < 8; ++p) {
            const uint32_t i = base + (uint32_t)(8 * h + p);
            const uint32_t x = el_get<WS>(s_el, i);
            uint32_t mm = 0;
#pragma unroll
            for (int o = 1; o <= 32; ++o) or_if_equal(mm, v[p + 32 - o], x, 1u << (o - 1));
            if (i < 64u) mm &= i > 32u ? (1u << (i - 32u)) - 1u : 0u;
            m[8 * h + p] = mm & far_mask;
        }
    }
}

// The AND-chain longest match of E4 for one set of masks: per position of the
// segment (run length | (offset_base + nearest offset) << 8), two per word.
// Same steps as the kernel's own E4 (register triangle, lockstep continuation
// with whole-segment skips); used by the far pass.
template <int SEGP>
__device__ __forceinline__ void and_chains(const uint32_t (&m)[SEGP], const uint32_t* s_om,
                                           const uint32_t* s_sa, uint32_t seg_a, uint32_t E,
                                           uint32_t off_base, uint32_t (&lw)[SEGP / 2]) {
    uint32_t cc[SEGP], cl[SEGP];  // running AND (0 once dead), last nonzero value
    uint32_t A = 0;
#pragma unroll
    for (int p = 0; p < SEGP; ++p) {
        cc[p] = m[p];
        cl[p] = m[p];
        or_if_nonzero(A, m[p], 1u << p);
    }
    uint32_t lb[SEGP / 4];
#pragma unroll
    for (int w = 0; w < SEGP / 4; ++w) lb[w] = expand4((A >> (4 * w)) & 15u);
    uint32_t P = A & (1u << (SEGP - 1));
#pragma unroll
    for (int k = 1; k < SEGP; ++k) {
        const uint32_t act = A & ((1u << (SEGP - k)) - 1u);
        if (!__any_sync(FULL, act != 0u)) break;
        uint32_t An = 0;
#pragma unroll
        for (int p = 0; p + k < SEGP; ++p) {
            chain_step(cc[p], cl[p], An, m[p + k], 1u << p);
        }
#pragma unroll
        for (int w = 0; w < SEGP / 4; ++w) lb[w] += expand4((An >> (4 * w)) & 15u);
        P |= An & (1u << (SEGP - 1 - k));
        A = An;
    }
    if (P) {
        uint32_t A2 = P;
        uint32_t st = 0;
        while (A2 != 0u && seg_a + (uint32_t)SEGP + st < E) {
            const uint32_t q0 = seg_a + (uint32_t)SEGP + st;
            if (A2 == (1u << SEGP) - 1u || st >= (uint32_t)SEGP) {
                const uint32_t j = q0 / (uint32_t)SEGP;
                const uint32_t p0 = (uint32_t)__ffs(A2) - 1u;
                const uint32_t room = (uint32_t)kMaxLen - (SEGP - p0 + st);
                uint32_t take = 0, sa = 0;
                if (room > 4u * SEGP && q0 + 4u * SEGP <= E) {
                    sa = s_sa[j] & s_sa[j + 1] & s_sa[j + 2] & s_sa[j + 3];
                    if (chains_live<SEGP>(cc, A2, sa)) take = 4u * SEGP;
                }
                if (!take && room > (uint32_t)SEGP) {
                    sa = s_sa[j];
                    if (chains_live<SEGP>(cc, A2, sa)) take = SEGP;
                }
                if (take) {
#pragma unroll
                    for (int p = 0; p < SEGP; ++p) {
                        cc[p] &= sa;  // dead chains stay 0
                        if ((A2 >> p) & 1u) cl[p] = cc[p];
                    }
#pragma unroll
                    for (int w = 0; w < SEGP / 4; ++w) lb[w] += take * expand4((A2 >> (4 * w)) & 15u);
                    st += take;
                    continue;
                }
            }
            const uint32_t* omq = s_om + om_idx(q0);  // one 16-mask block
            for (int k = 0; k < SEGP && A2 != 0u; ++k, ++st) {
                const uint32_t om = omq[k];
                uint32_t An = 0;
#pragma unroll
                for (int p = 0; p < SEGP; ++p) {
                    chain_step(cc[p], cl[p], An, om, 1u << p);
                }
#pragma unroll
                for (int w = 0; w < SEGP / 4; ++w) lb[w] += expand4((An >> (4 * w)) & 15u);
                const int over = (int)(SEGP + st + 1u) - kMaxLen;
                if (over >= 0) {
                    const int lim = over < SEGP - 1 ? over : SEGP - 1;
                    An &= ~((2u << lim) - 1u);
#pragma unroll
                    for (int p = 0; p < SEGP; ++p)
                        if (p <= lim) cc[p] = 0;  // capped chains end here
                }
                A2 = An;
            }
        }
    }
#pragma unroll
    for (int p = 0; p < SEGP; p += 2) {
        const uint32_t l0 = (lb[p >> 2] >> (8 * (p & 3))) & 0xFFu;
        const uint32_t l1 = (lb[p >> 2] >> (8 * ((p + 1) & 3))) & 0xFFu;
        const uint32_t lo0 = l0 ? (l0 | ((off_base + (uint32_t)__ffs(cl[p])) << 8)) : 0u;
        const uint32_t lo1 = l1 ? (l1 | ((off_base + (uint32_t)__ffs(cl[p + 1])) << 8)) : 0u;
        lw[p >> 1] = lo0 | (lo1 << 16);
    }
}

// Per 16-bit half (length | offset << 8): the second value where its length
// is strictly longer.
__device__ __forceinline__ uint32_t longer_halves(uint32_t a, uint32_t b) {
    const uint32_t lo = (b & 0xFFu) > (a & 0xFFu) ? (b & 0xFFFFu) : (a & 0xFFFFu);
    const uint32_t hi = ((b >> 16) & 0xFFu) > ((a >> 16) & 0xFFu) ? (b >> 16) : (a >> 16);
    return lo | (hi << 16);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int WS, int LEVEL, int SEGP, bool SINGLE, int NEARW = 32>
__global__ void __launch_bounds__(256, 4) encode_kernel(EncodeArgs a) {
    static_assert(NEARW == 32 || (NEARW == 64 && LEVEL == 0 && !SINGLE),
                  "wider near windows are a two-pass, level-0 option");
    extern __shared__ __align__(16) uint8_t smem[];
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    const uint32_t CS = a.chunk_size;
    const uint32_t E = a.elems;
    const EncLayout L = enc_layout(CS, E, LEVEL);
    uint8_t* s_el = smem + L.el;
    uint32_t* s_om = reinterpret_cast<uint32_t*>(smem + L.om);
    uint16_t* s_lo = reinterpret_cast<uint16_t*>(smem + L.lo);
    uint32_t* s_sa = reinterpret_cast<uint32_t*>(smem + L.sa);
    uint32_t* s_tab = reinterpret_cast<uint32_t*>(smem + L.tab);
    uint32_t* s_fl = reinterpret_cast<uint32_t*>(smem + L.fl);
    uint8_t* s_data = smem + L.data;
    uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + L.misc);
    constexpr uint32_t LMIN = (uint32_t)min_match_len(WS);
    constexpr uint32_t NONE = 0xFFFFFFFFu;

    if (!SINGLE) pdl_trigger();  // the pack pass may be scheduled as CTAs retire
    if (a.n_chunks == 0) {
        if (blockIdx.x == 0 && tid == 0) write_header(a, WS, kHeaderBytes);
        return;
    }
    const uint64_t body0 = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * a.n_chunks;
    const bool in_aligned = (reinterpret_cast<uintptr_t>(a.in) & 15u) == 0;
    const uint32_t seg_a = (uint32_t)tid * SEGP;  // this thread's positions [seg_a, seg_a + SEGP)

    // The chunk staged in s_fl/s_data whose offset is not known yet. Its
    // look-back runs after the next chunk's match search, by which time its
    // predecessors have published their sizes, so the wait is normally empty.
    uint32_t p_c = NONE, p_blk = 0, p_entry = 0, p_dbytes = 0, p_fw = 0, p_dw = 0;

    // Level-1 bucket entries are (tag << 16) | (position + 1), the tag counting
    // this CTA's chunks: an entry left by an earlier chunk has a smaller tag,
    // so it loses every atomicMax and reads as empty, and the table is cleared
    // only here (visible after the barrier that follows the first ticket) and
    // when the 16-bit tag wraps.
    uint32_t tag = 0;
    if (LEVEL) {
        for (uint32_t k = tid; k < 2u * E; k += nthreads) s_tab[k] = 0;
    }

    for (;;) {
        if (tid == 0) s_misc[0] = atomicAdd(a.ticket, 1u);
        __syncthreads();
        const uint32_t t = s_misc[0];
        const bool have = t < a.n_chunks;
        // Single pass: chunks in ticket order (the look-back needs it). Two
        // pass: the zero-padded tail chunk first, as it is often the slowest.
        const uint32_t c = (SINGLE || !have) ? t : (t == 0 ? a.n_chunks - 1u : t - 1u);

        bool nonzero = false;
        uint32_t items = 0, dbytes = 0, blk = 0, entry_items = 0, n_match = 0;
        uint32_t path = 0, mmask = 0, item_base = 0, match_base = 0;
        if (have) {
            // ---- E1: load the chunk (zero padded) ----
            const uint64_t begin = (uint64_t)c * CS;
            const uint64_t avail = a.n_bytes - begin;
            const uint32_t take = avail < CS ? (uint32_t)avail : CS;
            uint32_t nz = 0;
            if (in_aligned && take == CS) {
                const uint4* src = reinterpret_cast<const uint4*>(a.in + begin);
                for (uint32_t g = tid; g < CS / 16u; g += nthreads) {
                    const uint4 v = __ldg(src + g);
                    // 16 chunk bytes stay 16-byte aligned in the padded array
                    *reinterpret_cast<uint4*>(s_el + chunk_byte_addr<WS>(16u * g)) = v;
                    if (LEVEL && !SINGLE) reinterpret_cast<uint4*>(s_data)[g] = v;
                    nz |= v.x | v.y | v.z | v.w;
                }
            } else {
                for (uint32_t b4 = tid; b4 < CS / 4u; b4 += nthreads) {
                    uint32_t v = 0;
                    for (uint32_t k = 0; k < 4u; ++k) {
                        const uint32_t b = 4u * b4 + k;
                        if (b < take) v |= (uint32_t)a.in[begin + b] << (8u * k);
                    }
                    *reinterpret_cast<uint32_t*>(s_el + chunk_byte_addr<WS>(4u * b4)) = v;
                    if (LEVEL && !SINGLE) reinterpret_cast<uint32_t*>(s_data)[b4] = v;
                    nz |= v;
                }
            }
            if (LEVEL) {
                if (++tag == 0x10000u) {
                    for (uint32_t k = tid; k < 2u * E; k += nthreads) s_tab[k] = 0;
                    tag = 1;
                }
            }
            // ---- E2: zero test ----
            nonzero = __syncthreads_or(nz != 0) != 0;

            if (nonzero) {
                // ---- E3: near equality masks of this thread's segment ----
                uint32_t m[SEGP];
                near_masks<WS, SEGP>(s_el, seg_a, m);
                {
                    uint4* dst = reinterpret_cast<uint4*>(s_om + om_idx(seg_a));
                    uint32_t sa = m[0];
#pragma unroll
                    for (int q = 0; q < SEGP / 4; ++q) {
                        dst[q] = make_uint4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
                        sa &= m[4 * q] & m[4 * q + 1] & m[4 * q + 2] & m[4 * q + 3];
                    }
                    s_sa[tid] = sa;  // the offsets that match at every position of the segment
                }
                __syncthreads();

                // ---- E4: AND-chain longest match, nearest offset ----
                // The chains of the segment's positions advance together in
                // registers; one that is still alive at the segment end is
                // finished from the shared-memory masks.
                {
                    // cc[p]: chain p's running AND, 0 once it died; cl[p]: its
                    // last nonzero value (the nearest offset is its lowest bit)
                    uint32_t cc[SEGP], cl[SEGP];
                    uint32_t A = 0;
#pragma unroll
                    for (int p = 0; p < SEGP; ++p) {
                        cc[p] = m[p];
                        cl[p] = m[p];
                        or_if_nonzero(A, m[p], 1u << p);
                    }
                    uint32_t lb[SEGP / 4];
#pragma unroll
                    for (int w = 0; w < SEGP / 4; ++w) lb[w] = expand4((A >> (4 * w)) & 15u);
                    uint32_t P = A & (1u << (SEGP - 1));
#pragma unroll
                    for (int k = 1; k < SEGP; ++k) {
                        const uint32_t act = A & ((1u << (SEGP - k)) - 1u);
                        if (!__any_sync(FULL, act != 0u)) break;
                        uint32_t An = 0;
#pragma unroll
                        for (int p = 0; p + k < SEGP; ++p) {
                            chain_step(cc[p], cl[p], An, m[p + k], 1u << p);
                        }
#pragma unroll
                        for (int w = 0; w < SEGP / 4; ++w) lb[w] += expand4((An >> (4 * w)) & 15u);
                        P |= An & (1u << (SEGP - 1 - k));
                        A = An;
                    }
                    // Chains still alive at the segment end continue over the
                    // following positions' masks in lockstep: one shared-memory
                    // load per step serves all of them, so a long run costs
                    // O(run) loads rather than O(run^2). Once the chains look
                    // long (all of them alive, or a whole segment survived),
                    // four following segments, else one, are taken in one step
                    // when the AND of their masks keeps every live chain nonzero
                    // and no chain reaches the length cap in them, so a run of
                    // one repeated word costs a few steps per thread; otherwise
                    // (and for the last steps before the cap) the segment goes
                    // position by position.
                    if (P) {
                        uint32_t A2 = P;
                        uint32_t st = 0;  // positions taken past the segment end
                        while (A2 != 0u && seg_a + (uint32_t)SEGP + st < E) {
                            const uint32_t q0 = seg_a + (uint32_t)SEGP + st;  // a segment start
                            if (A2 == (1u << SEGP) - 1u || st >= (uint32_t)SEGP) {
                                const uint32_t j = q0 / (uint32_t)SEGP;
                                const uint32_t p0 = (uint32_t)__ffs(A2) - 1u;        // longest live chain
                                const uint32_t room = (uint32_t)kMaxLen - (SEGP - p0 + st);  // steps until p0 is capped
                                uint32_t take = 0, sa = 0;
                                if (room > 4u * SEGP && q0 + 4u * SEGP <= E) {
                                    sa = s_sa[j] & s_sa[j + 1] & s_sa[j + 2] & s_sa[j + 3];
                                    if (chains_live<SEGP>(cc, A2, sa)) take = 4u * SEGP;
                                }
                                if (!take && room > (uint32_t)SEGP) {
                                    sa = s_sa[j];
                                    if (chains_live<SEGP>(cc, A2, sa)) take = SEGP;
                                }
                                if (take) {
#pragma unroll
                                    for (int p = 0; p < SEGP; ++p) {
                                        cc[p] &= sa;  // dead chains stay 0
                                        if ((A2 >> p) & 1u) cl[p] = cc[p];
                                    }
#pragma unroll
                                    for (int w = 0; w < SEGP / 4; ++w)
                                        lb[w] += take * expand4((A2 >> (4 * w)) & 15u);
                                    st += take;
                                    continue;
                                }
                            }
                            // the segment's masks are contiguous (one 16-mask block)
                            const uint32_t* omq = s_om + om_idx(q0);
                            for (int k = 0; k < SEGP && A2 != 0u; ++k, ++st) {
                                const uint32_t om = omq[k];
                                uint32_t An = 0;
#pragma unroll
                                for (int p = 0; p < SEGP; ++p) chain_step(cc[p], cl[p], An, om, 1u << p);
#pragma unroll
                                for (int w = 0; w < SEGP / 4; ++w) lb[w] += expand4((An >> (4 * w)) & 15u);
                                // length of chain p is now SEGP - p + st + 1: stop at the cap
                                const int over = (int)(SEGP + st + 1u) - kMaxLen;
                                if (over >= 0) {
                                    const int lim = over < SEGP - 1 ? over : SEGP - 1;
                                    An &= ~((2u << lim) - 1u);
#pragma unroll
                                    for (int p = 0; p < SEGP; ++p)
                                        if (p <= lim) cc[p] = 0;  // capped chains end here
                                }
                                A2 = An;
                            }
                        }
                    }
                    uint32_t lw[SEGP / 2];
#pragma unroll
                    for (int p = 0; p < SEGP; p += 2) {
                        const uint32_t l0 = (lb[p >> 2] >> (8 * (p & 3))) & 0xFFu;
                        const uint32_t l1 = (lb[p >> 2] >> (8 * ((p + 1) & 3))) & 0xFFu;
                        // cl[p] is 0 exactly when the length is 0 (no offset matched)
                        const uint32_t lo0 = l0 | ((uint32_t)__ffs(cl[p]) << 8);
                        const uint32_t lo1 = l1 | ((uint32_t)__ffs(cl[p + 1]) << 8);
                        lw[p >> 1] = lo0 | (lo1 << 16);
                    }
                    uint4* dlo = reinterpret_cast<uint4*>(s_lo + seg_a);
#pragma unroll
                    for (int q = 0; q < SEGP / 8; ++q)
                        dlo[q] = make_uint4(lw[4 * q], lw[4 * q + 1], lw[4 * q + 2], lw[4 * q + 3]);
                }
                if constexpr (NEARW > 32) __syncthreads();  // the far pass reuses the masks' area

                // ---- E4b (near windows wider than 32): offsets 33..window ----
                // A second set of masks over the same positions replaces the
                // first (dead once E4 is done); a far run replaces the near
                // one only when it is strictly longer.
                if constexpr (NEARW > 32) {
                    uint32_t m2[SEGP];
                    near_masks_far<WS, SEGP>(s_el, seg_a, a.far_mask, m2);
                    {
                        uint4* dst = reinterpret_cast<uint4*>(s_om + om_idx(seg_a));
                        uint32_t sa = m2[0];
#pragma unroll
                        for (int q = 0; q < SEGP / 4; ++q) {
                            dst[q] = make_uint4(m2[4 * q], m2[4 * q + 1], m2[4 * q + 2], m2[4 * q + 3]);
                            sa &= m2[4 * q] & m2[4 * q + 1] & m2[4 * q + 2] & m2[4 * q + 3];
                        }
                        s_sa[tid] = sa;
                    }
                    __syncthreads();
                    uint32_t lw2[SEGP / 2];
                    and_chains<SEGP>(m2, s_om, s_sa, seg_a, E, 32u, lw2);
                    uint4* dlo = reinterpret_cast<uint4*>(s_lo + seg_a);
#pragma unroll
                    for (int q = 0; q < SEGP / 8; ++q) {
                        const uint4 o = dlo[q];
                        dlo[q] = make_uint4(longer_halves(o.x, lw2[4 * q]), longer_halves(o.y, lw2[4 * q + 1]),
                                            longer_halves(o.z, lw2[4 * q + 2]), longer_halves(o.w, lw2[4 * q + 3]));
                    }
                    __syncthreads();
                }

                // ---- E5: level-1 hashed candidates over 8 sub-blocks ----
                // The sub-block phases only look the buckets up and insert;
                // the candidates are checked afterwards, with no barrier in
                // between. Thread tid owns position s*SB + r*nthreads + tid of
                // each sub-block s (r < R = SEGP/8, so SB = R*nthreads); the
                // bucket and candidate offset of an owned position stay in its
                // registers. Sub-block 0 finds an empty table and the last
                // sub-block's inserts are never looked up, so neither is done.
                // A candidate at offset d <= 32 never wins: the near search
                // already found the longest run over offsets 1..32 with the
                // same caps, nearest first. For d > 32 it wins only with a run
                // longer than the near length l0. In the two-pass kernel the
                // staging buffer is idle until E7 and holds an unpadded copy of
                // the chunk (written in E1) for the hashing and the compares.
                if (LEVEL) {
                    constexpr int R = SEGP / 8;
                    constexpr int NP = kSubBlocks * R;
                    const uint32_t SB = E / kSubBlocks;
                    uint32_t cd[NP / 4];  // candidate offset of owned position j in byte j
#pragma unroll
                    for (int w = 0; w < NP / 4; ++w) cd[w] = 0;
                    uint32_t cm = 0;      // owned positions with a candidate
#pragma unroll
                    for (int s = 0; s < kSubBlocks; ++s) {
                        // only the chunk's last position (the last sub-block's last
                        // owned position of the last thread) has no two-word key
                        uint32_t hk[R];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint32_t i = (uint32_t)s * SB + (uint32_t)r * (uint32_t)nthreads + (uint32_t)tid;
                            const bool key = (s + 1 < kSubBlocks || r + 1 < R) || (uint32_t)tid + 1u < (uint32_t)nthreads;
                            const uint32_t i1 = key ? i + 1u : i;
                            hk[r] = SINGLE ? key_hash(el_get<WS>(s_el, i), el_get<WS>(s_el, i1), a.hash_bits)
                                           : key_hash(lin_get<WS>(s_data, i), lin_get<WS>(s_data, i1), a.hash_bits);
                        }
                        if (s > 0) {
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const int j = s * R + r;
                                const uint32_t i = (uint32_t)s * SB + (uint32_t)r * (uint32_t)nthreads + (uint32_t)tid;
                                const bool key = (s + 1 < kSubBlocks || r + 1 < R) || (uint32_t)tid + 1u < (uint32_t)nthreads;
                                const uint32_t slot = s_tab[hk[r]];
                                const uint32_t d = i + 1u - (slot & 0xFFFFu);  // i - p for p = slot - 1
                                // this chunk's entry (tag), 32 < d <= kMaxOff, a key at i
                                const bool ok = ((slot ^ (tag << 16)) < 0x10000u) &
                                                (d - 33u < (uint32_t)(kMaxOff - 32)) & key;
                                if (ok) {
                                    cd[j >> 2] |= d << (8 * (j & 3));
                                    cm |= 1u << j;
                                }
                            }
                            if (s + 1 < kSubBlocks) __syncthreads();  // lookups before this sub-block's inserts
                        }
                        if (s + 1 < kSubBlocks) {
#pragma unroll
                            for (int r = 0; r < R; ++r) {
                                const uint32_t i = (uint32_t)s * SB + (uint32_t)r * (uint32_t)nthreads + (uint32_t)tid;
                                atomicMax(&s_tab[hk[r]], (tag << 16) | (i + 1u));  // s < 7: every position has a key
                            }
                            __syncthreads();  // inserts before the next sub-block's lookups
                        }
                    }
                    while (cm) {
                        const uint32_t j = (uint32_t)__ffs(cm) - 1u;
                        cm &= cm - 1u;
                        uint32_t dw = cd[0];
#pragma unroll
                        for (int w = 1; w < NP / 4; ++w) dw = (j >> 2) == (uint32_t)w ? cd[w] : dw;
                        const uint32_t d = (dw >> (8u * (j & 3u))) & 0xFFu;
                        const uint32_t i = (j / (uint32_t)R) * SB + (j % (uint32_t)R) * (uint32_t)nthreads + (uint32_t)tid;
                        const uint32_t cap = E - i < (uint32_t)kMaxLen ? E - i : (uint32_t)kMaxLen;
                        const uint32_t l0 = s_lo[i] & 0xFFu;
                        if (l0 >= cap) continue;
                        uint32_t k = 0;
                        if constexpr (!SINGLE) {
                            // run length from 0, four element pairs per round,
                            // from the unpadded copy in the staging buffer:
                            // reads past the cap (at most 3 elements past the
                            // chunk, inside the buffer's 16 spare bytes) can only
                            // lengthen the run, which the cap then cuts
                            const uint8_t* pa = s_data + i * WS;
                            const uint8_t* pb = pa - d * WS;
                            for (;;) {
                                uint32_t eq = 0;
#pragma unroll
                                for (int r = 0; r < 4; ++r)
                                    or_if_equal(eq, lin_at<WS>(pa, k + (uint32_t)r), lin_at<WS>(pb, k + (uint32_t)r), 1u << r);
                                const uint32_t lead = (uint32_t)__ffs(~eq) - 1u;  // 0..4
                                k += lead;
                                if (lead < 4u || k >= cap) break;
                            }
                        } else {
                            // the staging buffer holds the previous chunk's block
                            // here: compare in the padded element array
                            const uint32_t p = i - d;
                            if (el_get<WS>(s_el, i + l0) != el_get<WS>(s_el, p + l0)) continue;
                            for (;;) {
                                uint32_t eq = 0;
#pragma unroll
                                for (int r = 0; r < 4; ++r) {
                                    const uint32_t q = k + (uint32_t)r < cap ? k + (uint32_t)r : cap - 1u;
                                    eq |= (uint32_t)(el_get<WS>(s_el, i + q) == el_get<WS>(s_el, p + q)) << r;
                                }
                                const uint32_t lead = (uint32_t)__ffs(~eq) - 1u;  // 0..4
                                k += lead;
                                if (lead < 4u || k >= cap) break;
                            }
                        }
                        if (k > cap) k = cap;
                        if (k > l0) s_lo[i] = (uint16_t)(k | (d << 8));
                    }
                    __syncthreads();
                }

                // ---- E6: greedy parse, one SEGP-position segment per thread ----
                // Each thread walks its segment from the segment start using its
                // step bytes held in registers; then every thread whose true
                // entry (the previous segment's exit) differs from the entry its
                // path assumed re-walks from it, keeping its old path from the
                // first common position on. This repeats until a round changes no
                // exit (then the next round would read the same entries: every
                // entry equals the exit before it, which only the sequential
                // parse satisfies; most chunks stop after one round).
                // A frontier speeds up long matches: the last thread whose entry
                // is known exact (thread 0 from the start) and its exit. Every
                // thread after it whose segment starts at or before that exit
                // takes the exit as its entry at once (the threads it jumps
                // over pass it through), so a match spanning many segments costs
                // one round, not one per segment. It starts in the third round.
                // A thread it reaches takes the frontier exit, which in a round
                // that changes no exit equals the exit before it, so the
                // stopping rule is unchanged.
                uint32_t T[4] = {0u, 0u, 0u, 0u};  // step of each position, one byte each
                {
                    uint32_t lw[8];
                    const uint4* q = reinterpret_cast<const uint4*>(s_lo + seg_a);
                    const uint4 v0 = q[0];
                    lw[0] = v0.x; lw[1] = v0.y; lw[2] = v0.z; lw[3] = v0.w;
                    if (SEGP == 16) {
                        const uint4 v1 = q[1];
                        lw[4] = v1.x; lw[5] = v1.y; lw[6] = v1.z; lw[7] = v1.w;
                    } else {
                        lw[4] = lw[5] = lw[6] = lw[7] = 0u;
                    }
                    if (WS != 1) {
                        // four lengths per word (one byte permute); a byte below
                        // LMIN (0, or 1 for word size 2) is a literal: step 1
#pragma unroll
                        for (int w = 0; w < SEGP / 4; ++w) {
                            const uint32_t t = __byte_perm(lw[2 * w], lw[2 * w + 1], 0x6420u);
                            const uint32_t u = WS == 2 ? (t & 0xFEFEFEFEu) : t;
                            // 0x80 in each byte of u that is zero
                            const uint32_t z = ~(((u & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | u | 0x7F7F7F7Fu);
                            T[w] = t | (z >> 7);
                            const uint32_t mt = ((~z >> 7) & 0x01010101u) * 0x01020408u >> 24;  // 4 bits
                            mmask |= mt << (4 * w);
                        }
                    } else {
                        // bytes (LMIN 3): 0x80 where a length is >= 3 (bit 7 of
                        // (len | 0x80) - 3, or of len itself), then step = len
                        // there and 1 elsewhere
                        static_assert(WS != 1 || LMIN == 3u, "byte lengths below 3 are literals");
#pragma unroll
                        for (int w = 0; w < SEGP / 4; ++w) {
                            const uint32_t t = __byte_perm(lw[2 * w], lw[2 * w + 1], 0x6420u);
                            const uint32_t f = (((t | 0x80808080u) - 0x03030303u) | t) & 0x80808080u;
                            const uint32_t keep = (f >> 7) * 0xFFu;
                            T[w] = (t & keep) | (~keep & 0x01010101u);
                            mmask |= ((((f >> 7) & 0x01010101u) * 0x01020408u) >> 24) << (4 * w);
                        }
                    }
                }
                uint32_t cur_e = 0, exit_abs;
                {
                    uint32_t p = 0;
                    while (p < (uint32_t)SEGP) {
                        path |= 1u << p;
                        p += seg_step(T, p);
                    }
                    exit_abs = seg_a + p;
                }
                if (tid == 0) s_misc[24] = exit_abs;  // frontier: thread 0, its exit
                for (uint32_t rnd = 0;; ++rnd) {
                    const uint32_t exit_before = exit_abs;
                    uint32_t prev = __shfl_up_sync(FULL, exit_abs, 1);
                    if (lane == 31) s_misc[8 + warp] = exit_abs;
                    __syncthreads();
                    if (lane == 0) prev = warp == 0 ? 0u : s_misc[8 + warp - 1];
                    const bool use_fr = rnd >= 2u;
                    const uint32_t fb = rnd & 1u;
                    uint32_t fr = 0, fx = 0;
                    bool reached = false;
                    if (use_fr) {
                        fr = s_misc[24 + fb];
                        fx = fr & 0xFFFFu;
                        reached = (uint32_t)tid > (fr >> 16) && seg_a <= fx;
                        if (reached) prev = fx;
                    }
                    const uint32_t te = prev - seg_a;  // true entry, relative
                    const bool changed = te != cur_e;
                    if (changed) {
                        if (te >= (uint32_t)SEGP) {
                            path = 0;
                            exit_abs = prev;
                        } else {
                            const uint32_t old = path & ~((1u << te) - 1u);
                            uint32_t np = 0, p = te;
                            bool merged = false;
                            while (p < (uint32_t)SEGP) {
                                if ((old >> p) & 1u) {
                                    merged = true;
                                    break;
                                }
                                np |= 1u << p;
                                p += seg_step(T, p);
                            }
                            if (merged) {
                                path = np | (old & ~((1u << p) - 1u));
                            } else {
                                path = np;
                                exit_abs = seg_a + p;
                            }
                        }
                        cur_e = te;
                    }
                    // the thread whose segment holds the frontier exit now has
                    // an exact entry and becomes the next frontier
                    if (use_fr) {
                        if (reached && fx < seg_a + (uint32_t)SEGP)
                            s_misc[25 - fb] = ((uint32_t)tid << 16) | exit_abs;
                        else if (tid == 0 && fx >= E)
                            s_misc[25 - fb] = fr;
                    }
                    if (!__syncthreads_or(exit_abs != exit_before)) break;
                }

                // ---- E7 (sizes): team scan of item and match counts ----
                {
                    const uint32_t x =
                        (uint32_t)__popc(path) | ((uint32_t)__popc(path & mmask) << 16);
                    uint32_t incl = x;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t t = __shfl_up_sync(FULL, incl, o);
                        if (lane >= o) incl += t;
                    }
                    if (lane == 31) s_misc[16 + warp] = incl;
                    __syncthreads();
                    uint32_t wbase = 0, total = 0;
                    for (int w = 0; w < nwarps; ++w) {
                        const uint32_t v = s_misc[16 + w];
                        if (w < warp) wbase += v;
                        total += v;
                    }
                    const uint32_t excl = wbase + incl - x;
                    item_base = excl & 0xFFFFu;
                    match_base = excl >> 16;
                    items = total & 0xFFFFu;
                    n_match = total >> 16;
                    dbytes = WS * (items - n_match) + 2u * n_match;
                }
                // ---- E8: raw fallback ----
                blk = 4u * ((items + 31u) / 32u) + ((dbytes + 3u) & ~3u);
                if (blk >= CS) {
                    blk = CS;
                    entry_items = kRawBit;
                    dbytes = CS;
                } else {
                    entry_items = items;
                }
            }
            // publish this chunk's size now, so successors' look-backs resolve early
            if (SINGLE && tid == 0) publish_size(a, c, blk);
        }

        // ---- E9 + E10 for the pending chunk: offset, store-out, table, header ----
        if (SINGLE && p_c != NONE) {
            if (warp == 0) {
                bool to = false;
                const uint64_t prefix = p_c == 0 ? 0ull : lookback(a.desc, p_c, p_blk, a.epoch, lane, &to);
                if (lane == 0) {
                    if (to) atomicOr(a.status, kStatTimeout);
                    s_misc[40] = (uint32_t)prefix;
                    s_misc[41] = (uint32_t)(prefix >> 32);
                }
            }
            __syncthreads();
            const uint64_t prefix = (uint64_t)s_misc[40] | ((uint64_t)s_misc[41] << 32);
            const uint64_t dst = body0 + prefix;
            for (uint32_t j = tid; j < p_fw + p_dw; j += nthreads) {
                const uint32_t v = j < p_fw ? s_fl[j]
                                            : *reinterpret_cast<const uint32_t*>(s_data + 4u * (j - p_fw));
                store_u32_capped(a.out, dst + 4ull * j, v, a.capacity);
            }
            if (tid == 0) {
                const uint64_t eo = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * p_c;
                store_u32_capped(a.out, eo, p_entry, a.capacity);
                store_u32_capped(a.out, eo + 4, p_dbytes, a.capacity);
                if (p_c == a.n_chunks - 1u) write_header(a, WS, dst + p_blk);
            }
            __syncthreads();  // staging is free again
        }
        if (!have) break;

        // ---- E7: stage this chunk's block ----
        uint32_t fw = 0, dw = 0;
        if (nonzero) {
            if (entry_items == kRawBit) {
                dw = CS / 4u;
                for (uint32_t j = tid; j < dw; j += nthreads)
                    *reinterpret_cast<uint32_t*>(s_data + 4u * j) =
                        *reinterpret_cast<const uint32_t*>(s_el + chunk_byte_addr<WS>(4u * j));
            } else {
                fw = (items + 31u) / 32u;
                dw = (dbytes + 3u) / 4u;
                for (uint32_t k = tid; k < fw; k += nthreads) s_fl[k] = 0;
                __syncthreads();
                uint32_t bb = WS * (item_base - match_base) + 2u * match_base;
                if (a.split) {
                    // split mode: the chunk's literals, then its lengths, then its
                    // offsets, each in item order (the same bytes, regrouped)
                    const uint32_t lit_bytes = WS * (items - n_match);
                    uint32_t li = WS * (item_base - match_base), mi = match_base;
                    uint32_t fbits = 0, k = 0, rem = path;
                    while (rem) {
                        const uint32_t p = (uint32_t)__ffs(rem) - 1u;
                        rem &= rem - 1u;
                        const uint32_t pos = seg_a + p;
                        if ((mmask >> p) & 1u) {
                            const uint32_t lo = s_lo[pos];
                            s_data[lit_bytes + mi] = (uint8_t)lo;
                            s_data[lit_bytes + n_match + mi] = (uint8_t)(lo >> 8);
                            ++mi;
                            fbits |= 1u << k;
                        } else {
                            const uint32_t v = el_get<WS>(s_el, pos);
                            if (WS == 1) s_data[li] = (uint8_t)v;
                            else if (WS == 2) *reinterpret_cast<uint16_t*>(s_data + li) = (uint16_t)v;
                            else *reinterpret_cast<uint32_t*>(s_data + li) = v;
                            li += WS;
                        }
                        ++k;
                    }
                    if (fbits) or_bits(s_fl, item_base, fbits);
                    if (tid == 0)
                        for (uint32_t z = dbytes; z < ((dbytes + 3u) & ~3u); ++z) s_data[z] = 0;
                }
                if (!a.split) {
                    // the segment's tokens and elements in registers (vector
                    // loads), then its items written position by position
                    // (predicated, no loop over a data-dependent count)
                    uint32_t lo[SEGP / 2];
                    {
                        const uint4* q = reinterpret_cast<const uint4*>(s_lo + seg_a);
#pragma unroll
                        for (int h = 0; h < SEGP / 8; ++h) {
                            const uint4 v = q[h];
                            lo[4 * h] = v.x; lo[4 * h + 1] = v.y; lo[4 * h + 2] = v.z; lo[4 * h + 3] = v.w;
                        }
                    }
                    constexpr int NW = SEGP * WS / 4;  // words holding the segment's elements
                    uint32_t ew[NW];
                    {
                        const uint8_t* e0 = s_el + el_addr<WS>(seg_a);
                        if (NW >= 4) {
#pragma unroll
                            for (int h = 0; h < NW / 4; ++h) {
                                const uint4 v = reinterpret_cast<const uint4*>(e0)[h];
                                ew[4 * h] = v.x; ew[4 * h + 1] = v.y; ew[4 * h + 2] = v.z; ew[4 * h + 3] = v.w;
                            }
                        } else {
                            const uint2 v = *reinterpret_cast<const uint2*>(e0);
                            ew[0] = v.x; ew[NW - 1] = v.y;
                        }
                    }
                    uint32_t fbits = 0, k = 0;
                    if (WS == 1) {
                        // bytes: predicated stores and arithmetic offsets, no
                        // branch per position (+3 % on the byte stream; the
                        // wider words keep the branches, measured 0.4 % faster)
#pragma unroll
                        for (int p = 0; p < SEGP; ++p) {
                            const uint32_t on = (path >> p) & 1u;
                            const uint32_t ism = (mmask >> p) & 1u;
                            const uint32_t tok = (lo[p >> 1] >> (16 * (p & 1))) & 0xFFFFu;
                            const uint32_t e = (ew[p >> 2] >> (8 * (p & 3))) & 0xFFu;
                            st8_if(on, s_data + bb, ism ? tok : e);
                            st8_if(on & ism, s_data + bb + 1, tok >> 8);
                            bb += on * (1u + ism);
                            fbits |= (on & ism) << k;
                            k += on;
                        }
                    }
#pragma unroll
                    for (int p = 0; p < SEGP && WS != 1; ++p) {
                        if (!((path >> p) & 1u)) continue;
                        if ((mmask >> p) & 1u) {
                            const uint32_t v = (lo[p >> 1] >> (16 * (p & 1))) & 0xFFFFu;
                            *reinterpret_cast<uint16_t*>(s_data + bb) = (uint16_t)v;
                            bb += 2u;
                            fbits |= 1u << k;
                        } else {
                            if (WS == 2) {
                                *reinterpret_cast<uint16_t*>(s_data + bb) = (uint16_t)(ew[p >> 1] >> (16 * (p & 1)));
                            } else {
                                *reinterpret_cast<uint16_t*>(s_data + bb) = (uint16_t)ew[p];
                                *reinterpret_cast<uint16_t*>(s_data + bb + 2) = (uint16_t)(ew[p] >> 16);
                            }
                            bb += WS;
                        }
                        ++k;
                    }
                    if (fbits) or_bits(s_fl, item_base, fbits);
                    if (tid == 0)
                        for (uint32_t z = dbytes; z < ((dbytes + 3u) & ~3u); ++z) s_data[z] = 0;
                }
            }
        }
        p_c = c;
        p_blk = blk;
        p_entry = nonzero ? entry_items : 0u;
        p_dbytes = nonzero ? dbytes : 0u;
        p_fw = fw;
        p_dw = dw;
        __syncthreads();
        if (!SINGLE) {
            // ---- E10 (two pass): block to its slot, size and table entry ----
            uint8_t* slot = a.slots + (uint64_t)c * CS;
            for (uint32_t j = tid; j < fw + dw; j += nthreads) {
                const uint32_t v = j < fw ? s_fl[j]
                                          : *reinterpret_cast<const uint32_t*>(s_data + 4u * (j - fw));
                *reinterpret_cast<uint32_t*>(slot + 4u * j) = v;
            }
            if (tid == 0) {
                if (a.split) {
                    // literal bytes (the whole chunk if raw), matches, flag words
                    const bool raw = p_entry == kRawBit;
                    const uint32_t m = (nonzero && !raw) ? n_match : 0u;
                    a.sizes[c] = !nonzero ? 0u : (raw ? CS : WS * (items - n_match));
                    a.msizes[c] = m | (fw << 16);
                    const uint64_t eo = (uint64_t)kSplitHeaderBytes + (uint64_t)kEntryBytes * c;
                    store_u32_capped(a.out, eo, p_entry, a.capacity);
                    store_u32_capped(a.out, eo + 4, m, a.capacity);
                } else {
                    a.sizes[c] = blk;
                    const uint64_t eo = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * c;
                    store_u32_capped(a.out, eo, p_entry, a.capacity);
                    store_u32_capped(a.out, eo + 4, p_dbytes, a.capacity);
                }
            }
            __syncthreads();  // staging is free again
        }
    }
}

// ---------------------------------------------------------------------------
// Pack pass (two pass). offsets_pass: a CTA per tile of kTile chunks scans
// their sizes and finds the tile's stream offset by look-back over tile
// descriptors; it writes every chunk's block offset, and the last tile the
// header and the stream length. copy_pass: one warp per chunk moves the block
// from its slot to its offset (16-byte loads, 32-bit stores, nothing at or
// past capacity).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanThreads) offsets_pass(EncodeArgs a, uint32_t ws) {
    __shared__ TileSmem sm;
    const int tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();  // the encode kernel's sizes
    const uint32_t n_tiles = (a.n_chunks + kTile - 1) / kTile;
    if (a.n_chunks == 0) {
        if (blockIdx.x == 0 && tid == 0) write_header(a, ws, kHeaderBytes);
        return;
    }
    const uint64_t body0 = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * a.n_chunks;
    for (;;) {
        if (tid == 0) sm.tile = atomicAdd(a.ticket2, 1u);
        __syncthreads();
        const uint32_t t = sm.tile;
        if (t >= n_tiles) break;
        const uint64_t prefix = tile_scan(sm, t, a.n_chunks, a.tdesc, a.epoch, a.status,
                                          [&](uint32_t c) { return a.sizes[c]; });
        const uint32_t c0 = t * kTile;
        for (uint32_t j = (uint32_t)tid; j < kTile && c0 + j < a.n_chunks; j += kScanThreads)
            a.offsets[c0 + j] = body0 + prefix + sm.off[j];
        if (t == n_tiles - 1 && tid == 0) write_header(a, ws, body0 + prefix + sm.total);
        __syncthreads();
    }
}

constexpr int kCopyWarps = 8;

__global__ void __launch_bounds__(kCopyWarps * 32) copy_pass(EncodeArgs a) {
    const int lane = threadIdx.x & 31;
    pdl_wait();  // the offsets (and, through them, the slots)
    const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
    for (uint32_t c = gw; c < a.n_chunks; c += nw) {
        const uint32_t blk = a.sizes[c];
        const uint64_t dst = a.offsets[c];
        const uint8_t* src = a.slots + (uint64_t)c * a.chunk_size;
        for (uint32_t i = 16u * lane; i < blk; i += 512u) {
            const uint4 v = *reinterpret_cast<const uint4*>(src + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (i + 4u * k < blk) store_u32_capped(a.out, dst + i + 4u * k, w[k], a.capacity);
        }
    }
}

// ---------------------------------------------------------------------------
// Pack pass, split mode. offsets_pass_split: per tile of kTile chunks, three
// scans (flag words, literal bytes, matches), each with its own tile
// descriptors and look-back; the last tile writes the meta header and the
// port lengths. copy_pass_split: one warp per chunk moves its flag words to
// the meta port (after the header and size table) and its literals, lengths
// and offsets to their ports, nothing at or past a port's capacity.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kScanThreads) offsets_pass_split(EncodeArgs a, uint32_t ws) {
    __shared__ TileSmem sm;
    const int tid = threadIdx.x;
    pdl_trigger();
    pdl_wait();  // the encode kernel's sizes
    const uint32_t n_tiles = (a.n_chunks + kTile - 1) / kTile;
    if (a.n_chunks == 0) {
        if (blockIdx.x == 0 && tid == 0)
            write_header_split(a, ws, kSplitHeaderBytes, 0, 0);
        return;
    }
    for (;;) {
        if (tid == 0) sm.tile = atomicAdd(a.ticket2, 1u);
        __syncthreads();
        const uint32_t t = sm.tile;
        if (t >= n_tiles) break;
        const uint32_t c0 = t * kTile;
        uint64_t tot[3];
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const uint64_t prefix =
                tile_scan(sm, t, a.n_chunks, a.tdesc + (uint64_t)k * a.tdesc_stride, a.epoch, a.status,
                          [&](uint32_t c) {
                              return k == 0 ? a.msizes[c] >> 16 : (k == 1 ? a.sizes[c] : a.msizes[c] & 0xFFFFu);
                          });
            for (uint32_t j = (uint32_t)tid; j < kTile && c0 + j < a.n_chunks; j += kScanThreads)
                a.offsets[3ull * (c0 + j) + k] = prefix + sm.off[j];
            tot[k] = prefix + sm.total;
            __syncthreads();
        }
        if (t == n_tiles - 1 && tid == 0)
            write_header_split(a, ws,
                               (uint64_t)kSplitHeaderBytes + (uint64_t)kEntryBytes * a.n_chunks + 4ull * tot[0],
                               tot[1], tot[2]);
        __syncthreads();
    }
}

// Copy n bytes from a slot to a port at any byte offset: the head bytes up
// to a 4-byte boundary of the destination, then 32-bit stores of words
// assembled from two aligned slot words (a funnel shift), then the tail
// bytes; nothing at or past cap. The slot reads are aligned words that each
// hold at least one of the n bytes, so they stay inside the slot area (a
// multiple of 4 bytes long).
__device__ __forceinline__ void copy_bytes_capped(uint8_t* dst, uint64_t at, uint64_t cap,
                                                  const uint8_t* src, uint32_t n, int lane) {
    const uint32_t mis = (uint32_t)(reinterpret_cast<uintptr_t>(dst + at) & 3u);
    const uint32_t head = mis == 0u ? 0u : (4u - mis < n ? 4u - mis : n);
    if ((uint32_t)lane < head && at + lane < cap) dst[at + lane] = src[lane];
    const uint32_t nw = (n - head) / 4u;
    const uint8_t* s0 = src + head;
    const uint32_t sh = (uint32_t)(reinterpret_cast<uintptr_t>(s0) & 3u);
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(s0 - sh);
    uint32_t* dw = reinterpret_cast<uint32_t*>(dst + at + head);
    for (uint32_t i = lane; i < nw; i += 32u) {
        // the second word is needed only when shifting (no read past the bytes otherwise)
        const uint32_t i2 = sh == 0u ? i : i + 1u;
        const uint32_t v = __funnelshift_r(sw[i], sw[i2], 8u * sh);
        if (at + head + 4ull * i + 4 <= cap) dw[i] = v;
    }
    const uint32_t done = head + 4u * nw;
    if ((uint32_t)lane < n - done && at + done + lane < cap) dst[at + done + lane] = src[done + lane];
}

__global__ void __launch_bounds__(kCopyWarps * 32) copy_pass_split(EncodeArgs a) {
    const int lane = threadIdx.x & 31;
    pdl_wait();  // the offsets (and, through them, the slots)
    const uint32_t gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const uint32_t nw = (gridDim.x * blockDim.x) >> 5;
    const uint64_t flags0 = (uint64_t)kSplitHeaderBytes + (uint64_t)kEntryBytes * a.n_chunks;
    for (uint32_t c = gw; c < a.n_chunks; c += nw) {
        const uint32_t ms = a.msizes[c];
        const uint32_t fw = ms >> 16, m = ms & 0xFFFFu, lit = a.sizes[c];
        const uint64_t* o = a.offsets + 3ull * c;
        const uint8_t* src = a.slots + (uint64_t)c * a.chunk_size;
        copy_bytes_capped(a.out, flags0 + 4ull * o[0], a.capacity, src, 4u * fw, lane);
        copy_bytes_capped(a.port[0], o[1], a.port_cap[0], src + 4u * fw, lit, lane);
        copy_bytes_capped(a.port[1], o[2], a.port_cap[1], src + 4u * fw + lit, m, lane);
        copy_bytes_capped(a.port[2], o[2], a.port_cap[2], src + 4u * fw + lit + m, m, lane);
    }
}

struct LaunchShape {
    int dev = -1;
    uint32_t smem = 0;
    int sms = 0;
    int per_sm = 0;
};

// Occupancy-derived grid for a kernel, cached per (device, shared memory).
template <typename K>
cudaError_t shape_for(K kern, int threads, uint32_t smem, LaunchShape& cache) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (cache.dev == dev && cache.smem == smem) return cudaSuccess;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return err;
    int sms = 0, per_sm = 0;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem)) !=
        cudaSuccess)
        return err;
    cache.dev = dev;
    cache.smem = smem;
    cache.sms = sms;
    cache.per_sm = per_sm < 1 ? 1 : per_sm;
    return cudaSuccess;
}

template <int WS, int LEVEL, bool SINGLE, int NEARW = 32>
cudaError_t launch_t(const EncodeArgs& a, cudaStream_t stream) {
    static thread_local LaunchShape shape16, shape8, shape_copy;
    const EncLayout L = enc_layout(a.chunk_size, a.elems, LEVEL);
    const int threads = 32 * team_warps(a.elems);
    // positions per thread: 8, except 16 for 4096-element chunks (bytes at
    // chunk_size 4096, the only geometry with that many elements)
    const bool s16 = a.elems / (uint32_t)threads == 16u;
    void (*kern)(EncodeArgs) = encode_kernel<WS, LEVEL, 8, SINGLE, NEARW>;
    if constexpr (WS == 1) {
        if (s16) kern = encode_kernel<WS, LEVEL, 16, SINGLE, NEARW>;
    }
    LaunchShape& shape = s16 ? shape16 : shape8;
    cudaError_t err = shape_for(kern, threads, L.total, shape);
    if (err != cudaSuccess) return err;
    uint64_t grid = (uint64_t)shape.sms * (uint64_t)shape.per_sm;
    if (grid > a.n_chunks) grid = a.n_chunks;
    if (grid < 1) grid = 1;
    const KernelEvents ev = SINGLE ? KernelEvents{nullptr, nullptr} : kernel_events();
    if (ev.start && (err = cudaEventRecord(ev.start, stream)) != cudaSuccess) return err;
    kern<<<(unsigned)grid, threads, L.total, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (ev.stop && (err = cudaEventRecord(ev.stop, stream)) != cudaSuccess) return err;
    if (!SINGLE) {
        const uint64_t tiles = (a.n_chunks + kTile - 1) / kTile;
        uint64_t sgrid = (uint64_t)shape.sms * 4u;
        if (sgrid > tiles) sgrid = tiles;
        if (sgrid < 1) sgrid = 1;
        if ((err = pdl_launch(a.split ? offsets_pass_split : offsets_pass, dim3((unsigned)sgrid),
                              dim3(kScanThreads), 0, stream, a, (uint32_t)WS)) != cudaSuccess)
            return err;
        if (a.n_chunks > 0) {
            if ((err = shape_for(copy_pass, kCopyWarps * 32, 0, shape_copy)) != cudaSuccess)
                return err;
            uint64_t cgrid = (uint64_t)shape_copy.sms * (uint64_t)shape_copy.per_sm;
            const uint64_t need = (a.n_chunks + kCopyWarps - 1) / kCopyWarps;
            if (cgrid > need) cgrid = need;
            err = pdl_launch(a.split ? copy_pass_split : copy_pass, dim3((unsigned)cgrid),
                             dim3(kCopyWarps * 32), 0, stream, a);
        }
    }
    return err;
}

}  // namespace

cudaError_t launch_encode(const EncodeArgs& a, int word_size, int match_level, bool single_pass,
                          cudaStream_t stream) {
    if (a.far_mask != 0u) {  // near window of 33..64 elements: two pass, level 0
        if (single_pass || match_level != 0) return cudaErrorInvalidValue;
        if (word_size == 4) return launch_t<4, 0, false, 64>(a, stream);
        if (word_size == 2) return launch_t<2, 0, false, 64>(a, stream);
        return launch_t<1, 0, false, 64>(a, stream);
    }
    if (single_pass) {
        if (word_size == 4) return match_level ? launch_t<4, 1, true>(a, stream) : launch_t<4, 0, true>(a, stream);
        if (word_size == 2) return match_level ? launch_t<2, 1, true>(a, stream) : launch_t<2, 0, true>(a, stream);
        return match_level ? launch_t<1, 1, true>(a, stream) : launch_t<1, 0, true>(a, stream);
    }
    if (word_size == 4) return match_level ? launch_t<4, 1, false>(a, stream) : launch_t<4, 0, false>(a, stream);
    if (word_size == 2) return match_level ? launch_t<2, 1, false>(a, stream) : launch_t<2, 0, false>(a, stream);
    return match_level ? launch_t<1, 1, false>(a, stream) : launch_t<1, 0, false>(a, stream);
}

}  // namespace gpulz
