// GPULZ encode kernel for sm_103a.
//
// One CTA ("team" of 1..8 warps) codes one chunk at a time and loops over
// chunks in ticket order (persistent grid). Per chunk, following the GPULZ
// stage page of FZGPUModules:
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
//   E9 cross-chunk offsets     (single-pass decoupled look-back, bounded)
//   E10 store-out, size table, header and the stream length
//
// The greedy parse is computed in parallel: a warp walks 32-position windows,
// finding the on-path positions of each window from its first position by
// pointer doubling over next(i) = i + step(i) with warp reductions. With more
// than one warp, each warp walks its own segment from the segment start and
// warp 0 then repairs each segment from its true entry until the repaired
// path merges with the speculative one (paths that meet coincide afterwards).
#include <cuda_runtime.h>
#include <stdint.h>

#include "gpulz_internal.cuh"

namespace gpulz {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;

struct EncLayout {
    uint32_t el, om, lo, tab, fl, path, data, misc, total;
};

__host__ __device__ inline uint32_t align16(uint32_t v) { return (v + 15u) & ~15u; }

__host__ __device__ inline EncLayout enc_layout(uint32_t cs, uint32_t E, int level) {
    EncLayout L;
    uint32_t o = 0;
    L.el = o;   o = align16(o + cs + E);                 // elements, 16 B pad per 16 elements
    L.om = o;   o = align16(o + 4u * (E + E / 4u));      // omask, 4 pad words per 16 masks
    L.lo = o;   o = align16(o + 2u * E);                 // (len | off << 8) per position
    L.tab = o;  o = align16(o + (level ? 8u * E : 0u));  // level-1 table, 2E buckets of u32
    L.fl = o;   o = align16(o + E / 8u);                 // flag staging
    L.path = o; o = align16(o + E / 8u);                 // on-path bitmask
    L.data = o; o = align16(o + cs + 256u);              // item staging
    L.misc = o; o = align16(o + 256u);
    L.total = o;
    return L;
}

__host__ __device__ inline int team_warps(uint32_t E) { return E <= 512u ? 1 : (int)(E / 512u); }

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
// Word index of omask[i] in the padded omask array.
__device__ __forceinline__ uint32_t om_idx(uint32_t i) { return i + ((i >> 4) << 2); }

// Position of chunk byte b inside the padded element array.
template <int WS>
__device__ __forceinline__ uint32_t chunk_byte_addr(uint32_t b) {
    return b + ((b / (16u * WS)) << 4);
}

// ---------------------------------------------------------------------------
// Parse helpers (one warp).
// ---------------------------------------------------------------------------
// On-path lanes of a 32-position window whose first position is on the path.
// nxt = lane + step(lane) (relative; > lane). Pointer doubling: after round r
// the set holds the first 2^(r+1) path positions; 5 rounds cover a window.
__device__ __forceinline__ uint32_t window_path(uint32_t nxt, int lane) {
    uint32_t S = 1u;
    uint32_t J = nxt;
#pragma unroll
    for (int r = 0; r < 5; ++r) {
        uint32_t mine = (((S >> lane) & 1u) && J < 32u) ? (1u << J) : 0u;
        S |= __reduce_or_sync(FULL, mine);
        uint32_t Jn = __shfl_sync(FULL, J, J & 31u);
        J = (J < 32u) ? Jn : J;
    }
    return S;
}

template <int WS>
__device__ __forceinline__ uint32_t step_at(const uint16_t* s_lo, uint32_t pos, uint32_t E) {
    if (pos >= E) return 1u;
    uint32_t len = s_lo[pos] & 0xFFu;
    return len >= (uint32_t)min_match_len(WS) ? len : 1u;
}

// OR `bits` (relative to position `start`) into the bitmask.
__device__ __forceinline__ void or_bits(uint32_t* s_path, uint32_t start, uint32_t bits) {
    if (!bits) return;
    uint32_t w = start >> 5, sh = start & 31u;
    atomicOr(&s_path[w], bits << sh);
    if (sh && (bits >> (32u - sh))) atomicOr(&s_path[w + 1], bits >> (32u - sh));
}

// Clear bits [start, start + len) of the bitmask (warp-cooperative).
__device__ __forceinline__ void clear_bits(uint32_t* s_path, uint32_t start, uint32_t len,
                                           int lane) {
    if (!len) return;
    uint32_t end = start + len;
    uint32_t w0 = start >> 5, w1 = (end - 1) >> 5;
    for (uint32_t w = w0 + lane; w <= w1; w += 32) {
        uint32_t lo = (w == w0) ? (start & 31u) : 0u;
        uint32_t hi = (w == w1) ? ((end - 1) & 31u) : 31u;
        uint32_t m = (hi == 31u ? FULL : ((1u << (hi + 1)) - 1u)) & ~((1u << lo) - 1u);
        atomicAnd(&s_path[w], ~m);
    }
}

// Walk [cur, b) from `cur` (assumed on the path), recording path bits below b.
// Returns the first path position >= b.
template <int WS>
__device__ uint32_t walk_segment(uint32_t cur, uint32_t b, uint32_t E, const uint16_t* s_lo,
                                 uint32_t* s_path, int lane) {
    while (cur < b) {
        uint32_t nxt = (uint32_t)lane + step_at<WS>(s_lo, cur + lane, E);
        uint32_t S = window_path(nxt, lane);
        uint32_t lim = b - cur;
        uint32_t valid = lim >= 32u ? FULL : ((1u << lim) - 1u);
        uint32_t Sin = S & valid;
        if (lane == 0) or_bits(s_path, cur, Sin);
        int hi = 31 - __clz(Sin);
        cur += __shfl_sync(FULL, nxt, hi);
        __syncwarp();
    }
    return cur;
}

// Repair segment [a, b) whose speculative path started at a, given the true
// entry e >= a. Returns the true exit.
template <int WS>
__device__ uint32_t repair_segment(uint32_t e, uint32_t a, uint32_t b, uint32_t spec_exit,
                                   uint32_t E, const uint16_t* s_lo, uint32_t* s_path, int lane) {
    if (e == a) return spec_exit;
    clear_bits(s_path, a, e - a, lane);
    __syncwarp();
    uint32_t cur = e;
    while (cur < b) {
        uint32_t nxt = (uint32_t)lane + step_at<WS>(s_lo, cur + lane, E);
        uint32_t S = window_path(nxt, lane);
        uint32_t lim = b - cur;
        uint32_t valid = lim >= 32u ? FULL : ((1u << lim) - 1u);
        uint32_t Sin = S & valid;
        // speculative bits of [cur, cur + 32)
        uint32_t w = cur >> 5, sh = cur & 31u;
        uint32_t spec = s_path[w] >> sh;
        if (sh && w + 1 < (E >> 5)) spec |= s_path[w + 1] << (32u - sh);
        spec &= valid;
        uint32_t I = Sin & spec;
        __syncwarp();
        if (I) {
            uint32_t m = (uint32_t)__ffs(I) - 1u;  // first common position (relative)
            clear_bits(s_path, cur, m, lane);
            __syncwarp();
            if (lane == 0) or_bits(s_path, cur, Sin & ((1u << m) - 1u));
            __syncwarp();
            return spec_exit;
        }
        int hi = 31 - __clz(Sin);
        uint32_t nx = cur + __shfl_sync(FULL, nxt, hi);
        uint32_t upto = nx < b ? nx : b;
        clear_bits(s_path, cur, upto - cur, lane);
        __syncwarp();
        if (lane == 0) or_bits(s_path, cur, Sin);
        __syncwarp();
        cur = nx;
    }
    return cur;
}

// ---------------------------------------------------------------------------
// Look-back (warp 0): exclusive prefix of block bytes over earlier chunks.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void publish_aggregate(const EncodeArgs& a, uint32_t c,
                                                  uint64_t aggregate) {
    st_relaxed_u64(&a.desc[c],
                   make_desc(a.epoch, c == 0 ? kDescInclusive : kDescAggregate, aggregate));
}

// Exclusive prefix of block bytes over chunks [0, c) by decoupled look-back.
// The warp inspects kLookBackWidth predecessors per step (each lane loads
// kLookBackPerLane descriptors, so the loads overlap): it sums aggregates back
// to the nearest inclusive prefix. The aggregate of chunk c must already be
// published. Waits are bounded by kWaitLimitNs of device time.
constexpr int kLookBackPerLane = 8;
constexpr int kLookBackWidth = 32 * kLookBackPerLane;

__device__ uint64_t lookback_encode(const EncodeArgs& a, uint32_t c, uint64_t aggregate, int lane,
                                    bool* timed_out) {
    *timed_out = false;
    if (c == 0) return 0;
    const uint64_t* desc = a.desc;
    uint64_t prefix = 0;
    int64_t base = (int64_t)c - 1;
    uint64_t t0 = 0;
    for (;;) {
        uint64_t d[kLookBackPerLane];
#pragma unroll
        for (int k = 0; k < kLookBackPerLane; ++k) {
            int64_t idx = base - (k * 32 + lane);
            d[k] = idx >= 0 ? ld_relaxed_u64(&desc[idx]) : make_desc(a.epoch, kDescInclusive, 0);
        }
        uint32_t my_min = 0xFFFFFFFFu;
#pragma unroll
        for (int k = kLookBackPerLane - 1; k >= 0; --k) {
            bool incl = desc_epoch(d[k]) == a.epoch && desc_kind(d[k]) == kDescInclusive;
            if (incl) my_min = (uint32_t)(k * 32 + lane);
        }
        const uint32_t dmin = __reduce_min_sync(FULL, my_min);
        const uint32_t lim = dmin == 0xFFFFFFFFu ? (uint32_t)kLookBackWidth : dmin + 1u;
        bool bad = false;
        uint64_t v = 0;
#pragma unroll
        for (int k = 0; k < kLookBackPerLane; ++k) {
            if ((uint32_t)(k * 32 + lane) < lim) {
                bool valid = desc_epoch(d[k]) == a.epoch && desc_kind(d[k]) != 0;
                bad |= !valid;
                v += desc_value(d[k]);
            }
        }
        if (__any_sync(FULL, bad)) {
            uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > kWaitLimitNs) {
                *timed_out = true;
                break;
            }
            __nanosleep(32);
            continue;
        }
        prefix += warp_sum_u64(v);
        if (dmin != 0xFFFFFFFFu) break;
        base -= kLookBackWidth;
    }
    if (lane == 0)
        st_relaxed_u64(&a.desc[c], make_desc(a.epoch, kDescInclusive, prefix + aggregate));
    return prefix;
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

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <int WS, int LEVEL>
__global__ void __launch_bounds__(256) encode_kernel(EncodeArgs a) {
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
    uint32_t* s_tab = reinterpret_cast<uint32_t*>(smem + L.tab);
    uint32_t* s_fl = reinterpret_cast<uint32_t*>(smem + L.fl);
    uint32_t* s_path = reinterpret_cast<uint32_t*>(smem + L.path);
    uint8_t* s_data = smem + L.data;
    uint32_t* s_misc = reinterpret_cast<uint32_t*>(smem + L.misc);
    constexpr uint32_t LMIN = (uint32_t)min_match_len(WS);

    if (a.n_chunks == 0) {
        if (blockIdx.x == 0 && tid == 0) write_header(a, WS, kHeaderBytes);
        return;
    }
    const uint64_t body0 = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * a.n_chunks;
    const bool in_aligned = (reinterpret_cast<uintptr_t>(a.in) & 15u) == 0;

    for (;;) {
        if (tid == 0) s_misc[0] = atomicAdd(a.ticket, 1u);
        __syncthreads();
        const uint32_t c = s_misc[0];
        if (c >= a.n_chunks) break;

        // ---- E1: load the chunk (zero padded) ----
        const uint64_t begin = (uint64_t)c * CS;
        const uint64_t avail = a.n_bytes - begin;
        const uint32_t take = avail < CS ? (uint32_t)avail : CS;
        uint32_t nz = 0;
        if (in_aligned && take == CS) {
            const uint4* src = reinterpret_cast<const uint4*>(a.in + begin);
            for (uint32_t g = tid; g < CS / 16u; g += nthreads) {
                uint4 v = __ldg(src + g);
                uint32_t* dst = reinterpret_cast<uint32_t*>(s_el + chunk_byte_addr<WS>(16u * g));
                dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
                nz |= v.x | v.y | v.z | v.w;
            }
        } else {
            for (uint32_t b4 = tid; b4 < CS / 4u; b4 += nthreads) {
                uint32_t v = 0;
                for (uint32_t k = 0; k < 4u; ++k) {
                    uint32_t b = 4u * b4 + k;
                    if (b < take) v |= (uint32_t)a.in[begin + b] << (8u * k);
                }
                *reinterpret_cast<uint32_t*>(s_el + chunk_byte_addr<WS>(4u * b4)) = v;
                nz |= v;
            }
        }
        // clear per-chunk state
        for (uint32_t k = tid; k < E / 32u; k += nthreads) {
            s_fl[k] = 0;
            s_path[k] = 0;
        }
        if (LEVEL) {
            for (uint32_t k = tid; k < 2u * E; k += nthreads) s_tab[k] = 0;
        }
        // ---- E2: zero test ----
        const bool nonzero = __syncthreads_or(nz != 0) != 0;

        uint32_t items = 0, dbytes = 0, blk = 0, entry_items = 0;
        if (nonzero) {
            // ---- E3: near equality masks, 16 positions per thread step ----
            for (uint32_t g = tid; g < E / 16u; g += nthreads) {
                uint32_t v[48];
#pragma unroll
                for (int h = 0; h < 3; ++h) {
                    int grp = (int)g - 2 + h;
                    if (grp < 0) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[16 * h + k] = 0;
                        continue;
                    }
                    const uint4* p = reinterpret_cast<const uint4*>(s_el + el_addr<WS>(16u * grp));
#pragma unroll
                    for (int q = 0; q < WS; ++q) {
                        uint4 t = p[q];
                        uint32_t wd[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            if (WS == 4) {
                                v[16 * h + 4 * q + r] = wd[r];
                            } else if (WS == 2) {
                                v[16 * h + 8 * q + 2 * r] = wd[r] & 0xFFFFu;
                                v[16 * h + 8 * q + 2 * r + 1] = wd[r] >> 16;
                            } else {
#pragma unroll
                                for (int s = 0; s < 4; ++s)
                                    v[16 * h + 16 * q + 4 * r + s] = (wd[r] >> (8 * s)) & 0xFFu;
                            }
                        }
                    }
                }
                uint32_t m[16];
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    uint32_t x = v[32 + p];
                    uint32_t mm = 0;
#pragma unroll
                    for (int o = 1; o <= 32; ++o) mm |= (v[32 + p - o] == x) ? (1u << (o - 1)) : 0u;
                    uint32_t i = 16u * g + (uint32_t)p;
                    if (i < 32u) mm &= (1u << i) - 1u;
                    m[p] = mm;
                }
                uint4* dst = reinterpret_cast<uint4*>(s_om + om_idx(16u * g));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(m[4 * q], m[4 * q + 1], m[4 * q + 2], m[4 * q + 3]);
            }
            __syncthreads();

            // ---- E4: AND-chain longest match, nearest offset ----
            for (uint32_t i = tid; i < E; i += nthreads) {
                uint32_t mm = s_om[om_idx(i)];
                uint32_t lo = 0;
                if (mm) {
                    uint32_t cap = E - i < (uint32_t)kMaxLen ? E - i : (uint32_t)kMaxLen;
                    uint32_t len = 1;
                    while (len < cap) {
                        uint32_t nm = mm & s_om[om_idx(i + len)];
                        if (!nm) break;
                        mm = nm;
                        ++len;
                    }
                    lo = len | ((uint32_t)__ffs(mm) << 8);
                }
                s_lo[i] = (uint16_t)lo;
            }
            __syncthreads();

            // ---- E5: level-1 hashed candidates over 8 sub-blocks ----
            if (LEVEL) {
                const uint32_t SB = E / kSubBlocks;
                for (int s = 0; s < kSubBlocks; ++s) {
                    const uint32_t lo_i = (uint32_t)s * SB;
                    for (uint32_t i = lo_i + tid; i < lo_i + SB; i += nthreads) {
                        if (i + 1u >= E) continue;
                        uint32_t slot = s_tab[key_hash(el_get<WS>(s_el, i), el_get<WS>(s_el, i + 1u),
                                                       a.hash_bits)];
                        if (!slot) continue;
                        uint32_t p = slot - 1u;
                        uint32_t d = i - p;
                        if (d > (uint32_t)kMaxOff) continue;
                        uint32_t cap = E - i < (uint32_t)kMaxLen ? E - i : (uint32_t)kMaxLen;
                        uint32_t k = 0;
                        while (k < cap && el_get<WS>(s_el, i + k) == el_get<WS>(s_el, p + k)) ++k;
                        if (!k) continue;
                        uint32_t cur = s_lo[i];
                        uint32_t l0 = cur & 0xFFu, o0 = cur >> 8;
                        if (k > l0 || (k == l0 && d < o0)) s_lo[i] = (uint16_t)(k | (d << 8));
                    }
                    __syncthreads();
                    for (uint32_t p = lo_i + tid; p < lo_i + SB; p += nthreads) {
                        if (p + 1u >= E) continue;
                        atomicMax(&s_tab[key_hash(el_get<WS>(s_el, p), el_get<WS>(s_el, p + 1u),
                                                  a.hash_bits)],
                                  p + 1u);
                    }
                    __syncthreads();
                }
            }

            // ---- E6: greedy parse -> on-path bitmask ----
            const uint32_t SEG = E / (uint32_t)nwarps;
            {
                uint32_t sa = (uint32_t)warp * SEG;
                uint32_t ex = walk_segment<WS>(sa, sa + SEG, E, s_lo, s_path, lane);
                if (lane == 0) s_misc[8 + warp] = ex;
            }
            __syncthreads();
            if (nwarps > 1 && warp == 0) {
                uint32_t e = s_misc[8];
                for (int w = 1; w < nwarps; ++w) {
                    uint32_t sa = (uint32_t)w * SEG;
                    e = repair_segment<WS>(e, sa, sa + SEG, s_misc[8 + w], E, s_lo, s_path, lane);
                }
            }
            __syncthreads();

            // ---- count items and match tokens per segment ----
            {
                uint32_t sa = (uint32_t)warp * SEG;
                uint32_t n_it = 0, n_m = 0;
                for (uint32_t bp = sa; bp < sa + SEG; bp += 32u) {
                    uint32_t S = s_path[bp >> 5];
                    uint32_t len = s_lo[bp + lane] & 0xFFu;
                    bool ism = ((S >> lane) & 1u) && len >= LMIN;
                    uint32_t M = __ballot_sync(FULL, ism);
                    n_it += __popc(S);
                    n_m += __popc(M);
                }
                if (lane == 0) {
                    s_misc[16 + warp] = n_it;
                    s_misc[24 + warp] = n_m;
                }
            }
            __syncthreads();
            uint32_t item_base = 0, match_base = 0;
            for (int w = 0; w < nwarps; ++w) {
                uint32_t ni = s_misc[16 + w], nm = s_misc[24 + w];
                if (w < warp) {
                    item_base += ni;
                    match_base += nm;
                }
                items += ni;
                dbytes += WS * (ni - nm) + 2u * nm;
            }
            blk = 4u * ((items + 31u) / 32u) + ((dbytes + 3u) & ~3u);
            if (blk >= CS) {
                blk = CS;
                entry_items = kRawBit;
                dbytes = CS;
            }
            // publish this chunk's size before packing, so successors' look-backs resolve early
            if (tid == 0) publish_aggregate(a, c, blk);
            if (entry_items != kRawBit) {
                entry_items = items;
                // ---- E7: emit flags + items into staging ----
                uint32_t sa = (uint32_t)warp * SEG;
                uint32_t ib = item_base;
                uint32_t bb = WS * (item_base - match_base) + 2u * match_base;
                const uint32_t lt = lanemask_lt();
                for (uint32_t bp = sa; bp < sa + SEG; bp += 32u) {
                    uint32_t S = s_path[bp >> 5];
                    uint32_t pos = bp + lane;
                    uint32_t lo = s_lo[pos];
                    uint32_t len = lo & 0xFFu;
                    bool onp = (S >> lane) & 1u;
                    bool ism = onp && len >= LMIN;
                    uint32_t M = __ballot_sync(FULL, ism);
                    uint32_t rank = __popc(S & lt);
                    uint32_t mb = __popc(M & lt);
                    uint32_t boff = bb + WS * (rank - mb) + 2u * mb;
                    if (onp) {
                        if (ism) {
                            if (WS == 1) {
                                s_data[boff] = (uint8_t)len;
                                s_data[boff + 1] = (uint8_t)(lo >> 8);
                            } else {
                                *reinterpret_cast<uint16_t*>(s_data + boff) = (uint16_t)lo;
                            }
                        } else {
                            uint32_t v = el_get<WS>(s_el, pos);
                            if (WS == 1) {
                                s_data[boff] = (uint8_t)v;
                            } else if (WS == 2) {
                                *reinterpret_cast<uint16_t*>(s_data + boff) = (uint16_t)v;
                            } else {
                                *reinterpret_cast<uint16_t*>(s_data + boff) = (uint16_t)v;
                                *reinterpret_cast<uint16_t*>(s_data + boff + 2) = (uint16_t)(v >> 16);
                            }
                        }
                    }
                    uint32_t fb = __reduce_or_sync(FULL, ism ? (1u << rank) : 0u);
                    if (lane == 0 && fb) or_bits(s_fl, ib, fb);
                    uint32_t n = __popc(S), nm = __popc(M);
                    ib += n;
                    bb += WS * (n - nm) + 2u * nm;
                }
            }
        }
        if (!nonzero && tid == 0) publish_aggregate(a, c, 0);
        // ---- E9: look-back for this chunk's byte offset ----
        if (warp == 0) {
            bool to = false;
            uint64_t prefix = lookback_encode(a, c, blk, lane, &to);
            if (lane == 0) {
                if (to) atomicOr(a.status, kStatTimeout);
                s_misc[40] = (uint32_t)prefix;
                s_misc[41] = (uint32_t)(prefix >> 32);
            }
        }
        if (tid == 0 && entry_items != kRawBit && nonzero) {
            // zero the padding bytes after the last item
            for (uint32_t k = dbytes; k < ((dbytes + 3u) & ~3u); ++k) s_data[k] = 0;
        }
        __syncthreads();
        const uint64_t prefix = (uint64_t)s_misc[40] | ((uint64_t)s_misc[41] << 32);

        // ---- E10: store-out (32-bit coalesced), size-table entry, header ----
        const uint64_t dst = body0 + prefix;
        if (nonzero) {
            if (entry_items == kRawBit) {
                for (uint32_t j = tid; j < CS / 4u; j += nthreads) {
                    uint32_t v = *reinterpret_cast<const uint32_t*>(s_el + chunk_byte_addr<WS>(4u * j));
                    store_u32_capped(a.out, dst + 4ull * j, v, a.capacity);
                }
            } else {
                const uint32_t fw = (items + 31u) / 32u;
                const uint32_t dw = (dbytes + 3u) / 4u;
                for (uint32_t j = tid; j < fw + dw; j += nthreads) {
                    uint32_t v = j < fw ? s_fl[j]
                                        : *reinterpret_cast<const uint32_t*>(s_data + 4u * (j - fw));
                    store_u32_capped(a.out, dst + 4ull * j, v, a.capacity);
                }
            }
        }
        if (tid == 0) {
            uint64_t eo = (uint64_t)kHeaderBytes + (uint64_t)kEntryBytes * c;
            store_u32_capped(a.out, eo, nonzero ? entry_items : 0u, a.capacity);
            store_u32_capped(a.out, eo + 4, nonzero ? dbytes : 0u, a.capacity);
            if (c == a.n_chunks - 1u) write_header(a, WS, dst + blk);
        }
        __syncthreads();
    }
}

template <int WS, int LEVEL>
cudaError_t launch_t(const EncodeArgs& a, cudaStream_t stream) {
    const EncLayout L = enc_layout(a.chunk_size, a.elems, LEVEL);
    const int threads = 32 * team_warps(a.elems);
    auto kern = encode_kernel<WS, LEVEL>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)L.total);
    if (err != cudaSuccess) return err;
    int dev = 0, sms = 0, per_sm = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return err;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, L.total)) !=
        cudaSuccess)
        return err;
    if (per_sm < 1) per_sm = 1;
    uint64_t grid = (uint64_t)sms * (uint64_t)per_sm;
    if (grid > a.n_chunks) grid = a.n_chunks;
    if (grid < 1) grid = 1;
    kern<<<(unsigned)grid, threads, L.total, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode(const EncodeArgs& a, int word_size, int match_level,
                          cudaStream_t stream) {
    if (word_size == 4) return match_level ? launch_t<4, 1>(a, stream) : launch_t<4, 0>(a, stream);
    if (word_size == 2) return match_level ? launch_t<2, 1>(a, stream) : launch_t<2, 0>(a, stream);
    return match_level ? launch_t<1, 1>(a, stream) : launch_t<1, 0>(a, stream);
}

}  // namespace gpulz
