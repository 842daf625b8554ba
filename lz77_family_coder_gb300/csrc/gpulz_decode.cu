// GPULZ decode kernel for sm_103a.
//
// Block-parallel decode (GPULZ stage page of FZGPUModules, decode paragraph):
// the flag bitmap fixes every item's byte size (word_size for a literal, 2 for
// a match), so an item's byte offset follows from a popcount of the flags
// before it; one warp scan over item spans gives every item's element offset
// q; each element of a match points back to q - offset (always < q, so chains
// end) and pointer jumping resolves all of them in at most log2(elements)
// rounds, stopping early once nothing changes. Zero chunks are zero-filled
// (zero-chunk paragraph) and raw chunks copied (raw-fallback paragraph).
//
// A first kernel (offsets_kernel) scans the size table into every chunk's
// block offset; then each warp of decode_kernel decodes one chunk at a time,
// taking chunks by ticket.
//
// The header is parsed on the device; chunk geometry is not known to the host
// launcher, so the shared-memory slot per warp is sized from the header at run
// time and the CTA keeps as many warps as fit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gpulz_internal.cuh"

namespace gpulz {
namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr int kDecWarps = 24;
constexpr uint32_t kDecSmem = 112u * 1024u;
constexpr int kMaxJumpRounds = 16;
constexpr uint16_t kLit = 0x8000u;

struct Geo {
    uint32_t ws, cs, E, C;
    uint64_t orig, total, body0;
    uint64_t lit_total, m_total;  // split mode: literal bytes and matches in the ports
};

__device__ __forceinline__ uint32_t align16d(uint32_t v) { return (v + 15u) & ~15u; }

// Per-warp shared-memory slot: flags | flag-word prefix | item bytes | src.
struct DecSlot {
    uint32_t fl, wp, data, src, total;
};
__device__ __forceinline__ DecSlot dec_slot(uint32_t cs, uint32_t E) {
    DecSlot s;
    uint32_t o = 0;
    s.fl = o;   o = align16d(o + E / 8u);
    s.wp = o;   o = align16d(o + 4u * (E / 32u));
    s.data = o; o = align16d(o + cs + 16u);
    s.src = o;  o = align16d(o + 2u * E);
    s.total = o;
    return s;
}

__device__ __forceinline__ uint32_t read_u32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}
// Four bytes at any address (split-mode ports have no alignment rule).
__device__ __forceinline__ uint32_t read_u32_any(const uint8_t* p) {
    if ((reinterpret_cast<uintptr_t>(p) & 3u) == 0) return read_u32(p);
    return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
// Copy n bytes from any address into a warp's shared-memory data area.
__device__ __forceinline__ void stage_bytes(uint8_t* dst, const uint8_t* src, uint32_t n, int lane) {
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | n) & 3u) == 0) {
        for (uint32_t i = 4u * lane; i < n; i += 128u)
            *reinterpret_cast<uint32_t*>(dst + i) = read_u32(src + i);
    } else {
        for (uint32_t i = lane; i < n; i += 32u) dst[i] = src[i];
    }
}

// Split mode: a chunk's (flag words, literal bytes, matches) from its entry;
// false if the entry is invalid.
__device__ __forceinline__ bool split_entry(uint32_t items, uint32_t m, const Geo& g, uint32_t& fw,
                                            uint32_t& lit) {
    fw = 0;
    lit = 0;
    if (items == 0 && m == 0) return true;
    if (items == kRawBit && m == 0) {
        lit = g.cs;
        return true;
    }
    if ((items & kRawBit) || items > g.E || m > items) return false;
    fw = (items + 31u) / 32u;
    lit = g.ws * (items - m);
    return lit + 2u * m <= g.cs;
}

// Block size of a size-table entry; 0xFFFFFFFF if the entry is invalid.
__device__ __forceinline__ uint32_t entry_block(uint32_t items, uint32_t dbytes, const Geo& g) {
    if (items == 0 && dbytes == 0) return 0;
    if (items == kRawBit) return dbytes == g.cs ? g.cs : 0xFFFFFFFFu;
    if ((items & kRawBit) || items > g.E || dbytes > g.cs) return 0xFFFFFFFFu;
    uint32_t blk = 4u * ((items + 31u) / 32u) + ((dbytes + 3u) & ~3u);
    return blk < g.cs ? blk : 0xFFFFFFFFu;
}


// Output a chunk as 32-bit words: word j covers chunk bytes [4j, 4j+4).
template <typename F>
__device__ __forceinline__ void write_chunk(uint8_t* out, uint32_t take, bool out_aligned, int lane,
                                            F word_of) {
    const uint32_t full_words = take / 4u;
    if (out_aligned) {
        uint32_t* o = reinterpret_cast<uint32_t*>(out);
        for (uint32_t j = lane; j < full_words; j += 32) o[j] = word_of(j);
    } else {
        for (uint32_t j = lane; j < full_words; j += 32) {
            uint32_t v = word_of(j);
            for (int k = 0; k < 4; ++k) out[4u * j + k] = (uint8_t)(v >> (8 * k));
        }
    }
    if (take & 3u) {
        uint32_t j = full_words;
        uint32_t v = word_of(j);
        if (lane < (int)(take & 3u)) out[4u * j + lane] = (uint8_t)(v >> (8 * lane));
    }
}

// e = s_src[e] unless e is resolved (kLit set); `base` = shared address of s_src.
__device__ __forceinline__ void follow(uint32_t& e, uint32_t base) {
    asm volatile("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\tand.b32 t, %0, 32768;\n\tsetp.eq.u32 p, t, 0;\n\t"
                 "@p ld.shared.u16 %0, [%1];\n\t}"
                 : "+r"(e)
                 : "r"(base + 2u * e)
                 : "memory");
}

template <int WS>
__device__ uint32_t lit_word(const uint8_t* s_data, const uint16_t* s_src, uint32_t j) {
    // chunk bytes [4j, 4j + 4) = elements [4j/WS, (4j+4)/WS)
    if (WS == 4) {
        uint32_t b = s_src[j] & 0x7FFFu;
        return (uint32_t)*reinterpret_cast<const uint16_t*>(s_data + b) |
               ((uint32_t)*reinterpret_cast<const uint16_t*>(s_data + b + 2) << 16);
    } else if (WS == 2) {
        uint32_t b0 = s_src[2 * j] & 0x7FFFu, b1 = s_src[2 * j + 1] & 0x7FFFu;
        return (uint32_t)*reinterpret_cast<const uint16_t*>(s_data + b0) |
               ((uint32_t)*reinterpret_cast<const uint16_t*>(s_data + b1) << 16);
    } else {
        uint32_t v = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) v |= (uint32_t)s_data[s_src[4 * j + k] & 0x7FFFu] << (8 * k);
        return v;
    }
}

template <int WS>
// A warp's first chunk is its index among the kernel's decoding warps (no
// ticket storm at start-up); later chunks come by ticket, after those.
__device__ void decode_chunks(const DecodeArgs& a, const Geo& g, uint8_t* slot_base, int lane,
                              uint32_t first, uint32_t n_warps) {
    const DecSlot S = dec_slot(g.cs, g.E);
    uint32_t* s_fl = reinterpret_cast<uint32_t*>(slot_base + S.fl);
    uint32_t* s_wp = reinterpret_cast<uint32_t*>(slot_base + S.wp);
    uint8_t* s_data = slot_base + S.data;
    uint16_t* s_src = reinterpret_cast<uint16_t*>(slot_base + S.src);
    const uint32_t E = g.E, CS = g.cs;
    const bool out_aligned = (reinterpret_cast<uintptr_t>(a.out) & 3u) == 0;
    for (bool initial = true;; initial = false) {
        uint32_t c = first;
        if (!initial) {
            if (lane == 0) c = atomicAdd(a.ticket2, 1u) + n_warps;
            c = __shfl_sync(FULL, c, 0);
        }
        if (c >= g.C) break;

        const bool split = a.split != 0;
        const uint8_t* e = a.in + (split ? kSplitHeaderBytes : kHeaderBytes) + (uint64_t)kEntryBytes * c;
        const uint32_t items = read_u32(e), second = read_u32(e + 4);
        // single stream: second = data bytes; split: second = matches
        uint32_t dbytes = second, blk = 0, sfw = 0, slit = 0;
        bool bad;
        uint64_t src_off = 0, s_of = 0, s_ol = 0, s_om = 0;
        if (!split) {
            blk = entry_block(items, dbytes, g);
            bad = blk == 0xFFFFFFFFu;
            src_off = a.offsets[c];
            if (!bad && (src_off < g.body0 || src_off + blk > g.total)) bad = true;
        } else {
            bad = !split_entry(items, second, g, sfw, slit);
            s_of = a.offsets[3ull * c];
            s_ol = a.offsets[3ull * c + 1];
            s_om = a.offsets[3ull * c + 2];
            if (!bad && (g.body0 + 4ull * (s_of + sfw) > g.total || s_ol + slit > g.lit_total ||
                         s_om + second > g.m_total))
                bad = true;
            blk = (items == 0 && second == 0) ? 0u : 1u;
            dbytes = slit + 2u * second;
        }

        const uint64_t begin = (uint64_t)c * CS;
        const uint64_t avail = g.orig - begin;
        const uint32_t take = avail < CS ? (uint32_t)avail : CS;
        uint8_t* out = a.out + begin;
        const bool chunk_out_aligned = out_aligned;

        if (bad) {
            if (lane == 0) atomicOr(a.status, kStatCorrupt);
            continue;
        }
        if (blk == 0) {
            write_chunk(out, take, chunk_out_aligned, lane, [](uint32_t) { return 0u; });
            continue;
        }
        const uint8_t* src = a.in + src_off;
        if (items == kRawBit) {
            if (split) {
                const uint8_t* lsrc = a.port[0] + s_ol;
                write_chunk(out, take, chunk_out_aligned, lane,
                            [lsrc](uint32_t j) { return read_u32_any(lsrc + 4u * j); });
            } else {
                write_chunk(out, take, chunk_out_aligned, lane,
                            [src](uint32_t j) { return read_u32(src + 4u * j); });
            }
            continue;
        }

        // ---- D2: load flags and items into shared memory ----
        const uint32_t fw = (items + 31u) / 32u;
        const uint32_t dw = split ? 0u : (dbytes + 3u) / 4u;
        if (split) {
            // flags from the meta port; literals, lengths and offsets from
            // theirs, into [literals | lengths | offsets] of the data area
            const uint8_t* fsrc = a.in + g.body0 + 4ull * s_of;
            for (uint32_t j = lane; j < fw; j += 32) {
                uint32_t v = read_u32(fsrc + 4u * j);
                if (j == fw - 1u && (items & 31u)) v &= (1u << (items & 31u)) - 1u;
                s_fl[j] = v;
            }
            stage_bytes(s_data, a.port[0] + s_ol, slit, lane);
            stage_bytes(s_data + slit, a.port[1] + s_om, second, lane);
            stage_bytes(s_data + slit + second, a.port[2] + s_om, second, lane);
        }
        // single stream: flags and items from the block, four loads in flight
        // per lane (split mode staged them above)
        const uint32_t nwords = split ? 0u : fw + dw;
        for (uint32_t j0 = lane; j0 < nwords; j0 += 128) {
            uint32_t vv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t j = j0 + 32u * u;
                vv[u] = j < fw + dw ? read_u32(src + 4u * j) : 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t j = j0 + 32u * u;
                if (j >= fw + dw) break;
                uint32_t v = vv[u];
                if (j < fw) {
                    if (j == fw - 1u && (items & 31u)) v &= (1u << (items & 31u)) - 1u;
                    s_fl[j] = v;
                } else {
                    *reinterpret_cast<uint32_t*>(s_data + 4u * (j - fw)) = v;
                }
            }
        }
        __syncwarp();
        // flag-word prefix popcounts
        uint32_t run = 0;
        for (uint32_t j0 = 0; j0 < fw; j0 += 32) {
            uint32_t j = j0 + lane;
            uint32_t pc = j < fw ? __popc(s_fl[j]) : 0u;
            uint32_t incl = pc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                uint32_t t = __shfl_up_sync(FULL, incl, o);
                if (lane >= o) incl += t;
            }
            if (j < fw) s_wp[j] = run + incl - pc;
            run += __shfl_sync(FULL, incl, 31);
        }
        const uint32_t n_match = run;
        if (split ? n_match != second : (uint64_t)WS * (items - n_match) + 2ull * n_match != dbytes) {
            if (lane == 0) atomicOr(a.status, kStatCorrupt);
            continue;
        }
        __syncwarp();

        // ---- D3: item spans, warp scan -> element offsets ----
        const uint32_t K = (items + 31u) / 32u;
        const uint32_t j_lo = lane * K < items ? lane * K : items;
        const uint32_t j_hi = j_lo + K < items ? j_lo + K : items;
        // Single stream: the lane keeps its flag word and its match count in
        // registers and takes no branch between literals and matches; wider
        // words read each item's two bytes with one 16-bit load (every item
        // starts at an even byte). Split mode: per item.
        const bool uni = WS != 1 && !split;
        uint32_t span_sum = 0;
        if (uni) {
            uint32_t w = j_lo < j_hi ? s_fl[j_lo >> 5] : 0u;
            uint32_t pm = j_lo < j_hi ? s_wp[j_lo >> 5] + __popc(w & ((1u << (j_lo & 31u)) - 1u)) : 0u;
            for (uint32_t j = j_lo; j < j_hi; ++j) {
                if ((j & 31u) == 0u) w = s_fl[j >> 5];
                const uint32_t ism = (w >> (j & 31u)) & 1u;
                const uint32_t tok = *reinterpret_cast<const uint16_t*>(s_data + (WS * j - (WS - 2u) * pm));
                span_sum += ism ? (tok & 0xFFu) : 1u;
                pm += ism;
            }
        } else if (!split) {
            // bytes: item j's first byte is at j + pm (a match's length)
            uint32_t w = j_lo < j_hi ? s_fl[j_lo >> 5] : 0u;
            uint32_t pm = j_lo < j_hi ? s_wp[j_lo >> 5] + __popc(w & ((1u << (j_lo & 31u)) - 1u)) : 0u;
            for (uint32_t j = j_lo; j < j_hi; ++j) {
                if ((j & 31u) == 0u) w = s_fl[j >> 5];
                const uint32_t ism = (w >> (j & 31u)) & 1u;
                const uint32_t L = s_data[j + pm];
                span_sum += ism ? L : 1u;
                pm += ism;
            }
        } else {
            for (uint32_t j = j_lo; j < j_hi; ++j) {
                uint32_t w = s_fl[j >> 5];
                bool ism = (w >> (j & 31u)) & 1u;
                if (ism) {
                    uint32_t pm = s_wp[j >> 5] + __popc(w & ((1u << (j & 31u)) - 1u));
                    span_sum += s_data[slit + pm];
                } else {
                    span_sum += 1u;
                }
            }
        }
        uint32_t incl = span_sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t t = __shfl_up_sync(FULL, incl, o);
            if (lane >= o) incl += t;
        }
        const uint32_t total_span = __shfl_sync(FULL, incl, 31);
        if (total_span != E) {
            if (lane == 0) atomicOr(a.status, kStatCorrupt);
            continue;
        }

        // ---- D4: scatter literals and back-pointers ----
        // Bytes (4096-element chunks, long lane ranges): element q + k of a
        // match copies element q + k - O, which has the value of element
        // q - O + (k mod O); when that element lies in this lane's own range,
        // its entry is already final (a literal, or a pointer into an earlier
        // lane's range) and is copied, so pointer jumping only follows
        // pointers that cross lane ranges (about half the rounds there; for
        // wider words the extra load costs more than the rounds it saves).
        bool lane_bad = false;
        const uint32_t q_lane = incl - span_sum;  // first position of this lane's items
        uint32_t q = q_lane;
        if (uni) {
            // entries v0, v0 + 1, ... for a match (q - O onwards), one kLit | b
            // entry for a literal
            uint32_t w = j_lo < j_hi ? s_fl[j_lo >> 5] : 0u;
            uint32_t pm = j_lo < j_hi ? s_wp[j_lo >> 5] + __popc(w & ((1u << (j_lo & 31u)) - 1u)) : 0u;
            for (uint32_t j = j_lo; j < j_hi; ++j) {
                if ((j & 31u) == 0u) w = s_fl[j >> 5];
                const uint32_t ism = (w >> (j & 31u)) & 1u;
                const uint32_t b = WS * j - (WS - 2u) * pm;
                const uint32_t tok = *reinterpret_cast<const uint16_t*>(s_data + b);
                const uint32_t L = ism ? (tok & 0xFFu) : 1u, O = tok >> 8;
                if (ism && (L == 0u || O == 0u || O > q)) {
                    lane_bad = true;
                    break;
                }
                const uint32_t v0 = ism ? q - O : (kLit | b);
                for (uint32_t k = 0; k < L; ++k) s_src[q + k] = (uint16_t)(v0 + ism * k);
                q += L;
                pm += ism;
            }
        }
        uint32_t wr = (!uni && j_lo < j_hi) ? s_fl[j_lo >> 5] : 0u;
        uint32_t pmr = (!uni && j_lo < j_hi) ? s_wp[j_lo >> 5] + __popc(wr & ((1u << (j_lo & 31u)) - 1u)) : 0u;
        for (uint32_t j = uni ? j_hi : j_lo; j < j_hi; ++j) {
            if ((j & 31u) == 0u) wr = s_fl[j >> 5];
            const uint32_t w = wr;
            bool ism = (w >> (j & 31u)) & 1u;
            const uint32_t pm = pmr;
            pmr += ism;
            // single stream: the item's token or literal at b; split: the
            // literal at WS * (literals before it), length and offset bytes
            // at slit + pm and slit + matches + pm
            uint32_t b = split ? (ism ? slit + pm : WS * (j - pm)) : WS * j - (WS - 2u) * pm;
            if (ism) {
                uint32_t L = s_data[b], O = s_data[split ? slit + second + pm : b + 1];
                if (L == 0 || O == 0 || O > q) {
                    lane_bad = true;
                    break;
                }
                if (WS == 1) {
                    const uint32_t s0 = q - O;
                    uint32_t r = 0;
                    for (uint32_t k = 0; k < L; ++k) {
                        const uint32_t t = s0 + r;
                        s_src[q + k] = t >= q_lane ? s_src[t] : (uint16_t)t;
                        r = r + 1u == O ? 0u : r + 1u;
                    }
                } else {
                    for (uint32_t k = 0; k < L; ++k) s_src[q + k] = (uint16_t)(q + k - O);
                }
                q += L;
            } else {
                s_src[q] = (uint16_t)(kLit | b);
                q += 1;
            }
        }
        if (__any_sync(FULL, lane_bad)) {
            if (lane == 0) atomicOr(a.status, kStatCorrupt);
            continue;
        }
        __syncwarp();

        // ---- D5: pointer jumping ----
        // Elements in pairs: one 32-bit shared load and store per two; an
        // unresolved entry follows its pointer by a predicated load and a
        // resolved one loads nothing (no branch; measured +1-3 % decode over
        // a select of the address, which +5-13 % beat skipping resolved pairs
        // by a branch). Entries change only towards their final value, so a
        // concurrent reader sees an old or a new pointer, and both are valid.
        bool unresolved = true;
        uint32_t* s_src2 = reinterpret_cast<uint32_t*>(s_src);
        const uint32_t src_base = (uint32_t)__cvta_generic_to_shared(s_src);
        for (int r = 0; r < kMaxJumpRounds && unresolved; ++r) {
            bool mine = false;
#pragma unroll 4
            for (uint32_t j = lane; j < E / 2u; j += 32) {
                const uint32_t v = s_src2[j];
                uint32_t nlo = v & 0xFFFFu, nhi = v >> 16;
                follow(nlo, src_base);
                follow(nhi, src_base);
                s_src2[j] = nlo | (nhi << 16);
                mine |= (nlo & nhi & kLit) == 0u;
            }
            unresolved = __any_sync(FULL, mine);
            __syncwarp();
        }
        if (unresolved) {
            if (lane == 0) atomicOr(a.status, kStatCorrupt);
            continue;
        }

        // ---- D6: gather and store ----
        write_chunk(out, take, chunk_out_aligned, lane,
                    [s_data, s_src](uint32_t j) { return lit_word<WS>(s_data, s_src, j); });
        __syncwarp();
    }
}

// Parse and validate the stream header (every warp, lanes 0..7 load it).
// Records the reason in the status word (CTA 0, thread 0) and returns false
// when decoding must not proceed.
__device__ bool parse_header(const DecodeArgs& a, Geo& g) {
    const int lane = threadIdx.x & 31;
    uint32_t hw = 0;
    const uint32_t hdr = a.split ? kSplitHeaderBytes : kHeaderBytes;
    const bool hdr_fits = a.in_bytes >= hdr;
    if (lane < (int)(hdr / 4u) && hdr_fits) hw = read_u32(a.in + 4 * lane);
    uint32_t h[12];
#pragma unroll
    for (int k = 0; k < 12; ++k) h[k] = __shfl_sync(FULL, hw, k);
    g.ws = (h[1] >> 16) & 0xFFu;
    g.cs = h[2];
    g.C = h[3];
    g.orig = (uint64_t)h[4] | ((uint64_t)h[5] << 32);
    g.total = (uint64_t)h[6] | ((uint64_t)h[7] << 32);
    g.lit_total = a.split ? ((uint64_t)h[8] | ((uint64_t)h[9] << 32)) : 0;
    g.m_total = a.split ? ((uint64_t)h[10] | ((uint64_t)h[11] << 32)) : 0;
    bool ok = hdr_fits && h[0] == kMagic && (h[1] & 0xFFFFu) == (a.split ? kSplitVersion : kVersion) &&
              (h[1] >> 24) == 0 && valid_geometry((int)g.ws, (int)g.cs);
    if (ok) {
        g.E = g.cs / g.ws;
        ok = (uint64_t)g.C == (g.orig + g.cs - 1) / g.cs;
        g.body0 = (uint64_t)hdr + (uint64_t)kEntryBytes * g.C;
        ok = ok && g.total >= g.body0 && g.total <= a.in_bytes;
        if (a.split)
            ok = ok && g.lit_total <= a.port_len[0] && g.m_total <= a.port_len[1] &&
                 g.m_total <= a.port_len[2];
    }
    if (!ok) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatCorrupt);
        return false;
    }
    if (g.orig != a.n_bytes) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(a.status, kStatSizeMismatch);
        return false;
    }
    return true;
}

// ---- D1: stream offset of every chunk's block (scan of the size table) ----
__global__ void __launch_bounds__(kScanThreads) offsets_kernel(DecodeArgs a) {
    __shared__ TileSmem sm;
    pdl_trigger();  // the decode kernel may be scheduled now
    Geo g;
    if (!parse_header(a, g)) return;
    const int tid = threadIdx.x;
    const uint32_t n_tiles = (g.C + kTile - 1) / kTile;
    for (;;) {
        if (tid == 0) sm.tile = atomicAdd(a.ticket, 1u);
        __syncthreads();
        const uint32_t t = sm.tile;
        if (t >= n_tiles) break;
        const uint32_t c0 = t * kTile;
        if (a.split) {
            // three scans: flag words, literal bytes, matches (an invalid entry
            // counts 0 and fails in the decode kernel)
            uint64_t tot[3];
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const uint64_t prefix = tile_scan(
                    sm, t, g.C, a.tdesc + (uint64_t)k * a.tdesc_stride, a.epoch, a.status, [&](uint32_t c) {
                        const uint8_t* e = a.in + kSplitHeaderBytes + (uint64_t)kEntryBytes * c;
                        const uint32_t items = read_u32(e), m = read_u32(e + 4);
                        uint32_t fw, lit;
                        if (!split_entry(items, m, g, fw, lit)) return 0u;
                        return k == 0 ? fw : (k == 1 ? lit : m);
                    });
                for (uint32_t j = (uint32_t)tid; j < kTile && c0 + j < g.C; j += kScanThreads)
                    a.offsets[3ull * (c0 + j) + k] = prefix + sm.off[j];
                tot[k] = prefix + sm.total;
                __syncthreads();
            }
            if (t == n_tiles - 1 && tid == 0 &&
                (g.body0 + 4ull * tot[0] != g.total || tot[1] != g.lit_total || tot[2] != g.m_total))
                atomicOr(a.status, kStatCorrupt);
            __syncthreads();
            continue;
        }
        const uint64_t prefix = tile_scan(sm, t, g.C, a.tdesc, a.epoch, a.status, [&](uint32_t c) {
            const uint8_t* e = a.in + kHeaderBytes + (uint64_t)kEntryBytes * c;
            const uint32_t b = entry_block(read_u32(e), read_u32(e + 4), g);
            return b == 0xFFFFFFFFu ? 0u : b;
        });
        for (uint32_t j = (uint32_t)tid; j < kTile && c0 + j < g.C; j += kScanThreads)
            a.offsets[c0 + j] = g.body0 + prefix + sm.off[j];
        if (t == n_tiles - 1 && tid == 0 && g.body0 + prefix + sm.total != g.total)
            atomicOr(a.status, kStatCorrupt);
        __syncthreads();
    }
}

// ---- D2..D6: decode, one chunk per warp ----
__global__ void __launch_bounds__(kDecWarps * 32) decode_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    pdl_wait();  // the block offsets
    Geo g;
    if (!parse_header(a, g)) return;
    const DecSlot S = dec_slot(g.cs, g.E);
    const int slots = (int)(kDecSmem / S.total) < kDecWarps ? (int)(kDecSmem / S.total) : kDecWarps;
    if (warp >= slots) return;
    uint8_t* slot = smem + (size_t)warp * S.total;
    const uint32_t first = (uint32_t)warp * gridDim.x + blockIdx.x;  // spread over the SMs
    const uint32_t n_warps = gridDim.x * (uint32_t)slots;
    if (g.ws == 4)
        decode_chunks<4>(a, g, slot, lane, first, n_warps);
    else if (g.ws == 2)
        decode_chunks<2>(a, g, slot, lane, first, n_warps);
    else
        decode_chunks<1>(a, g, slot, lane, first, n_warps);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream) {
    // launch shape of the device last used by this host thread
    static thread_local int configured_dev = -1;
    static thread_local int grid_cache = 0;
    static thread_local int sms_cache = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_dev != dev) {
        err = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kDecSmem);
        if (err != cudaSuccess) return err;
        int sms = 0, per_sm = 0;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return err;
        if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel,
                                                                 kDecWarps * 32, kDecSmem)) !=
            cudaSuccess)
            return err;
        grid_cache = sms * (per_sm < 1 ? 1 : per_sm);
        sms_cache = sms;
        configured_dev = dev;
    }
    // Chunks per stream are bounded by n_bytes / 1024 (the smallest chunk).
    const uint64_t max_chunks = (a.n_bytes + 1023u) / 1024u;
    uint64_t tgrid = (max_chunks + kTile - 1) / kTile;
    if (tgrid > (uint64_t)sms_cache * 4u) tgrid = (uint64_t)sms_cache * 4u;
    if (tgrid < 1) tgrid = 1;
    offsets_kernel<<<(unsigned)tgrid, kScanThreads, 0, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const uint64_t max_ctas = (max_chunks + kDecWarps - 1) / kDecWarps;
    uint64_t grid = (uint64_t)grid_cache;
    if (grid > max_ctas) grid = max_ctas;
    if (grid < 1) grid = 1;
    const KernelEvents ev = kernel_events();
    if (ev.start && (err = cudaEventRecord(ev.start, stream)) != cudaSuccess) return err;
    if ((err = pdl_launch(decode_kernel, dim3((unsigned)grid), dim3(kDecWarps * 32), kDecSmem, stream, a)) !=
        cudaSuccess)
        return err;
    if (ev.stop && (err = cudaEventRecord(ev.stop, stream)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace gpulz
