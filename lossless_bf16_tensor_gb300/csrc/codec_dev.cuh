// Device building blocks of the LCT codec for sm_103a: byte split and join,
// the per-stream coder and decoder, block-wide scans and the bounded
// decoupled look-back that places each block's overflow bytes.
//
// Sources: [EXP] "LCT paper -- Lossless Huffman coding of BF16 training
// tensors -- What does it mean?", paragraphs "In bits" (byte split, 8-bit
// capped codes, escape + 8-bit literal, shift) and "Compressing is easy"
// (blocks, 256 round-robin streams of fixed length, overflow + marker).
#pragma once

#include <cstdint>

#include "internal.h"

namespace lct {
namespace dev {

template <int LEVEL>
struct Geo;
template <>
struct Geo<LCT_LEVEL_CLEAN> {
    static constexpr int B = 65536, W = 25, NJ = 256;
};
template <>
struct Geo<LCT_LEVEL_MEDIUM> {
    static constexpr int B = 32768, W = 16, NJ = 128;
};
template <>
struct Geo<LCT_LEVEL_HIGH> {
    static constexpr int B = 32768, W = 20, NJ = 128;
};

// Exponents of a block are staged in shared memory as rows of 256 (one symbol
// of every stream); a row is padded to 260 bytes so that a warp walking one
// stream down the rows hits 32 different banks.
constexpr int kRow = 260;

// Shared-memory carve-up; every region starts on a 128-byte boundary so that
// 16-byte vector accesses to the regions after the staging rows stay aligned.
template <int LEVEL>
struct Smem {
    static constexpr int kExpBytes = ((Geo<LEVEL>::NJ + 1) * kRow + 127) / 128 * 128;  // + guard row
    static constexpr int kSlotBytes = (Geo<LEVEL>::W + 1) * kStreams * 4;              // + zero row
    static_assert(kExpBytes % 128 == 0 && kSlotBytes % 128 == 0, "regions must stay 16-byte aligned");
};

__device__ __forceinline__ void latch(lct_header *h, uint32_t code)
{
    atomicCAS(&h->status, 0u, code);
}

// ------------------------------------------------------------ byte split

// Eight BF16 values (one uint4, little endian) -> 8 sign-fraction bytes and
// 8 exponent bytes, in element order.  High byte of a BF16 = sign | e[7:1],
// low byte = e[0] | fraction.
__device__ __forceinline__ void split8(const uint4 v, uint2 &sf, uint2 &ex)
{
    uint32_t hb = __byte_perm(v.x, v.y, 0x7531), lb = __byte_perm(v.x, v.y, 0x6420);
    ex.x = ((hb << 1) & 0xFEFEFEFEu) | ((lb >> 7) & 0x01010101u);
    sf.x = (hb & 0x80808080u) | (lb & 0x7F7F7F7Fu);
    hb = __byte_perm(v.z, v.w, 0x7531);
    lb = __byte_perm(v.z, v.w, 0x6420);
    ex.y = ((hb << 1) & 0xFEFEFEFEu) | ((lb >> 7) & 0x01010101u);
    sf.y = (hb & 0x80808080u) | (lb & 0x7F7F7F7Fu);
}

__device__ __forceinline__ uint4 join8(const uint2 sf, const uint2 ex)
{
    uint4 v;
    uint32_t hb = (sf.x & 0x80808080u) | ((ex.x >> 1) & 0x7F7F7F7Fu);
    uint32_t lb = ((ex.x << 7) & 0x80808080u) | (sf.x & 0x7F7F7F7Fu);
    v.x = __byte_perm(lb, hb, 0x5140);
    v.y = __byte_perm(lb, hb, 0x7362);
    hb = (sf.y & 0x80808080u) | ((ex.y >> 1) & 0x7F7F7F7Fu);
    lb = ((ex.y << 7) & 0x80808080u) | (sf.y & 0x7F7F7F7Fu);
    v.z = __byte_perm(lb, hb, 0x5140);
    v.w = __byte_perm(lb, hb, 0x7362);
    return v;
}

__device__ __forceinline__ uint8_t exp_of(uint16_t h) { return (uint8_t)((h >> 7) & 0xFF); }
__device__ __forceinline__ uint8_t sf_of(uint16_t h) { return (uint8_t)(((h >> 8) & 0x80) | (h & 0x7F)); }
__device__ __forceinline__ uint16_t join1(uint8_t sf, uint8_t e)
{
    return (uint16_t)(((uint32_t)(sf & 0x80) << 8) | ((uint32_t)e << 7) | (sf & 0x7F));
}

// Staged exponents of in-block group g (8 values, row g/32, column 8*(g%32)).
__device__ __forceinline__ uint8_t *stage_at(uint8_t *e_s, uint32_t i)
{
    return e_s + (i >> 8) * kRow + (i & 255);
}

// --------------------------------------------------------- code tables

// Encode table for shift delta: entry e = {code left-aligned in 32 bits, bit
// count}.  Symbol s = e - delta gets its own code when it has one; any other
// exponent costs the escape prefix plus the raw 8-bit exponent.
__device__ __forceinline__ uint2 enc_entry(const DevCodebook &cb, int delta, int e)
{
    const int s = e - delta;
    uint32_t code, len;
    if (s >= 0 && s <= 255 && cb.len[s] != 0) {
        code = cb.code[s];
        len = cb.len[s];
    } else {
        code = ((uint32_t)cb.esc_code << 8) | (uint32_t)e;
        len = cb.esc_len + 8u;
    }
    return make_uint2(code << (32u - len), len);
}

// Decode table for shift delta, by 8-bit window: bits 0..7 exponent (coded
// symbols), 8..15 bits consumed, 16..23 literal offset, bit 24 escape.
__device__ __forceinline__ uint32_t dec_entry(const DevCodebook &cb, int delta, int v)
{
    const uint32_t d = cb.dec[v], sym = d & 0x1FF, l = d >> 12;
    if (sym == 256) return (1u << 24) | (l << 16) | ((l + 8u) << 8);
    return (l << 8) | ((sym + (uint32_t)delta) & 0xFFu);
}

// ------------------------------------------------------ stream coding

// Code stream j: its symbols are column j of the staged rows.  Codes are
// appended most significant bit first while they fit the W-word slot; the
// first code that does not fit ends the slot (the marker).  Writes every slot
// word (unused bits zero) at slot_col[w * 256].  Returns the marker.
template <int W, int NJ>
__device__ __forceinline__ uint32_t encode_stream(const uint8_t *__restrict__ col, uint32_t nj,
                                                  const uint2 *__restrict__ tbl,
                                                  uint32_t *__restrict__ slot_col)
{
    uint32_t hi = 0, nbits = 0, wi = 0, rem = 32u * W, marker = nj;
    const uint32_t count = NJ > 0 ? (uint32_t)NJ : nj;
#pragma unroll 8
    for (uint32_t k = 0; k < count; ++k) {
        const uint2 ent = tbl[col[k * kRow]];
        if (ent.y > rem) {
            marker = k;
            break;
        }
        rem -= ent.y;
        const uint32_t merged = hi | (ent.x >> nbits);
        nbits += ent.y;
        if (nbits >= 32u) {
            slot_col[wi * kStreams] = merged;
            ++wi;
            hi = ent.x << (32u - (nbits - ent.y));
            nbits -= 32u;
        } else {
            hi = merged;
        }
    }
    if (wi < (uint32_t)W) {
        slot_col[wi * kStreams] = hi;
        for (uint32_t w = wi + 1; w < (uint32_t)W; ++w) slot_col[w * kStreams] = 0u;
    }
    return marker;
}

// Decode `count` symbols of one stream from its slot image (W words plus a
// zero guard word) into column j of the staged rows.  Returns the bits
// consumed; more than 32*W means the slot was corrupt (reads stay in the
// image because the word index is clamped).
template <int W>
__device__ __forceinline__ uint32_t decode_stream(const uint32_t *__restrict__ slot_col, uint32_t count,
                                                  const uint32_t *__restrict__ lut,
                                                  uint8_t *__restrict__ col)
{
    uint32_t p = 0;
#pragma unroll 4
    for (uint32_t k = 0; k < count; ++k) {
        const uint32_t w = min(p >> 5, (uint32_t)(W - 1));
        const uint32_t hiw = slot_col[w * kStreams], low = slot_col[(w + 1) * kStreams];
        const uint32_t win = __funnelshift_l(low, hiw, p);
        const uint32_t ent = lut[win >> 24];
        const uint32_t lit = (win << ((ent >> 16) & 0xFFu)) >> 24;
        col[k * kRow] = (uint8_t)((ent & (1u << 24)) ? lit : ent);
        p += (ent >> 8) & 0xFFu;
    }
    return p;
}

// ------------------------------------------------------------- scans

// Exclusive scan of one value per thread over `nthreads` consecutive threads
// starting at warp `first_warp` (nthreads a multiple of 32, at most 1024).
// `warp_tot` holds one word per warp.  Returns the exclusive prefix; *total
// gets the sum.  Must be called by all threads of the group; contains
// __syncthreads() so the whole CTA must call it.
__device__ __forceinline__ uint32_t group_exclusive_scan(uint32_t v, uint32_t *warp_tot, int group_warps,
                                                         int first_warp, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    uint32_t before = 0, sum = 0;
    for (int w = 0; w < group_warps; ++w) {
        const uint32_t t = warp_tot[first_warp + w];
        if (first_warp + w < warp) before += t;
        sum += t;
    }
    *total = sum;
    __syncthreads();
    return before + inc - v;
}

// ------------------------------------------------ decoupled look-back

constexpr unsigned long long kFlagAgg = 1ull << 62;  // block total published
constexpr unsigned long long kFlagInc = 2ull << 62;  // inclusive prefix published
constexpr unsigned long long kValMask = (1ull << 62) - 1;

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// independent prologue, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// One thread of block b: publish the block's overflow byte count, add up the
// predecessors' counts (stopping at the first inclusive prefix), publish the
// inclusive prefix and return the exclusive one.  Every wait is bounded by
// wait_ns of %globaltimer and an iteration cap; on expiry *timed_out is set
// and the prefix found so far is used, so later blocks are never stuck.
static __device__ __noinline__ unsigned long long lookback(unsigned long long *status, uint32_t b,
                                                     unsigned long long total, uint64_t wait_ns,
                                                     bool *timed_out)
{
    *timed_out = false;
    if (b == 0) {
        st_release(&status[0], kFlagInc | total);
        return 0;
    }
    st_release(&status[b], kFlagAgg | total);
    unsigned long long excl = 0;
    const uint64_t t0 = global_ns();
    uint32_t spins = 0;
    int64_t pred = (int64_t)b - 1;
    while (pred >= 0) {
        const unsigned long long v = ld_acquire(&status[pred]);
        const unsigned long long flag = v & ~kValMask;
        if (flag == 0) {
            ++spins;
            if (spins > (1u << 26) || ((spins & 63u) == 0 && global_ns() - t0 > wait_ns)) {
                *timed_out = true;
                break;
            }
            __nanosleep(64);
            continue;
        }
        excl += v & kValMask;
        if (flag == kFlagInc) break;
        --pred;
    }
    st_release(&status[b], kFlagInc | ((excl + total) & kValMask));
    return excl;
}

}  // namespace dev
}  // namespace lct
