// Device building blocks of the LCT codec for sm_103a: byte split and join,
// per-stream coding and decoding, block-wide scans, TMA bulk copies with
// bounded mbarrier waits, and the bounded decoupled look-back that places
// each block's overflow bytes.
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

// Staged exponent rows hold one symbol of every stream; a row is padded to
// 260 bytes so that a warp walking one stream down the rows hits 32 banks.
constexpr int kRow = 260;
constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ void latch(lct_header *h, uint32_t code) { atomicCAS(&h->status, 0u, code); }

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------ byte split

__device__ __forceinline__ uint8_t exp_of(uint32_t h) { return (uint8_t)((h >> 7) & 0xFF); }
__device__ __forceinline__ uint8_t sf_of(uint32_t h) { return (uint8_t)(((h >> 8) & 0x80) | (h & 0x7F)); }

// --------------------------------------------------------- code tables

// Encode table for shift delta: entry e = {code left-aligned in 32 bits, bit
// count}.  Symbol s = e - delta gets its own code when it has one; any other
// exponent costs the escape prefix plus the raw 8-bit exponent.  With a zero
// atom, exponent 0 is symbol 0 whatever the shift, and a nonzero exponent
// the shift maps onto symbol 0 escapes.
__device__ __forceinline__ uint2 enc_entry(const DevCodebook &cb, int delta, int e)
{
    int s = e - delta;
    if (cb.zero_atom) s = e == 0 ? 0 : (s == 0 ? -1 : s);
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

// The encode-table entry of a BF16 value h (bits 0..15, higher bits zero):
// entry exp_of(h), addressed by its byte offset ((h >> 7) & 0xFF) * 8 in one
// shift and one mask.
__device__ __forceinline__ uint2 code_of(const uint2 *__restrict__ tbl, uint32_t h)
{
    return *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(tbl) + ((h >> 4) & 0x7F8u));
}

// Decode table for shift delta, indexed by the next 8 bits of the stream:
//   bits  0..4   s: a left funnel shift of (0 : window) by s brings the
//                escape literal to bits 7..14 (s = 15 + escape length); 0
//                for a coded symbol, which yields 0
//   bits  7..14  the exponent, for a symbol with its own code (0 for escape)
//   bits 27..31  bits consumed (code length, or escape length + 8)
__device__ __forceinline__ uint32_t dec_entry(const DevCodebook &cb, int delta, int v)
{
    const uint32_t d = cb.dec[v], sym = d & 0x1FF, l = d >> 12;
    if (sym == 256) return ((l + 8u) << 27) | (15u + l);
    const uint32_t e = cb.zero_atom && sym == 0 ? 0u : (sym + (uint32_t)delta) & 0xFFu;
    return (l << 27) | (e << 7);
}

// The escape literal of a table entry's symbol at the head of `win` in bits
// 7..14 (bits above are to be ignored), or 0 for a coded symbol: the
// funnel shift takes its amount from the entry's low 5 bits.
__device__ __forceinline__ uint32_t esc_literal(uint32_t win, uint32_t ent)
{
    return __funnelshift_l(win, 0u, ent);
}

// ------------------------------------------------------ stream decoding

// One symbol of a stream read most significant bit first from its slot image
// column (word w at col[w * 256]); p is the bit position, advanced past the
// symbol.  Returns the exponent in bits 7..14 (other bits are to be ignored).
// The word index is clamped to the slot and the image has a zero guard row
// after it, so a corrupt stream never reads outside the image (it shows up as
// p > 32*W instead).
template <int W>
__device__ __forceinline__ uint32_t rd_take(uint32_t &p, const uint32_t *__restrict__ col,
                                            const uint32_t *__restrict__ lut)
{
    const uint32_t w = min(p >> 5, (uint32_t)(W - 1));
    const uint32_t hi = col[w * kStreams], lo = col[(w + 1) * kStreams];
    const uint32_t win = __funnelshift_l(lo, hi, p);  // the next 32 bits
    const uint32_t ent = lut[win >> 24];
    p += ent >> 27;
    return ent | esc_literal(win, ent);
}

// ------------------------------------------- pair reader, deferred literal

// Shared-memory loads by 32-bit shared address.
__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// a * b + c on the FMA pipe.  The multipliers below are powers of two that
// the kernels receive as launch arguments: a constant one would be folded
// into a shift on the integer ALU pipe, which is the busiest pipe of the
// decoders.
__device__ __forceinline__ uint32_t imad(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Runtime multipliers: x = 32 (bit position -> byte offset of a slot word
// row, (p & 0x3E0) * 32 = (p >> 5) * 1024), y = 4 (table index -> byte
// offset), z = 0x01010000 (a sign-fraction byte into bytes 2 and 3).
struct Mul {
    uint32_t x, y, z;
};

// One input stream for the pair reader: bit position and the shared address
// of the stream's column in the slot image (word w at col + 1024 * w).
struct Rd {
    uint32_t p, col;
};

// Two symbols at bit p, with the escape literals left out: ent0 and ent1 are
// the decode-table entries (exponent in bits 7..14 for a coded symbol, 0 for
// an escape, whose literal shift is in bits 0..4) and w0, w1 the 32-bit
// windows at each symbol, from which lit_fix recovers a literal.  A warp
// pays for the literals only when one of its lanes met an escape.  The word
// index is taken modulo 32: a position past the slot only arises from
// corrupt data, whose reads then stay inside the CTA's shared memory (every
// kernel keeps 33 KB from each slot image on), and the final position check
// reports it.
__device__ __forceinline__ void rd_pair(Rd &r, uint32_t lut, const Mul m, uint32_t &w0, uint32_t &w1, uint32_t &ent0,
                                        uint32_t &ent1)
{
    const uint32_t a = imad(r.p & 0x3E0u, m.x, r.col);
    const uint32_t hi = lds32(a), lo = lds32(a + kStreams * 4);
    w0 = __funnelshift_l(lo, hi, r.p);  // the next 32 bits
    ent0 = lds32(imad(w0 >> 24, m.y, lut));
    const uint32_t l0 = ent0 >> 27;
    w1 = w0 << l0;
    ent1 = lds32(imad(w1 >> 24, m.y, lut));
    r.p += l0 + (ent1 >> 27);
}

// A decode-table entry with its escape literal added (exponent in bits 7..14).
__device__ __forceinline__ uint32_t lit_fix(uint32_t w, uint32_t ent) { return ent | esc_literal(w, ent); }

// Nonzero when an entry decodes an escape (its literal shift is not 0).
__device__ __forceinline__ uint32_t esc_bits(uint32_t ent_or) { return ent_or & 31u; }

// Two float32 results -> two BF16 (round to nearest even, subnormals kept)
// packed lo | hi << 16; a NaN half becomes this library's NaN 0x7FC0 (the
// conversion writes 0x7FFF; the NaN test sets a half to 0xFFFF, and 0x7FFF
// exclusive-or 0x003F is 0x7FC0).
__device__ __forceinline__ uint32_t bf16x2_rne(float lo, float hi)
{
    uint32_t d, nan;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    asm("set.nan.u32.bf16x2 %0, %1, %1;" : "=r"(nan) : "r"(d));
    return d ^ (nan & 0x003F003Fu);
}

// ------------------------------ float-ready decode table (update kernels)

// A second decode-table layout for the kernels that compute on the values,
// indexed like dec_entry by the next 8 bits of the stream:
//   bits  0..4   L: bits consumed (code length, or escape length + 8)
//   bits  5..9   zero
//   bits 10..14  literal shift: escape length - 1 for an escape (a left
//                shift of the window by it brings the literal to bits
//                23..30), 31 for a coded symbol (the shifted window then
//                keeps nothing below bit 31)
//   bit  15      an escape, or a coded exponent of 255 (the warp takes the
//                path that adds literals and canonicalises NaN)
//   bits 23..30  the exponent, for a symbol with its own code (0 for escape)
// Every field the position update does not want sits at bit 10 or above, so
// the position may be advanced by the raw entries: its low 10 bits (all the
// reader uses: word index and shift) stay exact, and the true advance over a
// few symbols is (p_after - p_before) & 0x3FF.  The exponent sits where a
// float32 has it, so joining it with its sign-fraction byte gives the
// float32 bits of the BF16 value in one logic operation (join_f).
constexpr uint32_t kEntFlag = 0x8000u;

__device__ __forceinline__ uint32_t dec_entry_f(const DevCodebook &cb, int delta, int v)
{
    const uint32_t d = cb.dec[v], sym = d & 0x1FF, l = d >> 12;
    if (sym == 256) return kEntFlag | (((l - 1u) & 31u) << 10) | (l + 8u);
    const uint32_t e = cb.zero_atom && sym == 0 ? 0u : (sym + (uint32_t)delta) & 0xFFu;
    return (e << 23) | (e == 255u ? kEntFlag : 0u) | (31u << 10) | l;
}

// Two symbols at bit p with raw entries (see dec_entry_f); w0, w1 are the
// windows at each symbol for lit_fix_f.  The second window is the first one
// shifted by the first symbol's length, taken from the entry's low 5 bits by
// the funnel shift itself; the position is advanced by the raw entries.  Word
// indices are taken modulo 32 as in rd_pair.
__device__ __forceinline__ void rd_pair_f(Rd &r, uint32_t lut, const Mul m, uint32_t &w0, uint32_t &w1, uint32_t &ent0,
                                          uint32_t &ent1)
{
    const uint32_t a = imad(r.p & 0x3E0u, m.x, r.col);
    const uint32_t hi = lds32(a), lo = lds32(a + kStreams * 4);
    w0 = __funnelshift_l(lo, hi, r.p);  // the next 32 bits
    ent0 = lds32(imad(w0 >> 24, m.y, lut));
    w1 = __funnelshift_l(0u, w0, ent0);  // w0 << L0
    ent1 = lds32(imad(w1 >> 24, m.y, lut));
    r.p = r.p + ent0 + ent1;
}

// One symbol at exact bit p of a slot image column (word w at col[w * 256]),
// for the checked paths: the entry with its literal added; p advanced
// exactly.  The word index is clamped to the slot (zero guard row after it).
template <int W>
__device__ __forceinline__ uint32_t rd_take_f(uint32_t &p, const uint32_t *__restrict__ col,
                                              const uint32_t *__restrict__ lut)
{
    const uint32_t w = min(p >> 5, (uint32_t)(W - 1));
    const uint32_t hi = col[w * kStreams], lo = col[(w + 1) * kStreams];
    const uint32_t win = __funnelshift_l(lo, hi, p);
    const uint32_t ent = lut[win >> 24];
    p += ent & 31u;
    return ent | __funnelshift_l(0u, win, ent >> 10);
}

// The entry with its escape literal added in bits 23..30 (a coded symbol's
// shift of 31 only touches bit 31, which join_f ignores).
__device__ __forceinline__ uint32_t lit_fix_f(uint32_t w, uint32_t ent)
{
    return ent | __funnelshift_l(0u, w, ent >> 10);
}

// float32 bits of the BF16 value with sign-fraction byte sf and the entry's
// exponent: sf * 0x01010000 (mz) puts the sign at bit 31 and the fraction at
// bits 16..22, and one logic operation takes bits 23..30 from the entry.
__device__ __forceinline__ uint32_t join_f(uint32_t sf, uint32_t ent, uint32_t mz)
{
    return (ent & 0x7F800000u) | (imad(sf, mz, 0u) & 0x807FFFFFu);
}

// Two float32 results -> two BF16 (round to nearest even, subnormals kept)
// packed lo | hi << 16, with NaN left as the conversion writes it (0x7FFF);
// nan_canon2 turns such halves into this library's 0x7FC0.
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}
__device__ __forceinline__ uint32_t nan_canon2(uint32_t d)
{
    uint32_t nan;
    asm("set.nan.u32.bf16x2 %0, %1, %1;" : "=r"(nan) : "r"(d));
    return d ^ (nan & 0x003F003Fu);
}

// Sign-fraction bytes of two packed BF16 values, in byte 0 and byte 2 (the
// other bytes are to be ignored).
__device__ __forceinline__ uint32_t sf_of2(uint32_t p) { return ((p >> 8) & 0x00800080u) | (p & 0xFF7FFF7Fu); }

// ------------------------------------------------------- stream coding

// Appends codes most significant bit first into one stream's W-word slot
// image (word w at col[w * 256]) until the first code that does not fit; that
// symbol's index is the marker.  Every append (of at most 32 bits) is
// followed by a flush, so before an append fewer than 32 bits are pending and
// they all sit in `hi`; an append ORs the code's head into `hi` and leaves the
// bits that run past the word in `lo`, which a flush moves up.  `rem`, the
// bits the slot still has room for, is kept exact: the unchecked paths
// subtract what they appended.
struct Writer {
    uint32_t hi, lo, nbits, wi, rem, marker;
    bool alive;
};

template <int W>
__device__ __forceinline__ void wr_init(Writer &w, uint32_t nj)
{
    w.hi = 0;
    w.lo = 0;
    w.nbits = 0;
    w.wi = 0;
    w.rem = 32u * W;
    w.marker = nj;
    w.alive = true;
}

// Append one code (left-aligned in ent.x, ent.y <= 32 bits); nbits < 32.
__device__ __forceinline__ void wr_add(Writer &w, const uint2 ent)
{
    w.hi |= ent.x >> w.nbits;
    w.lo = __funnelshift_r(0u, ent.x, w.nbits);  // low word of (ent.x : 0) >> nbits; 0 when nbits = 0
    w.nbits += ent.y;
}

// Append two codes (together at most 32 bits) with one accumulator update:
// the pair is assembled in one register first.
__device__ __forceinline__ void wr_add2(Writer &w, const uint2 a, const uint2 b)
{
    wr_add(w, make_uint2(a.x | (b.x >> a.y), a.y + b.y));
}

// Write out the current word if it is complete (leaves nbits < 32).
__device__ __forceinline__ void wr_flush(Writer &w, uint32_t *__restrict__ col)
{
    if (w.nbits >= 32u) {
        col[w.wi * kStreams] = w.hi;
        ++w.wi;
        w.hi = w.lo;
        w.nbits -= 32u;
    }
}

// Append with the fit check; returns true when symbol k spilled (it, and
// every later symbol of the stream, goes to the overflow region).
__device__ __forceinline__ bool wr_put_checked(Writer &w, const uint2 ent, uint32_t k, uint32_t *col)
{
    if (w.alive && ent.y <= w.rem) {
        w.rem -= ent.y;
        wr_add(w, ent);
        wr_flush(w, col);
        return false;
    }
    if (w.alive) {
        w.alive = false;
        w.marker = k;
    }
    return true;
}

// Write the partly filled word and zero the rest of the slot.
template <int W>
__device__ __forceinline__ void wr_finish(const Writer &w, uint32_t *col)
{
    if (w.wi < (uint32_t)W) {
        col[w.wi * kStreams] = w.hi;
        for (uint32_t i = w.wi + 1; i < (uint32_t)W; ++i) col[i * kStreams] = 0u;
    }
}

// ------------------------------------------------------------ join

// One sign-fraction byte + an exponent in bits 7..14 (other bits ignored) ->
// one BF16 in bits 0..15 (bits 16 and up are to be ignored).  sf * 0x101 puts
// the sign at bit 15 and keeps the fraction in bits 0..6.
__device__ __forceinline__ uint32_t join_one(uint32_t sf, uint32_t e)
{
    return ((sf * 0x101u) & 0x807Fu) | (e & 0xFFFF7F80u);
}

// float32 -> BF16 (bits 0..15), round to nearest even, subnormals kept.  The
// conversion writes NaN as 0x7FFF; this library's NaN is 0x7FC0.
__device__ __forceinline__ uint32_t bf16_rne(float r)
{
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(r));
    return h == 0x7FFFu ? 0x7FC0u : (uint32_t)h;
}

// BF16 in bits 0..15 -> float32 (exact).
__device__ __forceinline__ float bf16_f(uint32_t h) { return __uint_as_float(h << 16); }

// ------------------------------------------------------------- scans

// Barrier over the CTA (BAR = 0) or over the first NT threads of the CTA on
// named barrier BAR (the consumer warps of a warp-specialised kernel, whose
// producer warp does not take part).
template <int BAR = 0, int NT = 0>
__device__ __forceinline__ void cta_sync()
{
    if constexpr (BAR == 0)
        __syncthreads();
    else
        asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

// Exclusive scan of one value per thread over `group_warps` warps starting at
// warp `first_warp`; *total gets the group's sum.  Contains two barriers
// (cta_sync<BAR, NT>), so every thread taking part in them must call it.
template <int BAR = 0, int NT = 0>
__device__ __forceinline__ uint32_t group_exclusive_scan(uint32_t v, uint32_t *warp_tot, int group_warps,
                                                         int first_warp, uint32_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    cta_sync<BAR, NT>();
    uint32_t before = 0, sum = 0;
    for (int w = 0; w < group_warps; ++w) {
        const uint32_t t = warp_tot[first_warp + w];
        if (first_warp + w < warp) before += t;
        sum += t;
    }
    *total = sum;
    cta_sync<BAR, NT>();
    return before + inc - v;
}

// ------------------------------------------- TMA bulk copies, mbarriers

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make initialised mbarriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// One arrival (consumer release of a ring slot).
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, giving up after limit_ns of
// %globaltimer.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try(bar, parity)) return true;
        if ((i & 15u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// Global -> shared bulk copy (TMA, no tensor map); completes on `bar`.  Both
// addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Shared -> global bulk copy, tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (before a bulk store reads them).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Thread-block clusters: a barrier over every thread of the cluster (release
// and acquire: shared-memory writes before it are visible to the cluster's
// reads after it), and a read of a peer CTA's shared memory.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ld_peer_shared(const void *local, uint32_t rank)
{
    uint32_t remote, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
    return v;
}

// Programmatic dependent launch: let the next kernel in the stream start its
// independent work, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------ decoupled look-back

// A block's status word (one per block, in the tensor's scratch region):
//   bits 62..63  0: nothing published yet, 1: the block's own overflow
//                count, 2: the block's inclusive prefix
//   bits 41..61  the block's own overflow count (at most 65,536 bytes)
//   bits  0..40  the count (flag 1) or the inclusive prefix (flag 2)
// Every word carries the block's own count, so the block offsets can also be
// computed from the words afterwards (k_block_offsets), whatever mix of
// flags the blocks left.
constexpr unsigned long long kFlagAgg = 1ull << 62;  // block count published
constexpr unsigned long long kFlagInc = 2ull << 62;  // inclusive prefix published
constexpr unsigned long long kValMask = (1ull << 41) - 1;
constexpr int kOwnShift = 41;
constexpr unsigned long long kOwnMask = (1ull << 21) - 1;

__device__ __forceinline__ unsigned long long status_word(unsigned long long flag, unsigned long long own,
                                                          unsigned long long value)
{
    return flag | ((own & kOwnMask) << kOwnShift) | (value & kValMask);
}

// A status word is read and written whole (one aligned 64-bit access) and
// carries everything a successor uses from it: the flag and the counts.  No
// other data is handed over through it, so relaxed accesses at GPU scope are
// enough; a release would first have to make every earlier global store of
// the CTA (its sign-fraction bytes and markers) visible.
__device__ __forceinline__ unsigned long long ld_status(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_status(unsigned long long *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Blocks below kAllPrev take every predecessor's own count at once: at most
// kAllPrev / 32 loads per lane, all in flight together.
constexpr uint32_t kAllPrev = 320;

// A warp whose streams each spilled at most this many symbols writes its
// overflow bytes lane by lane (each lane its own stream's run); otherwise one
// stream at a time with the lanes over its symbols (coalesced for long runs).
constexpr uint32_t kFewSpills = 8;

// One full warp of block b < kAllPrev: publish the block's overflow byte
// count, wait until every predecessor has published (each status word carries
// its block's own count, whatever its flag), add all their counts in one
// round, and publish the inclusive prefix.  When the blocks finish at nearly
// the same time (a grid that fits the GPU at once) this takes one round of
// loads after the last predecessor publishes, where walking back to the
// nearest inclusive prefix takes one round per window of 32 blocks that has
// none yet.  Every wait is bounded as in warp_lookback_walk.
__device__ __forceinline__ unsigned long long warp_lookback_all(unsigned long long *status, uint32_t b,
                                                                unsigned long long total, uint64_t wait_ns,
                                                                bool *timed_out)
{
    const int lane = threadIdx.x & 31;
    *timed_out = false;
    if (b == 0) {
        if (lane == 0) st_status(&status[0], status_word(kFlagInc, total, total));
        return 0;
    }
    if (lane == 0) st_status(&status[b], status_word(kFlagAgg, total, total));
    const uint64_t t0 = global_ns();
    uint32_t spins = 0;
    unsigned long long sum;
    for (;;) {
        unsigned long long v[kAllPrev / 32];
#pragma unroll
        for (int k = 0; k < (int)(kAllPrev / 32); ++k) {
            const uint32_t idx = (uint32_t)lane + 32u * k;
            v[k] = idx < b ? ld_status(&status[idx]) : kFlagInc;  // beyond b: ready, own count 0
        }
        bool ready = true;
        sum = 0;
#pragma unroll
        for (int k = 0; k < (int)(kAllPrev / 32); ++k) {
            ready = ready && (v[k] >> 62) != 0;
            sum += (v[k] >> kOwnShift) & kOwnMask;
        }
        if (__all_sync(kFull, ready)) break;
        ++spins;
        if (spins > (1u << 24) || ((spins & 63u) == 0 && global_ns() - t0 > wait_ns)) {
            *timed_out = true;
            break;
        }
        __nanosleep(32);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
    if (lane == 0) st_status(&status[b], status_word(kFlagInc, total, sum + total));
    return sum;
}

// One full warp of block b: publish the block's overflow byte count, then
// read the status words of the 32 nearest predecessors at once, add their
// counts up to the nearest published inclusive prefix, and move 32 further
// back while none is found.  Publishes the inclusive prefix and returns the
// exclusive one (same value in every lane).  Every wait is bounded by wait_ns
// of %globaltimer and an iteration cap; on expiry *timed_out is set and the
// prefix found so far is used, so later blocks are never stuck.
static __device__ __noinline__ unsigned long long warp_lookback_walk(unsigned long long *status, uint32_t b,
                                                                     unsigned long long total, uint64_t wait_ns,
                                                                     bool *timed_out)
{
    const int lane = threadIdx.x & 31;
    *timed_out = false;
    if (b == 0) {
        if (lane == 0) st_status(&status[0], status_word(kFlagInc, total, total));
        return 0;
    }
    if (lane == 0) st_status(&status[b], status_word(kFlagAgg, total, total));
    unsigned long long excl = 0;
    int64_t nearest = (int64_t)b - 1;
    const uint64_t t0 = global_ns();
    uint32_t spins = 0;
    for (;;) {
        const int64_t idx = nearest - lane;
        const unsigned long long v = idx >= 0 ? ld_status(&status[idx]) : kFlagInc;
        const uint32_t flag = (uint32_t)(v >> 62);
        const uint32_t inc = __ballot_sync(kFull, flag == 2u);
        const uint32_t not_ready = __ballot_sync(kFull, flag == 0u);
        const uint32_t upto = inc ? ((inc & (0u - inc)) << 1) - 1u : kFull;  // lanes up to the nearest inclusive
        if (not_ready & upto) {
            ++spins;
            if (spins > (1u << 24) || ((spins & 63u) == 0 && global_ns() - t0 > wait_ns)) {
                *timed_out = true;
                break;
            }
            __nanosleep(32);
            continue;
        }
        unsigned long long mine = ((upto >> lane) & 1u) ? (v & kValMask) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(kFull, mine, o);
        excl += mine;
        if (inc) break;
        nearest -= 32;
    }
    if (lane == 0) st_status(&status[b], status_word(kFlagInc, total, excl + total));
    return excl;
}

// The exclusive overflow prefix of block b (see warp_lookback_all and
// warp_lookback_walk); the inclusive one is published for later blocks.
__device__ __forceinline__ unsigned long long warp_lookback(unsigned long long *status, uint32_t b,
                                                           unsigned long long total, uint64_t wait_ns,
                                                           bool *timed_out)
{
    if (b < kAllPrev) return warp_lookback_all(status, b, total, wait_ns, timed_out);
    return warp_lookback_walk(status, b, total, wait_ns, timed_out);
}

// For a block with no overflow bytes when the offsets are computed
// afterwards (deferred placement): publish the count (0), then look back
// through at most `rounds` windows of 32 predecessors without ever waiting.
// If every one of them up to a published inclusive prefix has published its
// count, this block's inclusive prefix is published as well, which keeps the
// look-backs of later blocks that do have bytes to place short; otherwise the
// count stays, which is all k_block_offsets needs.
static __device__ __noinline__ void warp_publish_try(unsigned long long *status, uint32_t b, int rounds)
{
    const int lane = threadIdx.x & 31;
    if (b == 0) {
        if (lane == 0) st_status(&status[0], status_word(kFlagInc, 0, 0));
        return;
    }
    if (lane == 0) st_status(&status[b], status_word(kFlagAgg, 0, 0));
    unsigned long long excl = 0;
    int64_t nearest = (int64_t)b - 1;
    for (int r = 0; r < rounds; ++r) {
        const int64_t idx = nearest - lane;
        const unsigned long long v = idx >= 0 ? ld_status(&status[idx]) : kFlagInc;
        const uint32_t flag = (uint32_t)(v >> 62);
        const uint32_t inc = __ballot_sync(kFull, flag == 2u);
        const uint32_t not_ready = __ballot_sync(kFull, flag == 0u);
        const uint32_t upto = inc ? ((inc & (0u - inc)) << 1) - 1u : kFull;
        if (not_ready & upto) return;
        unsigned long long mine = ((upto >> lane) & 1u) ? (v & kValMask) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(kFull, mine, o);
        excl += mine;
        if (inc) {
            if (lane == 0) st_status(&status[b], status_word(kFlagInc, 0, excl));
            return;
        }
        nearest -= 32;
    }
}

// With deferred placement, every 32nd block waits in the look-back and
// publishes its inclusive prefix even when it has nothing to place, so that
// the look-back of a block that does (walking back over blocks that only
// published their counts) reaches an inclusive prefix within two windows.
__device__ __forceinline__ bool lookback_leader(uint32_t b) { return (b & 31u) == 31u; }

// The same protocol as warp_lookback run by a single thread (used by the
// wait-timeout test hook).
static __device__ __noinline__ unsigned long long lookback(unsigned long long *status, uint32_t b,
                                                           unsigned long long total, uint64_t wait_ns,
                                                           bool *timed_out)
{
    *timed_out = false;
    if (b == 0) {
        st_status(&status[0], status_word(kFlagInc, total, total));
        return 0;
    }
    st_status(&status[b], status_word(kFlagAgg, total, total));
    unsigned long long excl = 0;
    const uint64_t t0 = global_ns();
    uint32_t spins = 0;
    int64_t pred = (int64_t)b - 1;
    while (pred >= 0) {
        const unsigned long long v = ld_status(&status[pred]);
        const unsigned long long flag = v >> 62;
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
        if (flag == 2) break;
        --pred;
    }
    st_status(&status[b], status_word(kFlagInc, total, excl + total));
    return excl;
}

// Launch a kernel as a programmatic dependent of the previous work in `s`.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Args &&>(args)...);
}

// The same, as thread-block clusters of cluster_x CTAs along x (gridDim.x a
// multiple of cluster_x).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, k, static_cast<Args &&>(args)...);
}

}  // namespace dev
}  // namespace lct
