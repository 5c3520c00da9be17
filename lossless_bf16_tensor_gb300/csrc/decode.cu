// Decode path of liblct: one CTA per block rebuilds the block's BF16 values.
//
// [EXP] "In bits": every value decodes exactly -- the sign-fraction byte is
// copied back and the exponent comes from its code (or the escape literal).
// [EXP] "Compressing is easy": each of the 256 streams decodes independently
// from its fixed-length slot up to its spill marker, then takes its spilled
// exponents from the uncompressed overflow region.
//
// Thread j owns stream j.  The block's slot image arrives by one TMA bulk
// copy; the sign-fraction bytes stream through a ring of row chunks that TMA
// keeps filled ahead of the decoders; each row the 256 threads decode together
// is written as 512 contiguous bytes.  A chunk in which no stream of a warp
// reaches its spill marker takes a fast path with no per-value checks.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kDecThreads = 256;
constexpr int kDecRows = 32;  // rows per sign-fraction chunk
constexpr int kDecRing = 2;   // chunks in flight

template <int LEVEL>
struct DecodeSmem {
    static constexpr int W = Geo<LEVEL>::W;
    static constexpr int kSlot = (W + 1) * kStreams * 4;  // slot image + zero guard row
    static constexpr int kRing = kDecRing * kDecRows * kStreams;
    static constexpr int kLut = 256 * 2;
    // the readers' reads (word indices modulo 32, up to three words ahead)
    // stay inside the CTA's shared memory: at least 35 KB from the slot image on
    static constexpr int kBytes = kSlot + kRing + kLut < 35 * 1024 ? 35 * 1024 : kSlot + kRing + kLut;
    static_assert(kDecRows % 8 == 0, "eight-row groups");
};

// The decoder's table: 16-bit entries (half the shared-memory footprint of
// the 32-bit ones, so a warp-wide lookup meets fewer bank conflicts: 2.8
// instead of 3.2 wavefronts on average on the matched workloads, in a CPU
// count of the oracle's streams), indexed by the next 8 bits of the stream:
//   bits  0..4   bits consumed (code length, or escape length + 8)
//   bits  7..14  the exponent, for a symbol with its own code (0 for escape)
//   bit  15      an escape
__device__ __forceinline__ uint32_t dec_entry16(const DevCodebook &cb, int delta, int v)
{
    const uint32_t d = cb.dec[v], sym = d & 0x1FF, l = d >> 12;
    if (sym == 256) return 0x8000u | (l + 8u);
    const uint32_t e = cb.zero_atom && sym == 0 ? 0u : (sym + (uint32_t)delta) & 0xFFu;
    return (e << 7) | l;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Two symbols at bit p with 16-bit entries (see rd_pair): the second window
// is the first one shifted by the first symbol's length, which the wrap-mode
// funnel shift takes from the entry's low 5 bits; m.z = 2 scales a table
// index to its byte offset.
__device__ __forceinline__ void rd_pair16(Rd &r, uint32_t lut, const Mul m, uint32_t &w0, uint32_t &w1,
                                          uint32_t &ent0, uint32_t &ent1)
{
    const uint32_t a = imad(r.p & 0x3E0u, m.x, r.col);
    const uint32_t hi = lds32(a), lo = lds32(a + kStreams * 4);
    w0 = __funnelshift_l(lo, hi, r.p);  // the next 32 bits
    ent0 = lds16(imad(w0 >> 24, m.z, lut));
    w1 = __funnelshift_l(0u, w0, ent0);  // w0 << L0
    ent1 = lds16(imad(w1 >> 24, m.z, lut));
    r.p += (ent0 & 31u) + (ent1 & 31u);
}

// A 16-bit entry with its escape literal added in bits 7..14 (bits above 14
// are to be ignored): the literal follows the escape prefix of L - 8 bits, so
// a left funnel shift of (0 : window) by L + 7 brings it there.
__device__ __forceinline__ uint32_t lit_fix16(uint32_t w, uint32_t ent)
{
    return (ent & 0x8000u) ? (ent | __funnelshift_l(w, 0u, (ent & 31u) + 7u)) : ent;
}

// One symbol for the checked path (word index clamped to the slot; the zero
// guard row follows it): the entry with its literal added, p advanced.
template <int W>
__device__ __forceinline__ uint32_t rd_take16(uint32_t &p, const uint32_t *__restrict__ col,
                                              const uint16_t *__restrict__ lut)
{
    const uint32_t w = min(p >> 5, (uint32_t)(W - 1));
    const uint32_t hi = col[w * kStreams], lo = col[(w + 1) * kStreams];
    const uint32_t win = __funnelshift_l(lo, hi, p);
    const uint32_t ent = lut[win >> 24];
    p += ent & 31u;
    return lit_fix16(win, ent);
}

// Two symbols with the stream's next three slot words held in registers
// (w0 = word p/32, w1, w2), for grids of at most two blocks per SM where the
// reader's dependent chain sets a block's time: the window needs no shared
// load on the chain.  The word after the three is loaded at the start of the
// pair (its address is known then) and shifted in when the pair crosses a
// word boundary (a pair is at most 32 bits, so it crosses at most one).
// Word indices are taken modulo 32 as in rd_pair; the load of the fourth
// word reaches at most 35 words past the column's start.
__device__ __forceinline__ void rd_pair16_w3(uint32_t &p, uint32_t &w0, uint32_t &w1, uint32_t &w2, uint32_t col,
                                             uint32_t lut, const Mul m, uint32_t &win0, uint32_t &win1,
                                             uint32_t &ent0, uint32_t &ent1)
{
    const uint32_t w3 = lds32(imad(p & 0x3E0u, m.x, col) + 3u * kStreams * 4u);
    win0 = __funnelshift_l(w1, w0, p);
    ent0 = lds16(imad(win0 >> 24, m.z, lut));
    win1 = __funnelshift_l(0u, win0, ent0);
    ent1 = lds16(imad(win1 >> 24, m.z, lut));
    const uint32_t q = p + (ent0 & 31u) + (ent1 & 31u);
    const bool cross = ((p ^ q) & 32u) != 0u;
    w0 = cross ? w1 : w0;
    w1 = cross ? w2 : w1;
    w2 = cross ? w3 : w2;
    p = q;
}

// A stream's spilled exponents are bytes [p, p + count) of the overflow
// region, taken one per row at the end of the stream: each load's address is
// known from the block's start, but its result is needed before the next row.
// Asking for their lines in L1 at the block's start takes the DRAM latency off
// every one of those rows.  The first two 128-byte lines hold all of a
// stream's spilled bytes in MEDIUM and HIGH (at most 96 and 88) and all but
// the longest CLEAN spills.
__device__ __forceinline__ void prefetch_spill(const uint8_t *p, uint32_t count)
{
    if (count == 0) return;
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
    const uint8_t *last = p + count - 1;
    if (((reinterpret_cast<uintptr_t>(p) ^ reinterpret_cast<uintptr_t>(last)) >> 7) != 0)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(p + 128 <= last ? p + 128 : last));
}

template <int LEVEL, bool WIN3>
__global__ void __launch_bounds__(kDecThreads, WIN3 ? 2 : 4) k_decode(const __grid_constant__ DecodeArgs a)
{
    using G = Geo<LEVEL>;
    using L = DecodeSmem<LEVEL>;
    constexpr int W = G::W, R = kDecRows, S = kDecRing;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *slot_s = reinterpret_cast<uint32_t *>(smem);
    uint8_t *sf_s = smem + L::kSlot;
    uint16_t *lut = reinterpret_cast<uint16_t *>(smem + L::kSlot + L::kRing);
    __shared__ __align__(8) uint64_t bar_slot, bar_sf[S];
    __shared__ uint32_t warp_tot[kDecThreads / 32];
    __shared__ uint32_t s_timeout;

    const int j = threadIdx.x;
    const uint32_t b = blockIdx.x + a.first_block;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.t.n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    if (j == 0) {
        mbar_init(&bar_slot, 1);
        for (int s = 0; s < S; ++s) mbar_init(&bar_sf[s], 1);
        fence_mbar_init();
        s_timeout = 0;
    }
    // Everything below reads what earlier work in the stream wrote.  The
    // copies and every global read of the block's start are issued before the
    // first barrier so that their latencies overlap.
    pdl_wait();
    if (j == 0) {
        mbar_expect_tx(&bar_slot, W * kStreams * 4);
        bulk_load(slot_s, a.t.slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
        for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) {
            mbar_expect_tx(&bar_sf[c], R * kStreams);
            bulk_load(sf_s + c * R * kStreams, a.t.sf + base + (uint64_t)c * R * kStreams, R * kStreams, &bar_sf[c]);
        }
    }
    lct_header *hdr = a.t.hdr;
    const bool hdr_ok = hdr->magic == LCT_MAGIC && hdr->n == a.t.n && hdr->level == LEVEL &&
                        hdr->cb_hash == a.cb.hash;
    const int delta = hdr->delta;
    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    uint32_t marker = a.t.markers[(uint64_t)b * kStreams + j];
    const uint64_t off0 = a.t.blk_off[b], off1 = a.t.blk_off[b + 1];
    if (!hdr_ok) {
        if (j == 0) {
            latch(hdr, LCT_ERR_CORRUPT);
            // let the copies issued above land before the CTA goes away
            mbar_wait(&bar_slot, 0, limit);
            for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) mbar_wait(&bar_sf[c], 0, limit);
        }
        return;
    }
    lut[j] = (uint16_t)dec_entry16(a.cb, delta, j);
    slot_s[W * kStreams + j] = 0u;
    __syncthreads();  // table built

    bool bad = marker > nj;
    marker = min(marker, nj);
    uint32_t total;
    const uint32_t pre = group_exclusive_scan(nj - marker, warp_tot, kDecThreads / 32, 0, &total);
    const bool ovf_ok = off1 <= a.t.ovf_cap && off0 <= off1 && off1 - off0 == total;
    const uint64_t ovf_at = off0 + pre - marker;  // overflow index of spilled symbol k is ovf_at + k
    if (ovf_ok) prefetch_spill(a.t.ovf + off0 + pre, nj - marker);

    if (!mbar_wait(&bar_slot, 0, limit)) s_timeout = 1;
    const uint32_t *col = slot_s + j;
    const uint32_t col_s = smem_addr(col), lut_s = smem_addr(lut);
    const Mul mul{a.mul_row, a.mul_ent, a.mul_ent / 2u};  // z = 2: 16-bit table entries
    uint32_t pos = 0;  // bit position in the slot
    uint16_t *yj = a.y + (base - (uint64_t)a.first_block * G::B) + j;

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot = c % S;
        if (bulk && !mbar_wait(&bar_sf[slot], (c / S) & 1u, s_timeout ? 1000000ull : limit)) s_timeout = 1;
        const uint8_t *sfc = sf_s + slot * R * kStreams + j;
        uint16_t *yc = yj + (uint64_t)c * R * kStreams;
        if (bulk && __all_sync(kFull, marker >= (c + 1) * R)) {
            // eight rows at a time: the symbols two by two with the escape
            // literals deferred (added only when a lane of the warp met an
            // escape), then the sign-fraction bytes and the joined values
            uint32_t x0 = 0, x1 = 0, x2 = 0;  // WIN3: slot words pos/32 .. pos/32 + 2
            if (WIN3) {
                const uint32_t a0 = imad(pos & 0x3E0u, mul.x, col_s);
                x0 = lds32(a0);
                x1 = lds32(a0 + kStreams * 4);
                x2 = lds32(a0 + 2 * kStreams * 4);
            }
#pragma unroll
            for (int g = 0; g < R / 8; ++g) {
                uint32_t wv[8], ev[8], esc = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    if (WIN3) {
                        rd_pair16_w3(pos, x0, x1, x2, col_s, lut_s, mul, wv[2 * q], wv[2 * q + 1], ev[2 * q],
                                     ev[2 * q + 1]);
                    } else {
                        Rd r{pos, col_s};
                        rd_pair16(r, lut_s, mul, wv[2 * q], wv[2 * q + 1], ev[2 * q], ev[2 * q + 1]);
                        pos = r.p;
                    }
                    esc |= ev[2 * q] | ev[2 * q + 1];
                }
                if (__any_sync(kFull, esc & 0x8000u)) {
#pragma unroll
                    for (int t = 0; t < 8; ++t) ev[t] = lit_fix16(wv[t], ev[t]);
                }
                uint32_t sf[8];
#pragma unroll
                for (int t = 0; t < 8; ++t) sf[t] = sfc[(g * 8 + t) * kStreams];
#pragma unroll
                for (int t = 0; t < 8; ++t) yc[(g * 8 + t) * kStreams] = (uint16_t)join_one(sf[t], ev[t]);
            }
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t k = c * R + r;
                if (k >= nj) break;
                uint32_t e;
                if (k < marker)
                    e = rd_take16<W>(pos, col, lut);
                else
                    e = ovf_ok ? (uint32_t)__ldg(a.t.ovf + ovf_at + k) << 7 : 0u;
                const uint32_t sf = bulk ? sfc[r * kStreams] : a.t.sf[base + (uint64_t)k * kStreams + j];
                yc[r * kStreams] = (uint16_t)join_one(sf, e);
            }
        }
        __syncthreads();  // every thread is done with this chunk's ring slot
        if (j == 0 && c + S < nbulk) {
            mbar_expect_tx(&bar_sf[slot], R * kStreams);
            bulk_load(sf_s + slot * R * kStreams, a.t.sf + base + (uint64_t)(c + S) * R * kStreams, R * kStreams,
                      &bar_sf[slot]);
        }
    }
    pdl_launch_dependents();
    if (j == 0 && s_timeout) {
        // a wait gave up: let every copy still in flight land before the CTA
        // (and its shared memory) goes away
        mbar_wait(&bar_slot, 0, limit);
        for (uint32_t s = 0; s < (uint32_t)S && s < nbulk; ++s) {
            const uint32_t last = s + (nbulk - 1 - s) / S * S;
            mbar_wait(&bar_sf[s], (last / S) & 1u, limit);
        }
    }
    bad |= pos > 32u * W;
    if (bad) latch(hdr, LCT_ERR_CORRUPT);
    if (j == 0) {
        if (!ovf_ok) latch(hdr, off1 > a.t.ovf_cap && off0 <= off1 ? LCT_ERR_OVERFLOW_CAPACITY : LCT_ERR_CORRUPT);
        if (s_timeout) latch(hdr, LCT_ERR_TIMEOUT);
    }
}

template <int LEVEL, bool WIN3>
cudaError_t launch_kernel(const DecodeArgs &a, uint32_t nblocks, cudaStream_t s)
{
    constexpr int smem = DecodeSmem<LEVEL>::kBytes;
    cudaError_t err = cudaFuncSetAttribute(k_decode<LEVEL, WIN3>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_decode<LEVEL, WIN3>, dim3(nblocks), dim3(kDecThreads), smem, s, a);
}

// Grids of at most two blocks per SM take the register-window reader (two
// CTAs per SM, more registers): there a block's latency sets the time.
template <int LEVEL>
cudaError_t launch_level(const DecodeArgs &a, uint32_t nblocks, cudaStream_t s)
{
    return small_grid(nblocks) ? launch_kernel<LEVEL, true>(a, nblocks, s) : launch_kernel<LEVEL, false>(a, nblocks, s);
}

}  // namespace dev

cudaError_t launch_decode(const DecodeArgs &a, uint32_t nblocks, cudaStream_t s)
{
    if (nblocks == 0) return cudaSuccess;
    switch (a.t.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_level<LCT_LEVEL_CLEAN>(a, nblocks, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_level<LCT_LEVEL_MEDIUM>(a, nblocks, s);
    default: return dev::launch_level<LCT_LEVEL_HIGH>(a, nblocks, s);
    }
}

}  // namespace lct
