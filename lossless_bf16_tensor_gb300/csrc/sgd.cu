// Fused compressed SGD step of liblct: W <- W - eta*M.
//
// [EXP] "Training adds a second problem": instead of decoding W and M to HBM,
// updating, and re-encoding (three round trips), one kernel reads the
// compressed inputs, does the arithmetic, and writes the new sign-fraction
// bytes and the re-coded exponents in a single pass over each block.
//
// Thread t of a block's CTA owns the neighbouring streams 2t and 2t+1 of W, of
// M and of the new W: per row it decodes two symbols of W and two of M,
// updates the two values, writes their sign-fraction bytes and appends their
// exponents to the new slots.  The slot images of W and M come in by TMA bulk
// copy; the sign-fraction bytes stream through a ring of row chunks.  A chunk
// in which no stream of a warp reaches a spill marker and every new slot has
// room takes a fast path with no per-value checks.  Spilled new exponents are
// kept for 64 rows (every row when W is updated in place); an out-of-place
// step whose stream spills more than that re-decodes the older rows of that
// stream at the end.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kSgdThreads = 128;
constexpr int kSgdRows = 8;    // rows per sign-fraction chunk
constexpr int kSgdRing = 3;    // chunks in flight
constexpr int kSgdSpill = 64;  // spilled new-exponent rows kept (out of place)

// Two float32 -> two BF16 (low half: r0), round to nearest even, subnormals
// kept.  The conversion writes NaN as 0x7FFF; this library's NaN is 0x7FC0.
__device__ __forceinline__ uint32_t bf16x2_rne(float r0, float r1)
{
    uint32_t h;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(r1), "f"(r0));
    if ((h & 0xFFFFu) == 0x7FFFu) h ^= 0x003Fu;
    if ((h >> 16) == 0x7FFFu) h ^= 0x003F0000u;
    return h;
}

// Two values of W and two of M (BF16 pairs) -> the two updated BF16:
// fl32(w - fl32(eta*m)), product and difference rounded separately.
__device__ __forceinline__ uint32_t sgd_pair(uint32_t w2, uint32_t m2, float eta)
{
    const float r0 = __fsub_rn(__uint_as_float(w2 << 16), __fmul_rn(eta, __uint_as_float(m2 << 16)));
    const float r1 = __fsub_rn(__uint_as_float(w2 & 0xFFFF0000u), __fmul_rn(eta, __uint_as_float(m2 & 0xFFFF0000u)));
    return bf16x2_rne(r0, r1);
}

template <int LEVEL, bool INPLACE>
struct SgdSmem {
    static constexpr int W = Geo<LEVEL>::W, NJ = Geo<LEVEL>::NJ;
    static constexpr int kSpillRows = INPLACE ? NJ : kSgdSpill;
    static constexpr int kSlotIn = (W + 1) * kStreams * 4;  // + zero guard row
    static constexpr int kSlotOut = W * kStreams * 4;
    static constexpr int kRing = kSgdRing * kSgdRows * kStreams;  // per input
    static constexpr int kLuts = 2 * 256 * 4 + 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;
    static constexpr int kBytes = 2 * kSlotIn + kSlotOut + 2 * kRing + kLuts + kSpill;
};

// Prologue: the new W's header (shift and codebook carried over, status
// cleared but inheriting an error already latched in W or M, or CORRUPT if
// either header is not valid) and cleared look-back words.
__global__ void __launch_bounds__(256) k_sgd_prologue(DevTensor w_in, DevTensor m, DevTensor w_out,
                                                       uint32_t hash_w, uint32_t hash_m)
{
    pdl_wait();
    pdl_launch_dependents();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < w_out.nblocks;
         i += (uint64_t)gridDim.x * blockDim.x)
        w_out.work[i] = 0ull;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const lct_header *hw = w_in.hdr;
        const lct_header *hm = m.hdr;
        uint32_t st = hw->status ? hw->status : hm->status;
        const bool ok_w = hw->magic == LCT_MAGIC && hw->n == w_in.n && hw->level == w_in.level && hw->cb_hash == hash_w;
        const bool ok_m = hm->magic == LCT_MAGIC && hm->n == m.n && hm->level == m.level && hm->cb_hash == hash_m;
        if (!st && !(ok_w && ok_m)) st = LCT_ERR_CORRUPT;
        const int delta = hw->delta;
        lct_header *h = w_out.hdr;
        h->magic = LCT_MAGIC;
        h->version = 1;
        h->n = w_out.n;
        h->level = w_out.level;
        h->delta = delta;
        h->status = st;
        h->cb_hash = hash_w;
        h->ovf_used = 0;
        h->ovf_cap = w_out.ovf_cap;
    }
}

// One stream of one compressed input (W or M) inside the kernel.
struct InStream {
    Reader rd;
    const uint32_t *col;  // slot image column in shared memory
    uint32_t marker;
    uint64_t ovf_at;      // overflow index of spilled symbol k is ovf_at + k
};

// Symbol k of an input stream as a decode-table entry (exponent in bits 7..14).
template <int W>
__device__ __forceinline__ uint32_t in_take(InStream &s, uint32_t k, const uint32_t *lut, const uint8_t *ovf,
                                            bool ovf_ok)
{
    if (k < s.marker) return rd_take<W>(s.rd, s.col, lut);
    return ovf_ok ? (uint32_t)__ldg(ovf + s.ovf_at + k) << 7 : 0u;
}

template <int LEVEL, bool INPLACE>
__global__ void __launch_bounds__(kSgdThreads, 2) k_sgd(const __grid_constant__ SgdArgs a)
{
    using G = Geo<LEVEL>;
    using L = SgdSmem<LEVEL, INPLACE>;
    constexpr int W = G::W, R = kSgdRows, S = kSgdRing, SP = L::kSpillRows;
    constexpr int NW = kSgdThreads / 32, HALF = kStreams / 2;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *slotW = reinterpret_cast<uint32_t *>(smem);
    uint32_t *slotM = reinterpret_cast<uint32_t *>(smem + L::kSlotIn);
    uint32_t *slotO = reinterpret_cast<uint32_t *>(smem + 2 * L::kSlotIn);
    uint8_t *sfW_s = smem + 2 * L::kSlotIn + L::kSlotOut;
    uint8_t *sfM_s = sfW_s + L::kRing;
    uint32_t *lutW = reinterpret_cast<uint32_t *>(sfM_s + L::kRing);
    uint32_t *lutM = lutW + 256;
    uint2 *tbl = reinterpret_cast<uint2 *>(lutM + 256);
    uint8_t *ring = reinterpret_cast<uint8_t *>(tbl + 256);
    __shared__ __align__(8) uint64_t bar_slot, bar_sf[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_flags;  // bit 0: a wait gave up, bit 1: corrupt input

    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t j0 = 2 * t, j1 = 2 * t + 1;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.w_in.n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    if (t == 0) {
        mbar_init(&bar_slot, 1);
        for (int s = 0; s < S; ++s) mbar_init(&bar_sf[s], 1);
        fence_mbar_init();
        s_flags = 0;
    }
    // inputs, the new header and the cleared look-back words are all ready
    pdl_wait();
    const lct_header *hw = a.w_in.hdr, *hm = a.m.hdr;
    bool bad = !(hw->magic == LCT_MAGIC && hw->n == a.w_in.n && hw->level == LEVEL && hw->cb_hash == a.cbw.hash) ||
               !(hm->magic == LCT_MAGIC && hm->n == a.m.n && hm->level == LEVEL && hm->cb_hash == a.cbm.hash);
    const int delta_w = a.w_out.hdr->delta;  // the prologue copied W's shift
    const int delta_m = hm->delta;
    for (int v = t; v < 256; v += kSgdThreads) {
        lutW[v] = dec_entry(a.cbw, delta_w, v);
        lutM[v] = dec_entry(a.cbm, delta_m, v);
        tbl[v] = enc_entry(a.cbw, delta_w, v);
    }
    reinterpret_cast<uint2 *>(slotW + W * kStreams)[t] = make_uint2(0u, 0u);
    reinterpret_cast<uint2 *>(slotM + W * kStreams)[t] = make_uint2(0u, 0u);
    __syncthreads();  // barriers initialised
    if (t == 0) {
        mbar_expect_tx(&bar_slot, 2 * W * kStreams * 4);
        bulk_load(slotW, a.w_in.slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
        bulk_load(slotM, a.m.slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
        for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) {
            mbar_expect_tx(&bar_sf[c], 2 * R * kStreams);
            bulk_load(sfW_s + c * R * kStreams, a.w_in.sf + base + (uint64_t)c * R * kStreams, R * kStreams, &bar_sf[c]);
            bulk_load(sfM_s + c * R * kStreams, a.m.sf + base + (uint64_t)c * R * kStreams, R * kStreams, &bar_sf[c]);
        }
    }

    // input markers, spill prefixes and overflow ranges
    const uint32_t nj0 = nb > j0 ? (nb - j0 + 255) / 256 : 0, nj1 = nb > j1 ? (nb - j1 + 255) / 256 : 0;
    InStream w0, w1, m0, m1;
    w0.col = slotW + j0;
    w1.col = slotW + j1;
    m0.col = slotM + j0;
    m1.col = slotM + j1;
    {
        const uint32_t mw = reinterpret_cast<const uint32_t *>(a.w_in.markers + (uint64_t)b * kStreams)[t];
        const uint32_t mm = reinterpret_cast<const uint32_t *>(a.m.markers + (uint64_t)b * kStreams)[t];
        bad |= (mw & 0xFFFFu) > nj0 || (mw >> 16) > nj1 || (mm & 0xFFFFu) > nj0 || (mm >> 16) > nj1;
        w0.marker = min(mw & 0xFFFFu, nj0);
        w1.marker = min(mw >> 16, nj1);
        m0.marker = min(mm & 0xFFFFu, nj0);
        m1.marker = min(mm >> 16, nj1);
    }
    bool ovf_ok_w, ovf_ok_m;
    {
        uint32_t tot_w, tot_m;
        const uint32_t spw0 = nj0 - w0.marker, spm0 = nj0 - m0.marker;
        const uint32_t pre_w = group_exclusive_scan(spw0 + nj1 - w1.marker, warp_tot, NW, 0, &tot_w);
        const uint32_t pre_m = group_exclusive_scan(spm0 + nj1 - m1.marker, warp_tot, NW, 0, &tot_m);
        const uint64_t a0 = a.w_in.blk_off[b], a1 = a.w_in.blk_off[b + 1];
        const uint64_t c0 = a.m.blk_off[b], c1 = a.m.blk_off[b + 1];
        ovf_ok_w = a1 <= a.w_in.ovf_cap && a0 <= a1 && a1 - a0 == tot_w;
        ovf_ok_m = c1 <= a.m.ovf_cap && c0 <= c1 && c1 - c0 == tot_m;
        w0.ovf_at = a0 + pre_w - w0.marker;
        w1.ovf_at = a0 + pre_w + spw0 - w1.marker;
        m0.ovf_at = c0 + pre_m - m0.marker;
        m1.ovf_at = c0 + pre_m + spm0 - m1.marker;
        bad |= !ovf_ok_w || !ovf_ok_m;
    }
    const uint8_t *ovf_w = a.w_in.ovf, *ovf_m = a.m.ovf;

    if (!mbar_wait(&bar_slot, 0, limit)) s_flags = 1;
    rd_init<W>(w0.rd, w0.col);
    rd_init<W>(w1.rd, w1.col);
    rd_init<W>(m0.rd, m0.col);
    rd_init<W>(m1.rd, m1.col);
    Writer o0, o1;
    wr_init<W>(o0, nj0);
    wr_init<W>(o1, nj1);
    uint32_t *colO0 = slotO + j0, *colO1 = slotO + j1;
    uint16_t *sft = reinterpret_cast<uint16_t *>(a.w_out.sf + base) + t;
    const float eta = a.eta;

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot = c % S;
        if (bulk && !mbar_wait(&bar_sf[slot], (c / S) & 1u, (s_flags & 1u) ? 1000000ull : limit)) s_flags = 1;
        const uint16_t *sfwc = reinterpret_cast<const uint16_t *>(sfW_s + slot * R * kStreams) + t;
        const uint16_t *sfmc = reinterpret_cast<const uint16_t *>(sfM_s + slot * R * kStreams) + t;
        uint16_t *sfo = sft + (uint64_t)c * R * HALF;
        const uint32_t kend = (c + 1) * R;
        const bool fast = bulk && __all_sync(kFull, w0.marker >= kend && w1.marker >= kend && m0.marker >= kend &&
                                                        m1.marker >= kend && o0.alive && o1.alive &&
                                                        o0.rem >= 16u * R && o1.rem >= 16u * R);
        if (fast) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const uint32_t ew0 = rd_take<W>(w0.rd, w0.col, lutW), ew1 = rd_take<W>(w1.rd, w1.col, lutW);
                const uint32_t em0 = rd_take<W>(m0.rd, m0.col, lutM), em1 = rd_take<W>(m1.rd, m1.col, lutM);
                const uint32_t h2 = sgd_pair(join_pair(sfwc[r * HALF], ew0, ew1), join_pair(sfmc[r * HALF], em0, em1),
                                             eta);
                sfo[r * HALF] = (uint16_t)sf_pair(h2);
                wr_put(o0, tbl[(h2 >> 7) & 0xFFu], colO0);
                wr_put(o1, tbl[(h2 >> 23) & 0xFFu], colO1);
            }
            wr_fix_rem<W>(o0);
            wr_fix_rem<W>(o1);
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t k = c * R + r;
                if (k >= nj0) break;  // nj1 <= nj0
                const bool v1 = k < nj1;
                const uint32_t ew0 = in_take<W>(w0, k, lutW, ovf_w, ovf_ok_w);
                const uint32_t em0 = in_take<W>(m0, k, lutM, ovf_m, ovf_ok_m);
                const uint32_t ew1 = v1 ? in_take<W>(w1, k, lutW, ovf_w, ovf_ok_w) : 0u;
                const uint32_t em1 = v1 ? in_take<W>(m1, k, lutM, ovf_m, ovf_ok_m) : 0u;
                const uint64_t at = base + (uint64_t)k * kStreams + j0;
                uint32_t fw, fm;
                if (bulk) {
                    fw = sfwc[r * HALF];
                    fm = sfmc[r * HALF];
                } else if (v1) {
                    fw = *reinterpret_cast<const uint16_t *>(a.w_in.sf + at);
                    fm = *reinterpret_cast<const uint16_t *>(a.m.sf + at);
                } else {
                    fw = a.w_in.sf[at];
                    fm = a.m.sf[at];
                }
                const uint32_t h2 = sgd_pair(join_pair(fw, ew0, ew1), join_pair(fm, em0, em1), eta);
                const uint32_t sf2 = sf_pair(h2);
                if (v1)
                    sfo[r * HALF] = (uint16_t)sf2;
                else
                    a.w_out.sf[at] = (uint8_t)sf2;
                const uint32_t e0 = (h2 >> 7) & 0xFFu, e1 = (h2 >> 23) & 0xFFu;
                if (wr_put_checked(o0, tbl[e0], k, colO0)) ring[(k % SP) * kRow + j0] = (uint8_t)e0;
                if (v1 && wr_put_checked(o1, tbl[e1], k, colO1)) ring[(k % SP) * kRow + j1] = (uint8_t)e1;
            }
        }
        __syncthreads();  // every thread is done with this chunk's ring slot
        if (t == 0 && c + S < nbulk) {
            mbar_expect_tx(&bar_sf[slot], 2 * R * kStreams);
            bulk_load(sfW_s + slot * R * kStreams, a.w_in.sf + base + (uint64_t)(c + S) * R * kStreams, R * kStreams,
                      &bar_sf[slot]);
            bulk_load(sfM_s + slot * R * kStreams, a.m.sf + base + (uint64_t)(c + S) * R * kStreams, R * kStreams,
                      &bar_sf[slot]);
        }
    }
    bad |= rd_consumed(w0.rd) > 32u * W || rd_consumed(w1.rd) > 32u * W || rd_consumed(m0.rd) > 32u * W ||
           rd_consumed(m1.rd) > 32u * W;
    if (bad) atomicOr(&s_flags, 2u);
    wr_finish<W>(o0, colO0);
    wr_finish<W>(o1, colO1);
    const uint32_t mk0 = o0.marker, mk1 = o1.marker, sp0 = nj0 - mk0, sp1 = nj1 - mk1;
    uint32_t total;
    const uint32_t pre0 = group_exclusive_scan(sp0 + sp1, warp_tot, NW, 0, &total);  // syncs: slot image complete
    const uint32_t pre1 = pre0 + sp0;

    if (t == 0) {
        fence_proxy_async();
        bulk_store(a.w_out.slots + (uint64_t)b * W * kStreams, slotO, W * kStreams * 4);
        bulk_commit();
    }
    reinterpret_cast<uint32_t *>(a.w_out.markers + (uint64_t)b * kStreams)[t] = mk0 | (mk1 << 16);

    if (warp == 0) {
        bool timed_out;
        const unsigned long long excl = warp_lookback(a.w_out.work, b, total, limit, &timed_out);
        if (lane == 0) {
            if (s_flags & 2u) latch(a.w_out.hdr, LCT_ERR_CORRUPT);
            if (timed_out || (s_flags & 1u)) latch(a.w_out.hdr, LCT_ERR_TIMEOUT);
            a.w_out.blk_off[b] = excl;
            if (b == a.w_out.nblocks - 1) {
                a.w_out.blk_off[b + 1] = excl + total;
                a.w_out.hdr->ovf_used = excl + total;
            }
            if (excl + total > a.w_out.ovf_cap) latch(a.w_out.hdr, LCT_ERR_OVERFLOW_CAPACITY);
            s_excl = excl;
        }
    }
    __syncthreads();

    const unsigned long long excl = s_excl;
    if (total > 0 && excl + total <= a.w_out.ovf_cap) {
        uint8_t *out = a.w_out.ovf + excl;
        // spilled rows still kept in shared memory: one warp per stream at a time
        for (int i = 0; i < 64; ++i) {
            const int src = i >> 1;
            const uint32_t smk = __shfl_sync(kFull, (i & 1) ? mk1 : mk0, src);
            const uint32_t ssp = __shfl_sync(kFull, (i & 1) ? sp1 : sp0, src);
            const uint32_t spr = __shfl_sync(kFull, (i & 1) ? pre1 : pre0, src);
            const uint32_t sj = (uint32_t)(warp * 64 + i);
            const uint32_t nj = smk + ssp;
            const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;
            for (uint32_t l = lane; l < ssp; l += 32) {
                const uint32_t k = smk + l;
                if (k >= kept_from) out[spr + l] = ring[(k % SP) * kRow + sj];
            }
        }
        if (!INPLACE) {
            // A stream that spilled past the kept rows: decode its W and M again
            // from the slot images (still in shared memory) and recompute the
            // older spilled exponents.  W's sign-fraction bytes are intact
            // because the step is out of place.
            for (int q = 0; q < 2; ++q) {
                const uint32_t nj = q ? nj1 : nj0, marker = q ? mk1 : mk0, pre = q ? pre1 : pre0;
                const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;
                if (marker >= kept_from) continue;
                const uint32_t j = q ? j1 : j0;
                InStream rw = q ? w1 : w0, rm = q ? m1 : m0;
                rd_init<W>(rw.rd, rw.col);
                rd_init<W>(rm.rd, rm.col);
                for (uint32_t k = 0; k < kept_from; ++k) {
                    const uint32_t ew = in_take<W>(rw, k, lutW, ovf_w, ovf_ok_w);
                    const uint32_t em = in_take<W>(rm, k, lutM, ovf_m, ovf_ok_m);
                    const uint64_t at = base + (uint64_t)k * kStreams + j;
                    const uint32_t h = sgd_pair(join_one(a.w_in.sf[at], ew), join_one(a.m.sf[at], em), eta);
                    if (k >= marker) out[pre + (k - marker)] = exp_of(h);
                }
            }
        }
    }
    pdl_launch_dependents();
    if (t == 0) {
        if (s_flags & 1u) {
            for (uint32_t s = 0; s < (uint32_t)S && s < nbulk; ++s) {
                const uint32_t last = s + (nbulk - 1 - s) / S * S;
                mbar_wait(&bar_sf[s], (last / S) & 1u, limit);
            }
        }
        bulk_wait_all();  // the slot image store has read shared memory
    }
}

template <int LEVEL, bool INPLACE>
cudaError_t launch_level(const SgdArgs &a, cudaStream_t s)
{
    constexpr int smem = SgdSmem<LEVEL, INPLACE>::kBytes;
    cudaError_t err = cudaFuncSetAttribute(k_sgd<LEVEL, INPLACE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_sgd<LEVEL, INPLACE>, dim3(a.w_out.nblocks), dim3(kSgdThreads), smem, s, a);
}

template <int LEVEL>
cudaError_t launch_sgd_level(const SgdArgs &a, cudaStream_t s)
{
    return a.in_place ? launch_level<LEVEL, true>(a, s) : launch_level<LEVEL, false>(a, s);
}

}  // namespace dev

cudaError_t launch_sgd(const SgdArgs &a, cudaStream_t s)
{
    const uint32_t zero_ctas = 1 + a.w_out.nblocks / 8192;
    cudaError_t err = dev::launch_pdl(dev::k_sgd_prologue, dim3(zero_ctas < 64 ? zero_ctas : 64), dim3(256), 0, s,
                                      a.w_in, a.m, a.w_out, a.cbw.hash, a.cbm.hash);
    if (err != cudaSuccess || a.w_out.nblocks == 0) return err;
    switch (a.w_out.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_sgd_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_sgd_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_sgd_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
