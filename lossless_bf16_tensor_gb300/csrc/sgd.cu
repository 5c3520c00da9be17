// Fused compressed SGD step of liblct: W <- W - eta*M.
//
// [EXP] "Training adds a second problem": instead of decoding W and M to HBM,
// updating, and re-encoding (three round trips), one kernel reads the
// compressed inputs, does the arithmetic, and writes the new sign-fraction
// bytes and the re-coded exponents in a single pass over each block.
//
// Thread j of a block's CTA owns stream j of W, of M and of the new W: per
// row it decodes one symbol of W and one of M, updates the value, writes its
// sign-fraction byte and appends its exponent to the new slot, whose words go
// straight to global memory.  The slot images of W and M come in by TMA bulk
// copy; the sign-fraction bytes stream through a ring of row chunks.  A chunk
// in which no stream of a warp reaches a spill marker and every new slot has
// room takes a fast path with no per-value checks.  Spilled new exponents are
// kept for 32 rows out of place, which leaves room for three CTAs per SM; an
// out-of-place step whose stream spills more than that re-decodes the older
// rows of that stream at the end.  In place every spilled exponent is kept:
// a code is at most 16 bits, so a stream holds at least 2W symbols of its
// slot and spills at most NJ - 2W.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kSgdThreads = 256;
constexpr int kSgdRows = 8;    // rows per sign-fraction chunk
constexpr int kSgdSpill = 32;  // spilled new-exponent rows kept (out of place; a power of two)

// One value of W and one of M (BF16 in bits 0..15) -> the updated BF16:
// fl32(w - fl32(eta*m)), product and difference rounded separately.
__device__ __forceinline__ uint32_t sgd_one(uint32_t w, uint32_t m, float eta)
{
    return bf16_rne(__fsub_rn(__uint_as_float(w << 16), __fmul_rn(eta, __uint_as_float(m << 16))));
}

template <int LEVEL, bool INPLACE>
struct SgdSmem {
    static constexpr int W = Geo<LEVEL>::W, NJ = Geo<LEVEL>::NJ;
    static constexpr int kSpillRows = INPLACE ? NJ - 2 * W : kSgdSpill;
    static constexpr int kStages = INPLACE ? 3 : 2;  // chunks in flight
    static constexpr int kSlotIn = (W + 1) * kStreams * 4;  // + zero guard row
    static constexpr int kRing = kStages * kSgdRows * kStreams;  // per input
    static constexpr int kLuts = 2 * 256 * 4 + 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;
    static constexpr int kBytes = 2 * kSlotIn + 2 * kRing + kLuts + kSpill;
    static constexpr int kCtas = INPLACE ? 1 : 3;  // CTAs per SM the launch bounds ask for
    static_assert(INPLACE || (kSgdSpill & (kSgdSpill - 1)) == 0, "ring index uses a mask");
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
    uint32_t pos;         // bit position in the slot
    const uint32_t *col;  // slot image column in shared memory
    uint32_t marker;
    uint64_t ovf_at;      // overflow index of spilled symbol k is ovf_at + k
};

// Symbol k of an input stream as a decode-table entry (exponent in bits 7..14).
template <int W>
__device__ __forceinline__ uint32_t in_take(InStream &s, uint32_t k, const uint32_t *lut, const uint8_t *ovf,
                                            bool ovf_ok)
{
    if (k < s.marker) return rd_take<W>(s.pos, s.col, lut);
    return ovf_ok ? (uint32_t)__ldg(ovf + s.ovf_at + k) << 7 : 0u;
}

// Slot of a spilled new exponent in the staging rows: t = k - marker counts
// the stream's spilled symbols; out of place the rows are a ring.
template <bool INPLACE, int SP>
__device__ __forceinline__ uint32_t stage_row(uint32_t t)
{
    return INPLACE ? t : (t & (SP - 1));
}

template <int LEVEL, bool INPLACE>
__global__ void __launch_bounds__(kSgdThreads, SgdSmem<LEVEL, INPLACE>::kCtas) k_sgd(const __grid_constant__ SgdArgs a)
{
    using G = Geo<LEVEL>;
    using L = SgdSmem<LEVEL, INPLACE>;
    constexpr int W = G::W, R = kSgdRows, S = L::kStages, SP = L::kSpillRows;
    constexpr int NW = kSgdThreads / 32;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *slotW = reinterpret_cast<uint32_t *>(smem);
    uint32_t *slotM = reinterpret_cast<uint32_t *>(smem + L::kSlotIn);
    uint8_t *sfW_s = smem + 2 * L::kSlotIn;
    uint8_t *sfM_s = sfW_s + L::kRing;
    uint32_t *lutW = reinterpret_cast<uint32_t *>(sfM_s + L::kRing);
    uint32_t *lutM = lutW + 256;
    uint2 *tbl = reinterpret_cast<uint2 *>(lutM + 256);
    uint8_t *ring = reinterpret_cast<uint8_t *>(tbl + 256);
    __shared__ __align__(8) uint64_t bar_slot, bar_sf[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_flags;  // bit 0: a wait gave up, bit 1: corrupt input

    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.w_in.n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    if (j == 0) {
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
    lutW[j] = dec_entry(a.cbw, delta_w, j);
    lutM[j] = dec_entry(a.cbm, hm->delta, j);
    tbl[j] = enc_entry(a.cbw, delta_w, j);
    slotW[W * kStreams + j] = 0u;
    slotM[W * kStreams + j] = 0u;
    __syncthreads();  // barriers initialised
    if (j == 0) {
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
    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    InStream sw, sm;
    sw.col = slotW + j;
    sm.col = slotM + j;
    {
        const uint32_t mw = a.w_in.markers[(uint64_t)b * kStreams + j], mm = a.m.markers[(uint64_t)b * kStreams + j];
        bad |= mw > nj || mm > nj;
        sw.marker = min(mw, nj);
        sm.marker = min(mm, nj);
    }
    bool ovf_ok_w, ovf_ok_m;
    {
        uint32_t tot_w, tot_m;
        const uint32_t pre_w = group_exclusive_scan(nj - sw.marker, warp_tot, NW, 0, &tot_w);
        const uint32_t pre_m = group_exclusive_scan(nj - sm.marker, warp_tot, NW, 0, &tot_m);
        const uint64_t a0 = a.w_in.blk_off[b], a1 = a.w_in.blk_off[b + 1];
        const uint64_t c0 = a.m.blk_off[b], c1 = a.m.blk_off[b + 1];
        ovf_ok_w = a1 <= a.w_in.ovf_cap && a0 <= a1 && a1 - a0 == tot_w;
        ovf_ok_m = c1 <= a.m.ovf_cap && c0 <= c1 && c1 - c0 == tot_m;
        sw.ovf_at = a0 + pre_w - sw.marker;
        sm.ovf_at = c0 + pre_m - sm.marker;
        bad |= !ovf_ok_w || !ovf_ok_m;
    }
    const uint8_t *ovf_w = a.w_in.ovf, *ovf_m = a.m.ovf;

    if (!mbar_wait(&bar_slot, 0, limit)) s_flags = 1;
    sw.pos = 0;
    sm.pos = 0;
    Writer wo;
    wr_init<W>(wo, nj);
    uint32_t *colO = a.w_out.slots + (uint64_t)b * W * kStreams + j;
    uint8_t *sfj = a.w_out.sf + base + j;
    uint8_t *ringj = ring + j;
    const float eta = a.eta;

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot = c % S;
        if (bulk && !mbar_wait(&bar_sf[slot], (c / S) & 1u, (s_flags & 1u) ? 1000000ull : limit)) s_flags = 1;
        const uint8_t *sfwc = sfW_s + slot * R * kStreams + j;
        const uint8_t *sfmc = sfM_s + slot * R * kStreams + j;
        uint8_t *sfo = sfj + (uint64_t)c * R * kStreams;
        const uint32_t kend = (c + 1) * R;
        if (bulk && __all_sync(kFull, sw.marker >= kend && sm.marker >= kend)) {
            // loads first (both decode chains, the sign-fraction bytes, the
            // new values' code-table entries), stores last, so nothing orders
            // a load behind a store
            uint32_t ew[R], em[R], h[R], need = 0;
            uint2 ent[R];
#pragma unroll
            for (int r = 0; r < R; r += 2) {
                rd_take2<W>(sw.pos, sw.col, lutW, ew[r], ew[r + 1]);
                rd_take2<W>(sm.pos, sm.col, lutM, em[r], em[r + 1]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r)
                h[r] = sgd_one(join_one(sfwc[r * kStreams], ew[r]), join_one(sfmc[r * kStreams], em[r]), eta);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ent[r] = tbl[exp_of(h[r])];
                need += ent[r].y;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) sfo[r * kStreams] = sf_of(h[r]);
            if (__all_sync(kFull, wo.alive && need <= wo.rem)) {
                // every new stream of the warp keeps the whole chunk in its slot
#pragma unroll
                for (int r = 0; r < R; r += 2) {  // two codes fit the accumulator, then one flush
                    wr_add2(wo, ent[r], ent[r + 1]);
                    wr_flush(wo, colO);
                }
                wo.rem -= need;
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t k = c * R + r;
                    if (wr_put_checked(wo, ent[r], k, colO))
                        ringj[stage_row<INPLACE, SP>(k - wo.marker) * kRow] = (uint8_t)exp_of(h[r]);
                }
            }
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t k = c * R + r;
                if (k >= nj) break;
                const uint32_t ew = in_take<W>(sw, k, lutW, ovf_w, ovf_ok_w);
                const uint32_t em = in_take<W>(sm, k, lutM, ovf_m, ovf_ok_m);
                const uint64_t at = base + (uint64_t)k * kStreams + j;
                const uint32_t fw = bulk ? sfwc[r * kStreams] : a.w_in.sf[at];
                const uint32_t fm = bulk ? sfmc[r * kStreams] : a.m.sf[at];
                const uint32_t h = sgd_one(join_one(fw, ew), join_one(fm, em), eta);
                const uint32_t e = exp_of(h);
                sfo[r * kStreams] = sf_of(h);
                if (wr_put_checked(wo, tbl[e], k, colO)) ringj[stage_row<INPLACE, SP>(k - wo.marker) * kRow] = (uint8_t)e;
            }
        }
        __syncthreads();  // every thread is done with this chunk's ring slot
        if (j == 0 && c + S < nbulk) {
            mbar_expect_tx(&bar_sf[slot], 2 * R * kStreams);
            bulk_load(sfW_s + slot * R * kStreams, a.w_in.sf + base + (uint64_t)(c + S) * R * kStreams, R * kStreams,
                      &bar_sf[slot]);
            bulk_load(sfM_s + slot * R * kStreams, a.m.sf + base + (uint64_t)(c + S) * R * kStreams, R * kStreams,
                      &bar_sf[slot]);
        }
    }
    bad |= sw.pos > 32u * W || sm.pos > 32u * W;
    if (bad) atomicOr(&s_flags, 2u);
    wr_finish<W>(wo, colO);
    const uint32_t marker = wo.marker, spill = nj - marker;
    uint32_t total;
    const uint32_t pre = group_exclusive_scan(spill, warp_tot, NW, 0, &total);
    a.w_out.markers[(uint64_t)b * kStreams + j] = (uint16_t)marker;

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
        for (int i = 0; i < 32; ++i) {
            const uint32_t smk = __shfl_sync(kFull, marker, i);
            const uint32_t ssp = __shfl_sync(kFull, spill, i);
            const uint32_t spr = __shfl_sync(kFull, pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            const uint32_t kept_from = INPLACE || ssp <= (uint32_t)SP ? 0u : ssp - SP;  // older ones were overwritten
            for (uint32_t l = lane; l < ssp; l += 32)
                if (l >= kept_from) out[spr + l] = ring[stage_row<INPLACE, SP>(l) * kRow + sj];
        }
        const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;
        if (!INPLACE && marker < kept_from) {
            // This stream spilled past the kept rows: decode its W and M again
            // from the slot images (still in shared memory) and recompute the
            // older spilled exponents.  W's sign-fraction bytes are intact
            // because the step is out of place.
            InStream rw = sw, rm = sm;
            rw.pos = 0;
            rm.pos = 0;
            for (uint32_t k = 0; k < kept_from; ++k) {
                const uint32_t ew = in_take<W>(rw, k, lutW, ovf_w, ovf_ok_w);
                const uint32_t em = in_take<W>(rm, k, lutM, ovf_m, ovf_ok_m);
                const uint64_t at = base + (uint64_t)k * kStreams + j;
                const uint32_t h = sgd_one(join_one(a.w_in.sf[at], ew), join_one(a.m.sf[at], em), eta);
                if (k >= marker) out[pre + (k - marker)] = exp_of(h);
            }
        }
    }
    pdl_launch_dependents();
    if (j == 0 && (s_flags & 1u)) {
        // a wait gave up: let every copy still in flight land before the CTA
        // (and its shared memory) goes away
        mbar_wait(&bar_slot, 0, limit);
        for (uint32_t s = 0; s < (uint32_t)S && s < nbulk; ++s) {
            const uint32_t last = s + (nbulk - 1 - s) / S * S;
            mbar_wait(&bar_sf[s], (last / S) & 1u, limit);
        }
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
