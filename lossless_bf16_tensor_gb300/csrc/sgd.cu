// Fused compressed weight updates of liblct: one pass over each block reads
// the compressed inputs, does the arithmetic and writes the new weight's
// sign-fraction bytes and re-coded exponents.
//   OP_SGD:    W <- W - eta*M                       (inputs W, M)
//   OP_ADAMW:  W <- (W - k7*W) - k4*M / (sqrt(V)*k5 + k6)   (inputs W, M, V)
//
// [EXP] "Training adds a second problem": instead of decoding the inputs to
// HBM, updating, and re-encoding (three round trips), one kernel reads the
// compressed inputs and writes the compressed result in a single pass.
// AdamW's moments are updated by the two-state pass (momentum.cu) first; this
// pass then applies them to the weight.
//
// Thread j of a block's CTA owns stream j of every input and of the new W:
// per row it decodes one symbol of each input, updates the value, writes its
// sign-fraction byte and appends its exponent to the new slot, whose words go
// straight to global memory.  The slot images of the inputs come in by TMA
// bulk copy; their sign-fraction bytes stream through a ring of row chunks.
// A chunk in which no stream of a warp reaches a spill marker and every new
// slot has room takes a fast path with no per-value checks.  A code is at
// most 16 bits, so a stream holds at least 2W symbols of its slot and spills
// at most NJ - 2W.  That many spilled new exponents are kept in place and for
// the 128-row levels (MEDIUM, HIGH).  Out of place in CLEAN 32 rows are kept
// (three CTAs per SM for the SGD), and a stream that spills more than that
// re-decodes its older rows at the end.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kSgdThreads = 256;
constexpr int kSgdRows = 8;    // rows per sign-fraction chunk
constexpr int kSgdSpill = 32;  // spilled new-exponent rows kept (out of place; a power of two)

template <int OP>
struct UpdateOp;

// W' = bf16(fl32(w - fl32(k0*m))): product and difference rounded separately.
template <>
struct UpdateOp<OP_SGD> {
    static constexpr int kInputs = 2;
    __device__ static __forceinline__ uint32_t apply(const uint32_t (&x)[2], const float *k)
    {
        return bf16_rne(__fsub_rn(bf16_f(x[0]), __fmul_rn(k[0], bf16_f(x[1]))));
    }
};

// W' = bf16((w - k7*w) - (k4*m) / (sqrt(v)*k5 + k6)), each operation rounded
// on its own (sqrt and the division correctly rounded).
template <>
struct UpdateOp<OP_ADAMW> {
    static constexpr int kInputs = 3;
    __device__ static __forceinline__ uint32_t apply(const uint32_t (&x)[3], const float *k)
    {
        const float w = bf16_f(x[0]);
        const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(bf16_f(x[2])), k[5]), k[6]);
        const float upd = __fdiv_rn(__fmul_rn(k[4], bf16_f(x[1])), den);
        return bf16_rne(__fsub_rn(__fsub_rn(w, __fmul_rn(k[7], w)), upd));
    }
};

template <int LEVEL, bool INPLACE, int NIN>
struct SgdSmem {
    static constexpr int W = Geo<LEVEL>::W, NJ = Geo<LEVEL>::NJ;
    // Every spilled new exponent stays staged (at most NJ - 2W per stream, a
    // code being at most 16 bits) in place, where nothing can be recomputed,
    // and for the 128-row levels, where that is 88 or 96 rows; otherwise a
    // 32-row ring, and a stream that spills more is recomputed at the end.
    static constexpr bool kKeepAll = INPLACE || NJ <= 128;
    static constexpr int kSpillRows = kKeepAll ? NJ - 2 * W : kSgdSpill;
    static constexpr int kStages = INPLACE ? 3 : 2;  // chunks in flight
    static constexpr int kSlotIn = (W + 1) * kStreams * 4;  // + zero guard row
    static constexpr int kRing = kStages * kSgdRows * kStreams;  // per input
    static constexpr int kLuts = NIN * 256 * 4 + 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;
    static constexpr int kBytes = NIN * kSlotIn + NIN * kRing + kLuts + kSpill;
    // CTAs per SM the launch bounds ask for: as many as fit the SM's 228 KB
    // (1 KB of it reserved per CTA), at most 3 for the SGD and 2 for AdamW
    static constexpr int kFit = 228 * 1024 / (kBytes + 1024 + 256);
    static constexpr int kWant = INPLACE ? 1 : (NIN == 2 ? 3 : 2);
    static constexpr int kCtas = kFit < kWant ? kFit : kWant;
    static_assert(kKeepAll || (kSgdSpill & (kSgdSpill - 1)) == 0, "ring index uses a mask");
    static_assert(kBytes <= 227 * 1024 && kCtas >= 1, "shared memory of one CTA");
};

// Prologue: the new W's header (shift and codebook carried over from W,
// status cleared but inheriting an error already latched in an input, or
// CORRUPT if an input header is not valid) and cleared look-back words.
__global__ void __launch_bounds__(256) k_update_prologue(const __grid_constant__ UpdateArgs a)
{
    pdl_wait();
    pdl_launch_dependents();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.w_out.nblocks;
         i += (uint64_t)gridDim.x * blockDim.x)
        a.w_out.work[i] = 0ull;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        uint32_t st = 0;
        bool ok = true;
        for (uint32_t i = 0; i < a.nin; ++i) {
            const lct_header *h = a.in[i].hdr;
            if (!st) st = h->status;
            ok = ok && h->magic == LCT_MAGIC && h->n == a.in[i].n && h->level == a.in[i].level &&
                 h->cb_hash == a.cb[i].hash;
        }
        if (!st && !ok) st = LCT_ERR_CORRUPT;
        const int delta = a.in[0].hdr->delta;
        lct_header *h = a.w_out.hdr;
        h->magic = LCT_MAGIC;
        h->version = 1;
        h->n = a.w_out.n;
        h->level = a.w_out.level;
        h->delta = delta;
        h->status = st;
        h->cb_hash = a.cb[0].hash;
        h->ovf_used = 0;
        h->ovf_cap = a.w_out.ovf_cap;
    }
}

// One stream of one compressed input inside the kernel.
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
// the stream's spilled symbols; unless every one is kept the rows are a ring.
template <bool KEEP_ALL, int SP>
__device__ __forceinline__ uint32_t stage_row(uint32_t t)
{
    return KEEP_ALL ? t : (t & (SP - 1));
}

template <int LEVEL, bool INPLACE, int OP>
__global__ void __launch_bounds__(kSgdThreads, SgdSmem<LEVEL, INPLACE, UpdateOp<OP>::kInputs>::kCtas)
    k_update(const __grid_constant__ UpdateArgs a)
{
    using G = Geo<LEVEL>;
    using Op = UpdateOp<OP>;
    constexpr int NIN = Op::kInputs;
    using L = SgdSmem<LEVEL, INPLACE, NIN>;
    constexpr int W = G::W, R = kSgdRows, S = L::kStages, SP = L::kSpillRows;
    constexpr int NW = kSgdThreads / 32;
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *slot[NIN];
    uint8_t *sf_s[NIN];
    uint32_t *lut[NIN];
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        slot[i] = reinterpret_cast<uint32_t *>(smem + i * L::kSlotIn);
        sf_s[i] = smem + NIN * L::kSlotIn + i * L::kRing;
        lut[i] = reinterpret_cast<uint32_t *>(smem + NIN * (L::kSlotIn + L::kRing)) + i * 256;
    }
    uint2 *tbl = reinterpret_cast<uint2 *>(lut[0] + NIN * 256);
    uint8_t *ring = reinterpret_cast<uint8_t *>(tbl + 256);
    __shared__ __align__(8) uint64_t bar_slot, bar_sf[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_flags;  // bit 0: a wait gave up, bit 1: corrupt input

    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.in[0].n - base);
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
    bool bad = false;
    const int delta_w = a.w_out.hdr->delta;  // the prologue copied W's shift
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        const lct_header *h = a.in[i].hdr;
        bad |= !(h->magic == LCT_MAGIC && h->n == a.in[i].n && h->level == LEVEL && h->cb_hash == a.cb[i].hash);
        lut[i][j] = dec_entry(a.cb[i], i == 0 ? delta_w : h->delta, j);
        slot[i][W * kStreams + j] = 0u;
    }
    tbl[j] = enc_entry(a.cb[0], delta_w, j);
    __syncthreads();  // barriers initialised
    auto issue = [&](uint32_t c) {
        mbar_expect_tx(&bar_sf[c % S], NIN * R * kStreams);
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_load(sf_s[i] + (c % S) * R * kStreams, a.in[i].sf + base + (uint64_t)c * R * kStreams,
                      R * kStreams, &bar_sf[c % S]);
    };
    if (j == 0) {
        mbar_expect_tx(&bar_slot, NIN * W * kStreams * 4);
#pragma unroll
        for (int i = 0; i < NIN; ++i)
            bulk_load(slot[i], a.in[i].slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
        for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) issue(c);
    }

    // input markers, spill prefixes and overflow ranges
    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    InStream in[NIN];
    bool ovf_ok[NIN];
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        in[i].col = slot[i] + j;
        const uint32_t mk = a.in[i].markers[(uint64_t)b * kStreams + j];
        bad |= mk > nj;
        in[i].marker = min(mk, nj);
        uint32_t tot;
        const uint32_t pre = group_exclusive_scan(nj - in[i].marker, warp_tot, NW, 0, &tot);
        const uint64_t o0 = a.in[i].blk_off[b], o1 = a.in[i].blk_off[b + 1];
        ovf_ok[i] = o1 <= a.in[i].ovf_cap && o0 <= o1 && o1 - o0 == tot;
        in[i].ovf_at = o0 + pre - in[i].marker;
        bad |= !ovf_ok[i];
        in[i].pos = 0;
    }

    if (!mbar_wait(&bar_slot, 0, limit)) s_flags = 1;
    Writer wo;
    wr_init<W>(wo, nj);
    uint32_t *colO = a.w_out.slots + (uint64_t)b * W * kStreams + j;
    uint8_t *sfj = a.w_out.sf + base + j;
    uint8_t *ringj = ring + j;
    float k[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) k[i] = a.k[i];

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot_c = c % S;
        if (bulk && !mbar_wait(&bar_sf[slot_c], (c / S) & 1u, (s_flags & 1u) ? 1000000ull : limit)) s_flags = 1;
        uint8_t *sfo = sfj + (uint64_t)c * R * kStreams;
        const uint32_t kend = (c + 1) * R;
        bool in_slot = true;
#pragma unroll
        for (int i = 0; i < NIN; ++i) in_slot = in_slot && in[i].marker >= kend;
        if (bulk && __all_sync(kFull, in_slot)) {
            // loads first (the decode chains, the sign-fraction bytes, the
            // new values' code-table entries), stores last, so nothing orders
            // a load behind a store
            uint32_t e[NIN][R], h[R], need = 0;
            uint2 ent[R];
#pragma unroll
            for (int r = 0; r < R; r += 2) {
#pragma unroll
                for (int i = 0; i < NIN; ++i) rd_take2<W>(in[i].pos, in[i].col, lut[i], e[i][r], e[i][r + 1]);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                uint32_t x[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i) x[i] = join_one(sf_s[i][slot_c * R * kStreams + r * kStreams + j], e[i][r]);
                h[r] = Op::apply(x, k);
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ent[r] = code_of(tbl, h[r]);
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
                    const uint32_t kk = c * R + r;
                    if (wr_put_checked(wo, ent[r], kk, colO))
                        ringj[stage_row<L::kKeepAll, SP>(kk - wo.marker) * kRow] = (uint8_t)exp_of(h[r]);
                }
            }
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t kk = c * R + r;
                if (kk >= nj) break;
                const uint64_t at = base + (uint64_t)kk * kStreams + j;
                uint32_t x[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i) {
                    const uint32_t ei = in_take<W>(in[i], kk, lut[i], a.in[i].ovf, ovf_ok[i]);
                    const uint32_t fi = bulk ? sf_s[i][slot_c * R * kStreams + r * kStreams + j] : a.in[i].sf[at];
                    x[i] = join_one(fi, ei);
                }
                const uint32_t hv = Op::apply(x, k);
                const uint32_t ev = exp_of(hv);
                sfo[r * kStreams] = sf_of(hv);
                if (wr_put_checked(wo, tbl[ev], kk, colO))
                    ringj[stage_row<L::kKeepAll, SP>(kk - wo.marker) * kRow] = (uint8_t)ev;
            }
        }
        __syncthreads();  // every thread is done with this chunk's ring slot
        if (j == 0 && c + S < nbulk) issue(c + S);
    }
#pragma unroll
    for (int i = 0; i < NIN; ++i) bad |= in[i].pos > 32u * W;
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
            const uint32_t ssp = __shfl_sync(kFull, spill, i);
            const uint32_t spr = __shfl_sync(kFull, pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            const uint32_t kept_from = L::kKeepAll || ssp <= (uint32_t)SP ? 0u : ssp - SP;  // older ones were overwritten
            for (uint32_t l = lane; l < ssp; l += 32)
                if (L::kKeepAll || l >= kept_from) out[spr + l] = ring[stage_row<L::kKeepAll, SP>(l) * kRow + sj];
        }
        const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;
        if (!L::kKeepAll && marker < kept_from) {
            // This stream spilled past the kept rows: decode its inputs again
            // from the slot images (still in shared memory) and recompute the
            // older spilled exponents.  W's sign-fraction bytes are intact
            // because the step is out of place.
            InStream re[NIN];
#pragma unroll
            for (int i = 0; i < NIN; ++i) {
                re[i] = in[i];
                re[i].pos = 0;
            }
            for (uint32_t kk = 0; kk < kept_from; ++kk) {
                const uint64_t at = base + (uint64_t)kk * kStreams + j;
                uint32_t x[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i)
                    x[i] = join_one(a.in[i].sf[at], in_take<W>(re[i], kk, lut[i], a.in[i].ovf, ovf_ok[i]));
                const uint32_t hv = Op::apply(x, k);
                if (kk >= marker) out[pre + (kk - marker)] = exp_of(hv);
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

template <int LEVEL, bool INPLACE, int OP>
cudaError_t launch_level(const UpdateArgs &a, cudaStream_t s)
{
    constexpr int smem = SgdSmem<LEVEL, INPLACE, UpdateOp<OP>::kInputs>::kBytes;
    cudaError_t err =
        cudaFuncSetAttribute(k_update<LEVEL, INPLACE, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_update<LEVEL, INPLACE, OP>, dim3(a.w_out.nblocks), dim3(kSgdThreads), smem, s, a);
}

template <int LEVEL, int OP>
cudaError_t launch_update_level(const UpdateArgs &a, cudaStream_t s)
{
    return a.in_place ? launch_level<LEVEL, true, OP>(a, s) : launch_level<LEVEL, false, OP>(a, s);
}

template <int OP>
cudaError_t launch_op(const UpdateArgs &a, cudaStream_t s)
{
    switch (a.w_out.level) {
    case LCT_LEVEL_CLEAN: return launch_update_level<LCT_LEVEL_CLEAN, OP>(a, s);
    case LCT_LEVEL_MEDIUM: return launch_update_level<LCT_LEVEL_MEDIUM, OP>(a, s);
    default: return launch_update_level<LCT_LEVEL_HIGH, OP>(a, s);
    }
}

}  // namespace dev

cudaError_t launch_update(const UpdateArgs &a, cudaStream_t s)
{
    const uint32_t zero_ctas = 1 + a.w_out.nblocks / 8192;
    cudaError_t err =
        dev::launch_pdl(dev::k_update_prologue, dim3(zero_ctas < 64 ? zero_ctas : 64), dim3(256), 0, s, a);
    if (err != cudaSuccess || a.w_out.nblocks == 0) return err;
    return a.op == OP_ADAMW ? dev::launch_op<OP_ADAMW>(a, s) : dev::launch_op<OP_SGD>(a, s);
}

}  // namespace lct
