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
// bulk copy; their sign-fraction bytes stream through a ring of row chunks
// that a producer warp keeps filled.  Rows go in groups of four: a group in
// which no input symbol of a warp's streams lies past its spill marker takes
// a fast path (symbols decoded two at a time, values rounded two at a time,
// the fit check per value only when some new slot may not hold the group);
// the rows from a warp's first spilled input symbol on go row by row.  A code
// is at most 16 bits, so a stream holds at least 2W symbols of its slot and
// spills at most NJ - 2W.  That many spilled new exponents are kept in place
// and for the 128-row levels (MEDIUM, HIGH).  Out of place in CLEAN 32 rows
// are kept (three CTAs per SM for the SGD), and a stream that spills more
// than that re-decodes its older rows at the end.  Where a block's latency,
// not the SM's throughput, sets the time -- grids of at most two blocks per
// SM for the SGD, and every in-place step (one CTA per SM) -- a
// software-pipelined instantiation runs (16-row chunks).
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kSgdThreads = 256;                 // consumer threads: one per stream
constexpr int kSgdBlock = kSgdThreads + 32;      // and one producer warp
constexpr int kSgdRows = 8;        // rows per sign-fraction chunk
constexpr int kSgdRowsClean = 8;   // rows per chunk out of place in CLEAN
constexpr int kSgdRowsPipe = 16;   // rows per chunk of the software-pipelined small-grid kernel
constexpr int kSgdSpill = 32;      // spilled new-exponent rows kept (out of place in CLEAN; 0 or a power of two)

template <int OP>
struct UpdateOp;

// W' = bf16(fl32(w - fl32(k0*m))): product and difference rounded separately
// (apply takes the inputs as float32 and returns the float32 result; the
// caller rounds it to BF16).  With finite inputs and a finite eta the result
// is never NaN (an overflowing product gives an infinity, not inf - inf).
template <>
struct UpdateOp<OP_SGD> {
    static constexpr int kInputs = 2;
    static constexpr bool kTryCopy = true;  // a small step: the exponents mostly stay
    static constexpr bool kNanFree = true;  // given finite inputs and a finite k[0]
    __device__ static __forceinline__ float apply(const float (&x)[2], const float *k)
    {
        return __fsub_rn(x[0], __fmul_rn(k[0], x[1]));
    }
};

// W' = bf16((w - k7*w) - (k4*m) / (sqrt(v)*k5 + k6)), each operation rounded
// on its own (sqrt and the division correctly rounded).
template <>
struct UpdateOp<OP_ADAMW> {
    static constexpr int kInputs = 3;
    static constexpr bool kTryCopy = false;  // steps of about lr: exponents change too often to try
    static constexpr bool kNanFree = false;  // sqrt of a negative input, 0/0
    __device__ static __forceinline__ float apply(const float (&x)[3], const float *k)
    {
        const float w = x[0];
        const float den = __fadd_rn(__fmul_rn(__fsqrt_rn(x[2]), k[5]), k[6]);
        const float upd = __fdiv_rn(__fmul_rn(k[4], x[1]), den);
        return __fsub_rn(__fsub_rn(w, __fmul_rn(k[7], w)), upd);
    }
};

template <int LEVEL, bool INPLACE, int NIN, bool PIPE = false>
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
    static constexpr int kRows = PIPE ? kSgdRowsPipe : (kKeepAll ? kSgdRows : kSgdRowsClean);  // rows per chunk
    static constexpr int kRing = kStages * kRows * kStreams;  // per input
    static constexpr int kLuts = NIN * 256 * 4 + 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;
    static constexpr int kBytes = NIN * kSlotIn + NIN * kRing + kLuts + kSpill;
    // CTAs per SM the launch bounds ask for: as many as fit the SM's 228 KB
    // (1 KB of it reserved per CTA), at most 3 for the SGD and 2 for AdamW
    static constexpr int kFit = 228 * 1024 / (kBytes + 1024 + 256);
    static constexpr int kWant = INPLACE ? 1 : (PIPE ? 2 : (NIN == 2 ? 3 : 2));
    static constexpr int kCtas = kFit < kWant ? kFit : kWant;
    static_assert(kKeepAll || (kSgdSpill & (kSgdSpill - 1)) == 0, "ring index uses a mask");
    static_assert(kRows % 4 == 0, "four-row groups");
    static_assert(kRows * 16 < 1024, "a chunk's advance fits the positions' exact low 10 bits");
    static_assert(kBytes <= 227 * 1024 && kCtas >= 1, "shared memory of one CTA");
    // the pair reader's reads from the last slot image stay inside the CTA
    static_assert((NIN - 1) * kSlotIn + 33 * 1024 <= kBytes, "33 KB after every slot image");
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

// Symbol k of an input stream as a float-ready decode-table entry (exponent
// in bits 23..30, literal added).
template <int W>
__device__ __forceinline__ uint32_t in_take(InStream &s, uint32_t k, const uint32_t *lut, const uint8_t *ovf,
                                            bool ovf_ok)
{
    if (k < s.marker) return rd_take_f<W>(s.pos, s.col, lut);
    return ovf_ok ? (uint32_t)__ldg(ovf + s.ovf_at + k) << 23 : 0u;
}

// Slot of a spilled new exponent in the staging rows: t = k - marker counts
// the stream's spilled symbols; unless every one is kept the rows are a ring.
template <bool KEEP_ALL, int SP>
__device__ __forceinline__ uint32_t stage_row(uint32_t t)
{
    return KEEP_ALL ? t : (t & (SP - 1));
}

// The four rows' values of a group from their entries (literals added) and
// sign-fraction bytes: updated, rounded two at a time (NaN canonicalised when
// CANON), sign-fraction bytes written; `same` collects where the new values
// differ from the old weight's.
template <int NIN, typename Op, bool CANON>
__device__ __forceinline__ void round_group(const uint32_t (&ev)[NIN][4], uint8_t *const (&sf_s)[NIN], uint32_t sf_at,
                                            const float *k, uint32_t mz, uint32_t (&P)[2], uint32_t &same,
                                            uint8_t *sfo)
{
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float r[2];
        uint32_t xw[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            float x[NIN];
#pragma unroll
            for (int i = 0; i < NIN; ++i) {
                const uint32_t f = join_f(sf_s[i][sf_at + (2 * q + t) * kStreams], ev[i][2 * q + t], mz);
                x[i] = __uint_as_float(f);
                if (i == 0) xw[t] = f;
            }
            r[t] = Op::apply(x, k);
        }
        P[q] = bf16x2_rn(r[0], r[1]);
        if (CANON) P[q] = nan_canon2(P[q]);
        if (Op::kTryCopy) same |= P[q] ^ __byte_perm(xw[0], xw[1], 0x7632);  // old weight values, packed the same way
        const uint32_t sfp = sf_of2(P[q]);
        sfo[(2 * q) * kStreams] = (uint8_t)sfp;
        sfo[(2 * q + 1) * kStreams] = (uint8_t)(sfp >> 16);
    }
}

// The decoded symbols of one group of four rows: windows and entries per
// input, the warp-wide OR of the entries (escape flags) and the old weight's
// bits of these rows.
template <int NIN>
struct GroupIn {
    uint32_t wv[NIN][4], ev[NIN][4], esc, bc;
};

// Four rows of every input stream, two symbols at a time, with raw
// float-ready entries (the positions carry the entries' upper fields above
// bit 9; the caller restores exact positions after the chunk).
template <int NIN>
__device__ __forceinline__ void decode_group(InStream (&in)[NIN], const uint32_t (&col_s)[NIN],
                                             const uint32_t (&lut_s)[NIN], const Mul mul, GroupIn<NIN> &d)
{
    d.esc = 0;
    const uint32_t p0 = in[0].pos;
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int i = 0; i < NIN; ++i) {
            Rd r{in[i].pos, col_s[i]};
            rd_pair_f(r, lut_s[i], mul, d.wv[i][2 * q], d.wv[i][2 * q + 1], d.ev[i][2 * q], d.ev[i][2 * q + 1]);
            in[i].pos = r.p;
            d.esc |= d.ev[i][2 * q] | d.ev[i][2 * q + 1];
        }
    d.bc = (in[0].pos - p0) & 0x3FFu;
}

// Escape literals into the group's entries (a coded symbol's is a no-op).
template <int NIN>
__device__ __forceinline__ void fix_group(GroupIn<NIN> &d)
{
#pragma unroll
    for (int i = 0; i < NIN; ++i)
#pragma unroll
        for (int t = 0; t < 4; ++t) d.ev[i][t] = lit_fix_f(d.wv[i][t], d.ev[i][t]);
}

// The new codes of a group whose values are rounded (P, two BF16 per word;
// `same` the difference from the old weight's values).  When no new exponent
// of the warp's streams differs from the old weight's, the new codes are the
// old weight's codes bit for bit (same codebook, same stored shift), so the
// rows' bits are appended straight from the old weight's stream window.
// Otherwise the new codes are looked up and appended, with the fit check per
// value only when some stream of the warp may not keep all four.
template <int NIN, typename Op, bool KEEP_ALL, int SP>
__device__ __forceinline__ void write_group(const GroupIn<NIN> &d, const uint32_t (&P)[2], uint32_t same,
                                            const uint2 *tbl, Writer &wo, uint32_t *colO, uint8_t *ringj,
                                            uint32_t k0)
{
    const uint32_t bc = d.bc;
    if (Op::kTryCopy && __all_sync(kFull, wo.alive && !(same & 0x7F807F80u) && bc <= 32u && bc <= wo.rem)) {
        wr_add(wo, make_uint2(d.wv[0][0] & ~(0xFFFFFFFFu >> bc), bc));
        wr_flush(wo, colO);
        wo.rem -= bc;
        return;
    }
    const uint32_t h[4] = {P[0], P[0] >> 16, P[1], P[1] >> 16};
    uint2 ent[4];
    uint32_t need = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        ent[t] = code_of(tbl, h[t]);
        need += ent[t].y;
    }
    if (__all_sync(kFull, wo.alive && need <= wo.rem)) {
        wr_add2(wo, ent[0], ent[1]);
        wr_flush(wo, colO);
        wr_add2(wo, ent[2], ent[3]);
        wr_flush(wo, colO);
        wo.rem -= need;
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t kk = k0 + t;
            if (wr_put_checked(wo, ent[t], kk, colO) && SP > 0)
                ringj[stage_row<KEEP_ALL, SP>(kk - wo.marker) * kRow] = (uint8_t)exp_of(h[t]);
        }
    }
}

// One fast-path chunk (every input symbol of its rows lies in its slot),
// group by group.  A warp adds escape literals, and canonicalises NaN, only
// when one of its lanes met an escape or an exponent of 255 (or every group
// does when canon_all); with no such symbol and finite inputs an SGD step
// cannot produce NaN.
template <int W, int NIN, typename Op, bool KEEP_ALL, int SP, int G>
__device__ __forceinline__ void update_chunk(InStream (&in)[NIN], const uint32_t (&col_s)[NIN],
                                             const uint32_t (&lut_s)[NIN], const Mul mul,
                                             uint8_t *const (&sf_s)[NIN], uint32_t sf_at, const float *k,
                                             bool canon_all, const uint2 *tbl, Writer &wo, uint32_t *colO,
                                             uint8_t *sfo, uint8_t *ringj, uint32_t k0)
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        GroupIn<NIN> d;
        decode_group(in, col_s, lut_s, mul, d);
        uint32_t P[2], same = 0;
        if (__any_sync(kFull, d.esc & kEntFlag) || canon_all) {
            fix_group(d);
            round_group<NIN, Op, true>(d.ev, sf_s, sf_at + g * 4 * kStreams, k, mul.z, P, same, sfo + g * 4 * kStreams);
        } else {
            round_group<NIN, Op, !Op::kNanFree>(d.ev, sf_s, sf_at + g * 4 * kStreams, k, mul.z, P, same,
                                                sfo + g * 4 * kStreams);
        }
        write_group<NIN, Op, KEEP_ALL, SP>(d, P, same, tbl, wo, colO, ringj, k0 + 4 * g);
    }
}

// The same chunk software-pipelined for grids of at most two blocks per SM,
// where a block's time is the latency of its streams' serial work: the next
// group's symbols are decoded (and their literals added, unconditionally)
// in the same straight-line code as this group's arithmetic and rounding
// (NaN always canonicalised), so that a warp, which issues in order, overlaps
// the two instead of waiting out the decode chain after every write.
template <int W, int NIN, typename Op, bool KEEP_ALL, int SP, int G>
__device__ __forceinline__ void update_chunk_pipelined(InStream (&in)[NIN], const uint32_t (&col_s)[NIN],
                                                       const uint32_t (&lut_s)[NIN], const Mul mul,
                                                       uint8_t *const (&sf_s)[NIN], uint32_t sf_at, const float *k,
                                                       const uint2 *tbl, Writer &wo, uint32_t *colO, uint8_t *sfo,
                                                       uint8_t *ringj, uint32_t k0)
{
    GroupIn<NIN> d[2];
    decode_group(in, col_s, lut_s, mul, d[0]);
    fix_group(d[0]);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (g + 1 < G) {
            decode_group(in, col_s, lut_s, mul, d[(g + 1) & 1]);
            fix_group(d[(g + 1) & 1]);
        }
        uint32_t P[2], same = 0;
        round_group<NIN, Op, true>(d[g & 1].ev, sf_s, sf_at + g * 4 * kStreams, k, mul.z, P, same,
                                   sfo + g * 4 * kStreams);
        write_group<NIN, Op, KEEP_ALL, SP>(d[g & 1], P, same, tbl, wo, colO, ringj, k0 + 4 * g);
    }
}

template <int LEVEL, bool INPLACE, int OP, bool PIPE>
__global__ void __launch_bounds__(kSgdBlock, SgdSmem<LEVEL, INPLACE, UpdateOp<OP>::kInputs, PIPE>::kCtas)
    k_update(const __grid_constant__ UpdateArgs a)
{
    using G = Geo<LEVEL>;
    using Op = UpdateOp<OP>;
    constexpr int NIN = Op::kInputs;
    using L = SgdSmem<LEVEL, INPLACE, NIN, PIPE>;
    constexpr int W = G::W, R = L::kRows, S = L::kStages, SP = L::kSpillRows;
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
    uint32_t col_s[NIN], lut_s[NIN];
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        col_s[i] = smem_addr(slot[i] + threadIdx.x);
        lut_s[i] = smem_addr(lut[i]);
    }
    const Mul mul{a.mul_row, a.mul_ent, a.mul_sf};
    // bar_sf[s]: stage s of the ring has landed; bar_free[s]: every consumer
    // warp is done with stage s (the producer may refill it)
    __shared__ __align__(8) uint64_t bar_slot, bar_sf[S], bar_free[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_flags;  // bit 0: a wait gave up, bit 1: corrupt input

    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.in[0].n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    if (warp == NW) {
        // Producer warp: initialise the barriers, issue the slot images and
        // the first stages of the ring at once, then refill each stage as soon
        // as all consumer warps have released it.
        if (lane == 0) {
            mbar_init(&bar_slot, 1);
            for (int s = 0; s < S; ++s) {
                mbar_init(&bar_sf[s], 1);
                mbar_init(&bar_free[s], NW);
            }
            fence_mbar_init();
            s_flags = 0;
        }
        pdl_wait();  // the inputs are complete
        auto issue = [&](uint32_t c) {
            const uint32_t st = c % S;
            mbar_expect_tx(&bar_sf[st], NIN * R * kStreams);
#pragma unroll
            for (int i = 0; i < NIN; ++i)
                bulk_load(sf_s[i] + st * R * kStreams, a.in[i].sf + base + (uint64_t)c * R * kStreams, R * kStreams,
                          &bar_sf[st]);
        };
        if (lane == 0) {
            mbar_expect_tx(&bar_slot, NIN * W * kStreams * 4);
#pragma unroll
            for (int i = 0; i < NIN; ++i)
                bulk_load(slot[i], a.in[i].slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
            for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) issue(c);
        }
        __syncthreads();  // barriers initialised, tables built
        if (lane == 0) {
            bool gave_up = false;
            for (uint32_t c = S; c < nbulk; ++c) {
                if (!mbar_wait(&bar_free[c % S], (c / S - 1) & 1u, gave_up ? 1000000ull : limit)) gave_up = true;
                issue(c);
            }
            if (gave_up) atomicOr(&s_flags, 1u);
        }
        return;
    }

    // Consumer warps, thread j = stream j.  Every global read of the block's
    // start is issued before the first barrier so that their latencies overlap.
    pdl_wait();  // inputs, the new header and the cleared look-back words are all ready
    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    const int delta_w = a.w_out.hdr->delta;  // the prologue copied W's shift
    uint32_t mk[NIN];
    uint64_t o0[NIN], o1[NIN];
    bool bad = false;
    int delta_in[NIN];
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        mk[i] = a.in[i].markers[(uint64_t)b * kStreams + j];
        o0[i] = a.in[i].blk_off[b];
        o1[i] = a.in[i].blk_off[b + 1];
        const lct_header *h = a.in[i].hdr;
        bad |= !(h->magic == LCT_MAGIC && h->n == a.in[i].n && h->level == LEVEL && h->cb_hash == a.cb[i].hash);
        delta_in[i] = h->delta;
    }
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        lut[i][j] = dec_entry_f(a.cb[i], i == 0 ? delta_w : delta_in[i], j);
        slot[i][W * kStreams + j] = 0u;
    }
    tbl[j] = enc_entry(a.cb[0], delta_w, j);
    __syncthreads();  // barriers initialised, tables built

    // input markers, spill prefixes and overflow ranges
    InStream in[NIN];
    bool ovf_ok[NIN];
#pragma unroll
    for (int i = 0; i < NIN; ++i) {
        in[i].col = slot[i] + j;
        bad |= mk[i] > nj;
        in[i].marker = min(mk[i], nj);
        uint32_t tot;
        const uint32_t pre = group_exclusive_scan<1, kSgdThreads>(nj - in[i].marker, warp_tot, NW, 0, &tot);
        ovf_ok[i] = o1[i] <= a.in[i].ovf_cap && o0[i] <= o1[i] && o1[i] - o0[i] == tot;
        in[i].ovf_at = o0[i] + pre - in[i].marker;
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
    const bool canon_all = !isfinite(k[0]);  // a non-finite eta can make NaN from finite inputs

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
            const uint32_t sf_at = slot_c * R * kStreams;
            uint32_t p_start[NIN];
#pragma unroll
            for (int i = 0; i < NIN; ++i) p_start[i] = in[i].pos;
            if (PIPE)
                update_chunk_pipelined<W, NIN, Op, L::kKeepAll, SP, R / 4>(in, col_s, lut_s, mul, sf_s, sf_at + j, k,
                                                                           tbl, wo, colO, sfo, ringj, c * R);
            else
                update_chunk<W, NIN, Op, L::kKeepAll, SP, R / 4>(in, col_s, lut_s, mul, sf_s, sf_at + j, k, canon_all,
                                                                 tbl, wo, colO, sfo, ringj, c * R);
            // exact positions again: a chunk advances a stream by at most
            // R * 16 < 1024 bits, which the low 10 bits hold exactly
#pragma unroll
            for (int i = 0; i < NIN; ++i) in[i].pos = p_start[i] + ((in[i].pos - p_start[i]) & 0x3FFu);
        } else {
            int r0 = 0;
            if (bulk) {
                // The groups of this chunk that end before the warp's first
                // spilled input symbol still take the fast path, one by one;
                // only the rows from there on go row by row.  (A stream whose
                // input spilled reaches its marker in its last rows, so this
                // keeps one such stream from slowing its whole warp's chunk.)
                uint32_t first = in[0].marker;
#pragma unroll
                for (int i = 1; i < NIN; ++i) first = min(first, in[i].marker);
                const uint32_t wmin = __reduce_min_sync(kFull, first);
                const uint32_t fast = wmin > c * R ? min((wmin - c * R) / 4u, (uint32_t)(R / 4)) : 0u;
                if (fast > 0) {
                    const uint32_t sf_at = slot_c * R * kStreams;
                    uint32_t p_start[NIN];
#pragma unroll
                    for (int i = 0; i < NIN; ++i) p_start[i] = in[i].pos;
#pragma unroll 1
                    for (uint32_t g = 0; g < fast; ++g)
                        update_chunk<W, NIN, Op, L::kKeepAll, SP, 1>(in, col_s, lut_s, mul, sf_s,
                                                                     sf_at + g * 4 * kStreams + j, k, canon_all, tbl,
                                                                     wo, colO, sfo + g * 4 * kStreams, ringj,
                                                                     c * R + 4 * g);
#pragma unroll
                    for (int i = 0; i < NIN; ++i) in[i].pos = p_start[i] + ((in[i].pos - p_start[i]) & 0x3FFu);
                    r0 = 4 * (int)fast;
                }
            }
            for (int r = r0; r < R; ++r) {
                const uint32_t kk = c * R + r;
                if (kk >= nj) break;
                const uint64_t at = base + (uint64_t)kk * kStreams + j;
                float x[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i) {
                    const uint32_t ei = in_take<W>(in[i], kk, lut[i], a.in[i].ovf, ovf_ok[i]);
                    const uint32_t fi = bulk ? sf_s[i][slot_c * R * kStreams + r * kStreams + j] : a.in[i].sf[at];
                    x[i] = __uint_as_float(join_f(fi, ei, mul.z));
                }
                const uint32_t hv = bf16_rne(Op::apply(x, k));
                const uint32_t ev = exp_of(hv);
                sfo[r * kStreams] = sf_of(hv);
                if (wr_put_checked(wo, tbl[ev], kk, colO) && SP > 0)
                    ringj[stage_row<L::kKeepAll, SP>(kk - wo.marker) * kRow] = (uint8_t)ev;
            }
        }
        if (bulk) {  // this warp is done with the chunk's ring stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_free[slot_c]);
        }
    }
#pragma unroll
    for (int i = 0; i < NIN; ++i) bad |= in[i].pos > 32u * W;
    if (bad) atomicOr(&s_flags, 2u);
    wr_finish<W>(wo, colO);
    const uint32_t marker = wo.marker, spill = nj - marker;
    uint32_t total;
    const uint32_t pre = group_exclusive_scan<1, kSgdThreads>(spill, warp_tot, NW, 0, &total);
    a.w_out.markers[(uint64_t)b * kStreams + j] = (uint16_t)marker;

    // Overflow offset of this block: the single-pass decoupled look-back, or,
    // with deferred placement, a count published without waiting when the
    // block has nothing to place (k_block_offsets writes the offsets after).
    const bool leave = a.deferred && total == 0 && !lookback_leader(b);
    if (warp == 0) {
        bool timed_out = false;
        unsigned long long excl = 0;
        if (leave)
            warp_publish_try(a.w_out.work, b, 2);
        else
            excl = warp_lookback(a.w_out.work, b, total, limit, &timed_out);
        if (lane == 0) {
            if (s_flags & 2u) latch(a.w_out.hdr, LCT_ERR_CORRUPT);
            if (timed_out || (s_flags & 1u)) latch(a.w_out.hdr, LCT_ERR_TIMEOUT);
            if (!a.deferred) {
                a.w_out.blk_off[b] = excl;
                if (b == a.w_out.nblocks - 1) {
                    a.w_out.blk_off[b + 1] = excl + total;
                    a.w_out.hdr->ovf_used = excl + total;
                }
                if (excl + total > a.w_out.ovf_cap) latch(a.w_out.hdr, LCT_ERR_OVERFLOW_CAPACITY);
            }
            s_excl = excl;
        }
    }
    if (!leave) cta_sync<1, kSgdThreads>();  // uniform: total is the block's

    const unsigned long long excl = leave ? 0ull : s_excl;
    if (total > 0 && excl + total <= a.w_out.ovf_cap) {
        uint8_t *out = a.w_out.ovf + excl;
        static_assert(L::kKeepAll || kFewSpills <= (uint32_t)SP, "a few spilled rows are all still staged");
        if (__reduce_max_sync(kFull, spill) <= kFewSpills) {
            // a few spilled rows per stream, all still staged: lane by lane
            for (uint32_t l = 0; l < spill; ++l) out[pre + l] = ringj[stage_row<L::kKeepAll, SP>(l) * kRow];
        } else {
            // spilled rows still kept in shared memory: one warp per stream at a time
            for (int i = 0; i < 32; ++i) {
                const uint32_t ssp = __shfl_sync(kFull, spill, i);
                const uint32_t spr = __shfl_sync(kFull, pre, i);
                const uint32_t sj = (uint32_t)(warp * 32 + i);
                const uint32_t kept_from = L::kKeepAll || ssp <= (uint32_t)SP ? 0u : ssp - SP;  // older ones were overwritten
                for (uint32_t l = lane; l < ssp; l += 32)
                    if (L::kKeepAll || l >= kept_from) out[spr + l] = ring[stage_row<L::kKeepAll, SP>(l) * kRow + sj];
            }
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
                float x[NIN];
#pragma unroll
                for (int i = 0; i < NIN; ++i)
                    x[i] = __uint_as_float(join_f(a.in[i].sf[at], in_take<W>(re[i], kk, lut[i], a.in[i].ovf, ovf_ok[i]),
                                                  mul.z));
                const uint32_t hv = bf16_rne(Op::apply(x, k));
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

template <int LEVEL, bool INPLACE, int OP, bool PIPE>
cudaError_t launch_kernel(const UpdateArgs &b, cudaStream_t s)
{
    constexpr int smem = SgdSmem<LEVEL, INPLACE, UpdateOp<OP>::kInputs, PIPE>::kBytes;
    const cudaError_t err =
        cudaFuncSetAttribute(k_update<LEVEL, INPLACE, OP, PIPE>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(k_update<LEVEL, INPLACE, OP, PIPE>, dim3(b.w_out.nblocks), dim3(kSgdBlock), smem, s, b);
}

template <int LEVEL, bool INPLACE, int OP>
cudaError_t launch_level(const UpdateArgs &a, cudaStream_t s)
{
    UpdateArgs b = a;
    b.deferred = deferred_placement(a.w_out.nblocks);
    // The software-pipelined kernel runs where a block's latency sets the
    // time: grids of at most two blocks per SM (the SGD) and every step that
    // runs one CTA per SM anyway (in place).
    cudaError_t err;
    constexpr bool one_cta = SgdSmem<LEVEL, INPLACE, UpdateOp<OP>::kInputs, false>::kCtas == 1;
    if constexpr (OP == OP_SGD || one_cta)
        err = (one_cta || small_grid(a.w_out.nblocks)) ? launch_kernel<LEVEL, INPLACE, OP, true>(b, s)
                                                       : launch_kernel<LEVEL, INPLACE, OP, false>(b, s);
    else
        err = launch_kernel<LEVEL, INPLACE, OP, false>(b, s);
    if (err != cudaSuccess || !b.deferred) return err;
    return launch_block_offsets(a.w_out, s);
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
