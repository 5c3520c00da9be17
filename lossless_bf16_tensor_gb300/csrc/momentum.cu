// Fused compressed two-state updates of liblct, one pass reading two
// compressed tensors and a dense BF16 gradient and writing both tensors back:
//   SGD with momentum:  M <- bf16(mu*M + g),  W <- bf16(W - eta*M)
//   AdamW's moments:    M <- bf16(b1*M + (1-b1)*g),  V <- bf16(b2*V + (1-b2)*g*g)
// (the AdamW weight update then runs in the one-pass weight kernel).  Below,
// "W" and "M" name the first and second state.
//
// [EXP] "Jargon", entry "Optimizer state": the momentum buffer of SGD with
// momentum is the optimizer state the pages have in mind; [ABS]: optimizer
// states are stored compressed; [EXP] "Training adds a second problem": the
// update reads the compressed tensors and writes them back compressed in one
// pass instead of a decode / update / encode round trip through HBM.  The
// update rule is a reading (heavy ball, no dampening, no Nesterov term); every
// float32 operation is rounded on its own and the weight step uses the new
// momentum as stored, in BF16.  Each output keeps its input's codebook and
// stored shift.
//
// Thread j of a block's CTA owns stream j of W, M and of both outputs.  The
// input slot images come in by TMA bulk copy; the two sign-fraction byte
// arrays and the dense BF16 gradient stream through a ring of row chunks.
// Each output's codes are appended straight into its slot words in global
// memory (there is no shared-memory output image), which leaves room for the
// spilled new exponents of both outputs.  Spilled exponents are kept for 32
// rows per output (every row when an output is updated in place); an
// out-of-place step whose stream spills more than that recomputes the older
// rows of that stream at the end.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kMomThreads = 256;               // consumer threads: one per stream
constexpr int kMomBlock = kMomThreads + 32;    // and one producer warp
constexpr int kMomRows = 16;    // rows per chunk
constexpr int kMomRing = 2;     // chunks in flight
constexpr int kMomSpill = 32;   // spilled new-exponent rows kept per output (out of place)

// The element update of the two states a and b with the gradient g (BF16 in
// bits 0..15): returns the new a, stores the new b in *bo.
template <int OP>
struct TwoStateOp;

// SGD with momentum, a = w, b = m: b' = bf16(fl32(fl32(mu*m) + g)),
// a' = bf16(fl32(w - fl32(eta*b'))), with k0 = eta, k1 = mu.
template <>
struct TwoStateOp<OP2_MOMENTUM> {
    __device__ static __forceinline__ uint32_t apply(uint32_t w, uint32_t m, uint32_t g, const float *k, uint32_t *bo)
    {
        const uint32_t mn = bf16_rne(__fadd_rn(__fmul_rn(k[1], bf16_f(m)), bf16_f(g)));
        *bo = mn;
        return bf16_rne(__fsub_rn(bf16_f(w), __fmul_rn(k[0], bf16_f(mn))));
    }
};

// AdamW's moments, a = m, b = v: a' = bf16(fl32(k0*m) + fl32(k1*g)),
// b' = bf16(fl32(k2*v) + fl32(k3*fl32(g*g))), every operation rounded on its own.
template <>
struct TwoStateOp<OP2_ADAM_MOMENTS> {
    __device__ static __forceinline__ uint32_t apply(uint32_t m, uint32_t v, uint32_t g, const float *k, uint32_t *bo)
    {
        const float gf = bf16_f(g);
        *bo = bf16_rne(__fadd_rn(__fmul_rn(k[2], bf16_f(v)), __fmul_rn(k[3], __fmul_rn(gf, gf))));
        return bf16_rne(__fadd_rn(__fmul_rn(k[0], bf16_f(m)), __fmul_rn(k[1], gf)));
    }
};

// The same updates for two values at once (xa, xb: the two states as BF16 in
// bits 0..15, g: gradients), each result rounded to BF16 and packed
// value 0 | value 1 << 16 (pa: new first state, pb: new second state).
template <int OP>
struct TwoStateOp2;

template <>
struct TwoStateOp2<OP2_MOMENTUM> {
    __device__ static __forceinline__ void apply(const uint32_t (&w)[2], const uint32_t (&m)[2],
                                                 const uint32_t (&g)[2], const float *k, uint32_t &pa, uint32_t &pb)
    {
        pb = bf16x2_rne(__fadd_rn(__fmul_rn(k[1], bf16_f(m[0])), bf16_f(g[0])),
                        __fadd_rn(__fmul_rn(k[1], bf16_f(m[1])), bf16_f(g[1])));
        // the weight step takes the new momentum as stored (BF16)
        const float m0 = __uint_as_float(pb << 16), m1 = __uint_as_float(pb & 0xFFFF0000u);
        pa = bf16x2_rne(__fsub_rn(bf16_f(w[0]), __fmul_rn(k[0], m0)), __fsub_rn(bf16_f(w[1]), __fmul_rn(k[0], m1)));
    }
};

template <>
struct TwoStateOp2<OP2_ADAM_MOMENTS> {
    __device__ static __forceinline__ void apply(const uint32_t (&m)[2], const uint32_t (&v)[2],
                                                 const uint32_t (&g)[2], const float *k, uint32_t &pa, uint32_t &pb)
    {
        const float g0 = bf16_f(g[0]), g1 = bf16_f(g[1]);
        pb = bf16x2_rne(__fadd_rn(__fmul_rn(k[2], bf16_f(v[0])), __fmul_rn(k[3], __fmul_rn(g0, g0))),
                        __fadd_rn(__fmul_rn(k[2], bf16_f(v[1])), __fmul_rn(k[3], __fmul_rn(g1, g1))));
        pa = bf16x2_rne(__fadd_rn(__fmul_rn(k[0], bf16_f(m[0])), __fmul_rn(k[1], g0)),
                        __fadd_rn(__fmul_rn(k[0], bf16_f(m[1])), __fmul_rn(k[1], g1)));
    }
};

template <int LEVEL, bool INPLACE>
struct MomSmem {
    static constexpr int W = Geo<LEVEL>::W, NJ = Geo<LEVEL>::NJ;
    static constexpr int kSpillRows = INPLACE ? NJ : kMomSpill;
    static constexpr int kSlotIn = (W + 1) * kStreams * 4;        // + zero guard row
    static constexpr int kChunk = kMomRows * kStreams * 4;        // sf W, sf M, 2-byte g
    static constexpr int kRing = kMomRing * kChunk;
    static constexpr int kLuts = 2 * 256 * 4 + 2 * 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;  // per output
    static constexpr int kBytes = 2 * kSlotIn + kRing + kLuts + 2 * kSpill;
    static_assert(kBytes <= 227 * 1024, "shared memory of one CTA");
    static_assert(kSlotIn + 33 * 1024 <= kBytes, "the pair reader's reads stay inside the CTA");
    static_assert(kMomRows % 4 == 0, "four-row groups");
};

// Prologue: both output headers (shift and codebook carried over from the
// matching input, status cleared but inheriting an error already latched in
// W or M, or CORRUPT if either input header is not valid) and cleared
// look-back words of both outputs.  Every input header field is read before
// any output header is written, since an output header may be its input's.
__global__ void __launch_bounds__(256) k_momentum_prologue(DevTensor w_in, DevTensor m_in, DevTensor w_out,
                                                            DevTensor m_out, uint32_t hash_w, uint32_t hash_m)
{
    pdl_wait();
    pdl_launch_dependents();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < w_out.nblocks;
         i += (uint64_t)gridDim.x * blockDim.x) {
        w_out.work[i] = 0ull;
        m_out.work[i] = 0ull;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const lct_header *hw = w_in.hdr;
        const lct_header *hm = m_in.hdr;
        uint32_t st = hw->status ? hw->status : hm->status;
        const bool ok_w = hw->magic == LCT_MAGIC && hw->n == w_in.n && hw->level == w_in.level && hw->cb_hash == hash_w;
        const bool ok_m = hm->magic == LCT_MAGIC && hm->n == m_in.n && hm->level == m_in.level && hm->cb_hash == hash_m;
        if (!st && !(ok_w && ok_m)) st = LCT_ERR_CORRUPT;
        const int32_t delta_w = hw->delta, delta_m = hm->delta;
        const DevTensor *outs[2] = {&w_out, &m_out};
        const int32_t deltas[2] = {delta_w, delta_m};
        const uint32_t hashes[2] = {hash_w, hash_m};
        for (int o = 0; o < 2; ++o) {
            lct_header *h = outs[o]->hdr;
            h->magic = LCT_MAGIC;
            h->version = 1;
            h->n = outs[o]->n;
            h->level = outs[o]->level;
            h->delta = deltas[o];
            h->status = st;
            h->cb_hash = hashes[o];
            h->ovf_used = 0;
            h->ovf_cap = outs[o]->ovf_cap;
        }
    }
}

// One stream of one compressed input inside the kernel.
struct MomIn {
    uint32_t pos;         // bit position in the slot
    const uint32_t *col;  // slot image column in shared memory
    uint32_t marker;
    uint64_t ovf_at;      // overflow index of spilled symbol k is ovf_at + k
};

template <int W>
__device__ __forceinline__ uint32_t mom_take(MomIn &s, uint32_t k, const uint32_t *lut, const uint8_t *ovf, bool ovf_ok)
{
    if (k < s.marker) return rd_take<W>(s.pos, s.col, lut);
    return ovf_ok ? (uint32_t)__ldg(ovf + s.ovf_at + k) << 7 : 0u;
}

// Appends one chunk's R new exponents of one output to its stream: without
// per-code checks when every stream of the warp has room for the whole
// chunk, else one checked append per code (a spilled exponent goes to the
// staging ring).
template <int R, int SP>
__device__ __forceinline__ void mom_put_chunk(Writer &wo, const uint32_t (&h)[R], const uint2 *__restrict__ tbl,
                                              uint32_t k0, uint32_t *__restrict__ col, uint8_t *__restrict__ stage)
{
    uint2 ent[R];
    uint32_t need = 0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        ent[r] = code_of(tbl, h[r]);
        need += ent[r].y;
    }
    if (__all_sync(kFull, wo.alive && need <= wo.rem)) {
#pragma unroll
        for (int r = 0; r < R; r += 2) {  // two codes fit the accumulator, then one flush
            wr_add2(wo, ent[r], ent[r + 1]);
            wr_flush(wo, col);
        }
        wo.rem -= need;
    } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint32_t k = k0 + r;
            if (wr_put_checked(wo, ent[r], k, col)) stage[(k % SP) * kRow] = (uint8_t)exp_of(h[r]);
        }
    }
}

// Appends four new exponents of one output (packed two BF16 values per
// word in p[0], p[1]) to its stream: without per-code checks when every
// stream of the warp has room for all four, else one checked append per code
// (a spilled exponent goes to the staging ring).
template <int SP>
__device__ __forceinline__ void mom_put4(Writer &wo, const uint32_t (&p)[2], const uint2 *__restrict__ tbl,
                                         uint32_t k0, uint32_t *__restrict__ col, uint8_t *__restrict__ stage)
{
    const uint32_t h[4] = {p[0], p[0] >> 16, p[1], p[1] >> 16};
    uint2 ent[4];
    uint32_t need = 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        ent[t] = code_of(tbl, h[t]);
        need += ent[t].y;
    }
    if (__all_sync(kFull, wo.alive && need <= wo.rem)) {
        wr_add2(wo, ent[0], ent[1]);
        wr_flush(wo, col);
        wr_add2(wo, ent[2], ent[3]);
        wr_flush(wo, col);
        wo.rem -= need;
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t k = k0 + t;
            if (wr_put_checked(wo, ent[t], k, col)) stage[(k % SP) * kRow] = (uint8_t)exp_of(h[t]);
        }
    }
}

// The decoded symbols of one group of four rows of both inputs: windows and
// entries, the warp-wide OR of the entries (escape flags) and the first
// state's old bits of these rows.
struct MomGroupIn {
    uint32_t wvw[4], evw[4], wvm[4], evm[4], esc, bc;
};

// Four rows of both input streams, two symbols at a time, escape literals
// left out.
__device__ __forceinline__ void mom_decode(MomIn &sw, MomIn &sm, const uint32_t colw_s, const uint32_t colm_s,
                                           const uint32_t lutw_s, const uint32_t lutm_s, const Mul mul, MomGroupIn &d)
{
    d.esc = 0;
    const uint32_t p0 = sw.pos;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        Rd rw{sw.pos, colw_s}, rm{sm.pos, colm_s};
        rd_pair(rw, lutw_s, mul, d.wvw[2 * q], d.wvw[2 * q + 1], d.evw[2 * q], d.evw[2 * q + 1]);
        rd_pair(rm, lutm_s, mul, d.wvm[2 * q], d.wvm[2 * q + 1], d.evm[2 * q], d.evm[2 * q + 1]);
        sw.pos = rw.p;
        sm.pos = rm.p;
        d.esc |= d.evw[2 * q] | d.evw[2 * q + 1] | d.evm[2 * q] | d.evm[2 * q + 1];
    }
    d.bc = sw.pos - p0;
}

// Escape literals into the group's entries (a coded symbol's is a no-op).
__device__ __forceinline__ void mom_fix(MomGroupIn &d)
{
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        d.evw[t] = lit_fix(d.wvw[t], d.evw[t]);
        d.evm[t] = lit_fix(d.wvm[t], d.evm[t]);
    }
}

// One decoded group (literals added): both new states rounded two values at
// a time, their sign-fraction bytes written and their codes appended.  The
// first state's new codes are its old ones bit for bit when no new exponent
// of the warp's streams differs (same codebook, same stored shift): then its
// rows' bits are appended straight from the old stream window.
template <int OP, int SP>
__device__ __forceinline__ void mom_finish(const MomGroupIn &d, const uint8_t *sfwc, const uint8_t *sfmc,
                                           const uint16_t *gc, const float *kc, Writer &ow, Writer &om,
                                           const uint2 *tblW, const uint2 *tblM, uint32_t *colW, uint32_t *colM,
                                           uint8_t *sfWo, uint8_t *sfMo, uint8_t *stageW, uint8_t *stageM,
                                           uint32_t k0)
{
    using Op2 = TwoStateOp2<OP>;
    uint32_t pa[2], pb[2], same = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uint32_t xa[2] = {join_one(sfwc[(2 * q) * kStreams], d.evw[2 * q]),
                                join_one(sfwc[(2 * q + 1) * kStreams], d.evw[2 * q + 1])};
        const uint32_t xb[2] = {join_one(sfmc[(2 * q) * kStreams], d.evm[2 * q]),
                                join_one(sfmc[(2 * q + 1) * kStreams], d.evm[2 * q + 1])};
        const uint32_t g2[2] = {gc[(2 * q) * kStreams], gc[(2 * q + 1) * kStreams]};
        Op2::apply(xa, xb, g2, kc, pa[q], pb[q]);
        if (OP == OP2_MOMENTUM) same |= pa[q] ^ __byte_perm(xa[0], xa[1], 0x5410);
        const uint32_t sa = sf_of2(pa[q]), sb = sf_of2(pb[q]);
        sfWo[(2 * q) * kStreams] = (uint8_t)sa;
        sfWo[(2 * q + 1) * kStreams] = (uint8_t)(sa >> 16);
        sfMo[(2 * q) * kStreams] = (uint8_t)sb;
        sfMo[(2 * q + 1) * kStreams] = (uint8_t)(sb >> 16);
    }
    // A weight moves by a small step, so its exponents mostly stay; AdamW's
    // first moment is re-weighted every step and nearly always changes.
    constexpr bool kTryCopy = OP == OP2_MOMENTUM;
    const uint32_t bc = d.bc;
    if (kTryCopy && __all_sync(kFull, ow.alive && !(same & 0x7F807F80u) && bc <= 32u && bc <= ow.rem)) {
        wr_add(ow, make_uint2(d.wvw[0] & ~(0xFFFFFFFFu >> bc), bc));
        wr_flush(ow, colW);
        ow.rem -= bc;
    } else {
        mom_put4<SP>(ow, pa, tblW, k0, colW, stageW);
    }
    mom_put4<SP>(om, pb, tblM, k0, colM, stageM);
}

// A fast-path chunk of G groups (every symbol of both inputs in its slot),
// software-pipelined: the next group's symbols are decoded (and their
// literals added, unconditionally) in the same straight-line code as this
// group's arithmetic and rounding, so that a warp, which issues in order,
// overlaps the two.  The kernel runs one CTA per SM in place and two out of
// place, where a block's latency weighs on the time.
template <int OP, int SP, int G>
__device__ __forceinline__ void mom_chunk_pipelined(MomIn &sw, MomIn &sm, const uint32_t colw_s,
                                                    const uint32_t colm_s, const uint32_t lutw_s,
                                                    const uint32_t lutm_s, const Mul mul, const uint8_t *sfwc,
                                                    const uint8_t *sfmc, const uint16_t *gc, const float *kc,
                                                    Writer &ow, Writer &om, const uint2 *tblW, const uint2 *tblM,
                                                    uint32_t *colW, uint32_t *colM, uint8_t *sfWo, uint8_t *sfMo,
                                                    uint8_t *stageW, uint8_t *stageM, uint32_t k0)
{
    MomGroupIn d[2];
    mom_decode(sw, sm, colw_s, colm_s, lutw_s, lutm_s, mul, d[0]);
    mom_fix(d[0]);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (g + 1 < G) {
            mom_decode(sw, sm, colw_s, colm_s, lutw_s, lutm_s, mul, d[(g + 1) & 1]);
            mom_fix(d[(g + 1) & 1]);
        }
        mom_finish<OP, SP>(d[g & 1], sfwc + g * 4 * kStreams, sfmc + g * 4 * kStreams, gc + g * 4 * kStreams, kc, ow,
                           om, tblW, tblM, colW, colM, sfWo + g * 4 * kStreams, sfMo + g * 4 * kStreams, stageW,
                           stageM, k0 + 4 * g);
    }
}

template <int LEVEL, bool INPLACE, int OP>
__global__ void __launch_bounds__(kMomBlock, INPLACE ? 1 : 2) k_momentum(const __grid_constant__ MomentumArgs a)
{
    using Op = TwoStateOp<OP>;
    using G = Geo<LEVEL>;
    using L = MomSmem<LEVEL, INPLACE>;
    constexpr int W = G::W, R = kMomRows, S = kMomRing, SP = L::kSpillRows;
    constexpr int NW = kMomThreads / 32;
    constexpr int kRowsB = R * kStreams;  // bytes of one sign-fraction chunk
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *slotW = reinterpret_cast<uint32_t *>(smem);
    uint32_t *slotM = reinterpret_cast<uint32_t *>(smem + L::kSlotIn);
    uint8_t *ring = smem + 2 * L::kSlotIn;  // per chunk: sf W | sf M | g
    uint32_t *lutW = reinterpret_cast<uint32_t *>(ring + L::kRing);
    uint32_t *lutM = lutW + 256;
    uint2 *tblW = reinterpret_cast<uint2 *>(lutM + 256);
    uint2 *tblM = tblW + 256;
    uint8_t *stageW = reinterpret_cast<uint8_t *>(tblM + 256);
    uint8_t *stageM = stageW + L::kSpill;
    // bar_in[s]: stage s of the ring has landed; bar_free[s]: every consumer
    // warp is done with stage s (the producer may refill it)
    __shared__ __align__(8) uint64_t bar_slot, bar_in[S], bar_free[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl[2];
    __shared__ uint32_t s_flags;  // bit 0: a wait gave up, bit 1: corrupt input

    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.w_in.n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    auto issue = [&](uint32_t c) {
        uint8_t *dst = ring + (c % S) * L::kChunk;
        const uint64_t at = base + (uint64_t)c * kRowsB;
        mbar_expect_tx(&bar_in[c % S], L::kChunk);
        bulk_load(dst, a.w_in.sf + at, kRowsB, &bar_in[c % S]);
        bulk_load(dst + kRowsB, a.m_in.sf + at, kRowsB, &bar_in[c % S]);
        bulk_load(dst + 2 * kRowsB, a.g + at, 2 * kRowsB, &bar_in[c % S]);
    };
    if (warp == NW) {
        // Producer warp: initialise the barriers, issue the slot images and
        // the first stages of the ring at once, then refill each stage as soon
        // as all consumer warps have released it.
        if (lane == 0) {
            mbar_init(&bar_slot, 1);
            for (int s = 0; s < S; ++s) {
                mbar_init(&bar_in[s], 1);
                mbar_init(&bar_free[s], NW);
            }
            fence_mbar_init();
            s_flags = 0;
        }
        pdl_wait();  // the inputs are complete
        if (lane == 0) {
            mbar_expect_tx(&bar_slot, 2 * W * kStreams * 4);
            bulk_load(slotW, a.w_in.slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
            bulk_load(slotM, a.m_in.slots + (uint64_t)b * W * kStreams, W * kStreams * 4, &bar_slot);
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
    pdl_wait();  // inputs, the new headers and the cleared look-back words are all ready
    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    const uint32_t mw = a.w_in.markers[(uint64_t)b * kStreams + j], mm = a.m_in.markers[(uint64_t)b * kStreams + j];
    const uint64_t a0 = a.w_in.blk_off[b], a1 = a.w_in.blk_off[b + 1];
    const uint64_t c0 = a.m_in.blk_off[b], c1 = a.m_in.blk_off[b + 1];
    const lct_header *hw = a.w_in.hdr, *hm = a.m_in.hdr;
    bool bad = !(hw->magic == LCT_MAGIC && hw->n == a.w_in.n && hw->level == LEVEL && hw->cb_hash == a.cbw.hash) ||
               !(hm->magic == LCT_MAGIC && hm->n == a.m_in.n && hm->level == LEVEL && hm->cb_hash == a.cbm.hash);
    const int delta_w = a.w_out.hdr->delta, delta_m = a.m_out.hdr->delta;  // copied by the prologue
    lutW[j] = dec_entry(a.cbw, delta_w, j);
    lutM[j] = dec_entry(a.cbm, delta_m, j);
    tblW[j] = enc_entry(a.cbw, delta_w, j);
    tblM[j] = enc_entry(a.cbm, delta_m, j);
    slotW[W * kStreams + j] = 0u;
    slotM[W * kStreams + j] = 0u;
    __syncthreads();  // barriers initialised, tables built

    // input markers, spill prefixes and overflow ranges
    MomIn sw, sm;
    sw.col = slotW + j;
    sm.col = slotM + j;
    bad |= mw > nj || mm > nj;
    sw.marker = min(mw, nj);
    sm.marker = min(mm, nj);
    bool ovf_ok_w, ovf_ok_m;
    {
        uint32_t tot_w, tot_m;
        const uint32_t pre_w = group_exclusive_scan<1, kMomThreads>(nj - sw.marker, warp_tot, NW, 0, &tot_w);
        const uint32_t pre_m = group_exclusive_scan<1, kMomThreads>(nj - sm.marker, warp_tot, NW, 0, &tot_m);
        ovf_ok_w = a1 <= a.w_in.ovf_cap && a0 <= a1 && a1 - a0 == tot_w;
        ovf_ok_m = c1 <= a.m_in.ovf_cap && c0 <= c1 && c1 - c0 == tot_m;
        sw.ovf_at = a0 + pre_w - sw.marker;
        sm.ovf_at = c0 + pre_m - sm.marker;
        bad |= !ovf_ok_w || !ovf_ok_m;
    }
    const uint32_t colw_s = smem_addr(slotW + j), colm_s = smem_addr(slotM + j);
    const uint32_t lutw_s = smem_addr(lutW), lutm_s = smem_addr(lutM);
    const Mul mul{a.mul_row, a.mul_ent, a.mul_sf};
    const uint8_t *ovf_w = a.w_in.ovf, *ovf_m = a.m_in.ovf;

    if (!mbar_wait(&bar_slot, 0, limit)) s_flags = 1;
    sw.pos = 0;
    sm.pos = 0;
    Writer ow, om;
    wr_init<W>(ow, nj);
    wr_init<W>(om, nj);
    uint32_t *colW = a.w_out.slots + (uint64_t)b * W * kStreams + j;
    uint32_t *colM = a.m_out.slots + (uint64_t)b * W * kStreams + j;
    uint8_t *sfWj = a.w_out.sf + base + j;
    uint8_t *sfMj = a.m_out.sf + base + j;
    float kc[8];  // the step's constants
#pragma unroll
    for (int i = 0; i < 8; ++i) kc[i] = a.k[i];

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot = c % S;
        if (bulk && !mbar_wait(&bar_in[slot], (c / S) & 1u, (s_flags & 1u) ? 1000000ull : limit)) s_flags = 1;
        const uint8_t *chunk = ring + slot * L::kChunk;
        const uint8_t *sfwc = chunk + j;
        const uint8_t *sfmc = chunk + kRowsB + j;
        const uint16_t *gc = reinterpret_cast<const uint16_t *>(chunk + 2 * kRowsB) + j;
        const uint64_t row0 = (uint64_t)c * kRowsB;
        const uint32_t k0 = c * R, kend = k0 + R;
        if (bulk && __all_sync(kFull, sw.marker >= kend && sm.marker >= kend)) {
            mom_chunk_pipelined<OP, SP, R / 4>(sw, sm, colw_s, colm_s, lutw_s, lutm_s, mul, sfwc, sfmc, gc, kc, ow, om,
                                               tblW, tblM, colW, colM, sfWj + row0, sfMj + row0, stageW + j,
                                               stageM + j, k0);
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t k = k0 + r;
                if (k >= nj) break;
                const uint32_t ew = mom_take<W>(sw, k, lutW, ovf_w, ovf_ok_w);
                const uint32_t em = mom_take<W>(sm, k, lutM, ovf_m, ovf_ok_m);
                const uint64_t at = base + (uint64_t)k * kStreams + j;
                const uint32_t fw = bulk ? sfwc[r * kStreams] : a.w_in.sf[at];
                const uint32_t fm = bulk ? sfmc[r * kStreams] : a.m_in.sf[at];
                const uint32_t gv = bulk ? gc[r * kStreams] : a.g[at];
                uint32_t hMo;
                const uint32_t hWo = Op::apply(join_one(fw, ew), join_one(fm, em), gv, kc, &hMo);
                const uint32_t eW = exp_of(hWo), eM = exp_of(hMo);
                sfWj[row0 + r * kStreams] = sf_of(hWo);
                sfMj[row0 + r * kStreams] = sf_of(hMo);
                if (wr_put_checked(ow, tblW[eW], k, colW)) stageW[(k % SP) * kRow + j] = (uint8_t)eW;
                if (wr_put_checked(om, tblM[eM], k, colM)) stageM[(k % SP) * kRow + j] = (uint8_t)eM;
            }
        }
        if (bulk) {  // this warp is done with the chunk's ring stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_free[slot]);
        }
    }
    bad |= sw.pos > 32u * W || sm.pos > 32u * W;
    if (bad) atomicOr(&s_flags, 2u);
    wr_finish<W>(ow, colW);
    wr_finish<W>(om, colM);
    const uint32_t mk_w = ow.marker, sp_w = nj - mk_w;
    const uint32_t mk_m = om.marker, sp_m = nj - mk_m;
    uint32_t tot_w, tot_m;
    const uint32_t pre_w = group_exclusive_scan<1, kMomThreads>(sp_w, warp_tot, NW, 0, &tot_w);
    const uint32_t pre_m = group_exclusive_scan<1, kMomThreads>(sp_m, warp_tot, NW, 0, &tot_m);
    a.w_out.markers[(uint64_t)b * kStreams + j] = (uint16_t)mk_w;
    a.m_out.markers[(uint64_t)b * kStreams + j] = (uint16_t)mk_m;

    // Warp 0 places W's overflow bytes, warp 1 places M's: the single-pass
    // decoupled look-back, or, with deferred placement, a count published
    // without waiting for an output with nothing to place (k_block_offsets
    // writes the offsets after).
    const bool leave = a.deferred && tot_w == 0 && tot_m == 0 && !lookback_leader(b);
    if (warp < 2) {
        const DevTensor &t = warp == 0 ? a.w_out : a.m_out;
        const uint32_t total = warp == 0 ? tot_w : tot_m;
        bool timed_out = false;
        unsigned long long excl = 0;
        if (a.deferred && total == 0 && !lookback_leader(b))
            warp_publish_try(t.work, b, 2);
        else
            excl = warp_lookback(t.work, b, total, limit, &timed_out);
        if (lane == 0) {
            if (s_flags & 2u) latch(t.hdr, LCT_ERR_CORRUPT);
            if (timed_out || (s_flags & 1u)) latch(t.hdr, LCT_ERR_TIMEOUT);
            if (!a.deferred) {
                t.blk_off[b] = excl;
                if (b == t.nblocks - 1) {
                    t.blk_off[b + 1] = excl + total;
                    t.hdr->ovf_used = excl + total;
                }
                if (excl + total > t.ovf_cap) latch(t.hdr, LCT_ERR_OVERFLOW_CAPACITY);
            }
            s_excl[warp] = excl;
        }
    }
    if (!leave) cta_sync<1, kMomThreads>();  // uniform: the totals are the block's

    const unsigned long long excl_w = leave ? 0ull : s_excl[0], excl_m = leave ? 0ull : s_excl[1];
    const bool room_w = tot_w > 0 && excl_w + tot_w <= a.w_out.ovf_cap;
    const bool room_m = tot_m > 0 && excl_m + tot_m <= a.m_out.ovf_cap;
    uint8_t *out_w = a.w_out.ovf + excl_w;
    uint8_t *out_m = a.m_out.ovf + excl_m;
    // spilled rows still kept in shared memory: a few per stream lane by lane,
    // otherwise one warp per stream at a time
    static_assert(kFewSpills <= (uint32_t)SP, "a few spilled rows are all still staged");
    const bool few = __reduce_max_sync(kFull, max(room_w ? sp_w : 0u, room_m ? sp_m : 0u)) <= kFewSpills;
    if (few) {
        const uint32_t sj = (uint32_t)j;
        if (room_w)
            for (uint32_t l = 0; l < sp_w; ++l) out_w[pre_w + l] = stageW[((mk_w + l) % SP) * kRow + sj];
        if (room_m)
            for (uint32_t l = 0; l < sp_m; ++l) out_m[pre_m + l] = stageM[((mk_m + l) % SP) * kRow + sj];
    }
    for (int i = 0; i < (few ? 0 : 32); ++i) {
        const uint32_t sj = (uint32_t)(warp * 32 + i);
        if (room_w) {
            const uint32_t smk = __shfl_sync(kFull, mk_w, i), ssp = __shfl_sync(kFull, sp_w, i);
            const uint32_t spr = __shfl_sync(kFull, pre_w, i);
            const uint32_t kept_from = smk + ssp > (uint32_t)SP ? smk + ssp - SP : 0u;
            for (uint32_t l = lane; l < ssp; l += 32) {
                const uint32_t k = smk + l;
                if (k >= kept_from) out_w[spr + l] = stageW[(k % SP) * kRow + sj];
            }
        }
        if (room_m) {
            const uint32_t smk = __shfl_sync(kFull, mk_m, i), ssp = __shfl_sync(kFull, sp_m, i);
            const uint32_t spr = __shfl_sync(kFull, pre_m, i);
            const uint32_t kept_from = smk + ssp > (uint32_t)SP ? smk + ssp - SP : 0u;
            for (uint32_t l = lane; l < ssp; l += 32) {
                const uint32_t k = smk + l;
                if (k >= kept_from) out_m[spr + l] = stageM[(k % SP) * kRow + sj];
            }
        }
    }
    if (!INPLACE) {
        const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;
        const bool redo_w = room_w && mk_w < kept_from, redo_m = room_m && mk_m < kept_from;
        if (redo_w || redo_m) {
            // This stream spilled past the kept rows: decode its W and M again
            // from the slot images (still in shared memory) and recompute the
            // older spilled exponents.  The input sign-fraction bytes are
            // intact because the step is out of place.
            MomIn rw = sw, rm = sm;
            rw.pos = 0;
            rm.pos = 0;
            const uint32_t first = min(redo_w ? mk_w : kept_from, redo_m ? mk_m : kept_from);
            for (uint32_t k = 0; k < kept_from; ++k) {
                const uint32_t ew = mom_take<W>(rw, k, lutW, ovf_w, ovf_ok_w);
                const uint32_t em = mom_take<W>(rm, k, lutM, ovf_m, ovf_ok_m);
                if (k < first) continue;
                const uint64_t at = base + (uint64_t)k * kStreams + j;
                uint32_t hMo;
                const uint32_t hWo = Op::apply(join_one(a.w_in.sf[at], ew), join_one(a.m_in.sf[at], em), a.g[at], kc,
                                               &hMo);
                if (redo_w && k >= mk_w) out_w[pre_w + (k - mk_w)] = exp_of(hWo);
                if (redo_m && k >= mk_m) out_m[pre_m + (k - mk_m)] = exp_of(hMo);
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
            mbar_wait(&bar_in[s], (last / S) & 1u, limit);
        }
    }
}

template <int LEVEL, bool INPLACE, int OP>
cudaError_t launch_level(const MomentumArgs &a, cudaStream_t s)
{
    constexpr int smem = MomSmem<LEVEL, INPLACE>::kBytes;
    cudaError_t err =
        cudaFuncSetAttribute(k_momentum<LEVEL, INPLACE, OP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    MomentumArgs b = a;
    b.deferred = deferred_placement(a.w_out.nblocks);
    err = launch_pdl(k_momentum<LEVEL, INPLACE, OP>, dim3(a.w_out.nblocks), dim3(kMomBlock), smem, s, b);
    if (err != cudaSuccess || !b.deferred) return err;
    return launch_block_offsets2(a.w_out, a.m_out, s);
}

template <int LEVEL, int OP>
cudaError_t launch_op_level(const MomentumArgs &a, cudaStream_t s)
{
    return a.in_place ? launch_level<LEVEL, true, OP>(a, s) : launch_level<LEVEL, false, OP>(a, s);
}

template <int LEVEL>
cudaError_t launch_momentum_level(const MomentumArgs &a, cudaStream_t s)
{
    return a.op == OP2_ADAM_MOMENTS ? launch_op_level<LEVEL, OP2_ADAM_MOMENTS>(a, s)
                                    : launch_op_level<LEVEL, OP2_MOMENTUM>(a, s);
}

}  // namespace dev

cudaError_t launch_momentum(const MomentumArgs &a, cudaStream_t s)
{
    const uint32_t zero_ctas = 1 + a.w_out.nblocks / 8192;
    cudaError_t err = dev::launch_pdl(dev::k_momentum_prologue, dim3(zero_ctas < 64 ? zero_ctas : 64), dim3(256), 0,
                                      s, a.w_in, a.m_in, a.w_out, a.m_out, a.cbw.hash, a.cbm.hash);
    if (err != cudaSuccess || a.w_out.nblocks == 0) return err;
    switch (a.w_out.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_momentum_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_momentum_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_momentum_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
