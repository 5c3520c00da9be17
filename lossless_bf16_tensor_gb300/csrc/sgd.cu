// Fused compressed SGD step of liblct: W <- W - eta*M.
//
// [EXP] "Training adds a second problem": instead of decoding W and M to HBM,
// updating, and re-encoding (three round trips), one kernel reads the
// compressed inputs, does the arithmetic, and writes the new sign-fraction
// bytes and the re-coded exponents in a single pass over each block.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

// float32 -> BF16, round to nearest even; subnormals kept; NaN -> 0x7FC0.
__device__ __forceinline__ uint32_t bf16_rne(float r)
{
    const uint32_t u = __float_as_uint(r);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0u;
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

// Two BF16 (one word) of W and M -> two updated BF16 (one word).
__device__ __forceinline__ uint32_t sgd2(uint32_t w2, uint32_t m2, float eta)
{
    const float w0 = __uint_as_float(w2 << 16), w1 = __uint_as_float(w2 & 0xFFFF0000u);
    const float m0 = __uint_as_float(m2 << 16), m1 = __uint_as_float(m2 & 0xFFFF0000u);
    const uint32_t r0 = bf16_rne(__fsub_rn(w0, __fmul_rn(eta, m0)));
    const uint32_t r1 = bf16_rne(__fsub_rn(w1, __fmul_rn(eta, m1)));
    return r0 | (r1 << 16);
}

__device__ __forceinline__ uint16_t sgd1(uint16_t w, uint16_t m, float eta)
{
    const float wf = __uint_as_float((uint32_t)w << 16), mf = __uint_as_float((uint32_t)m << 16);
    return (uint16_t)bf16_rne(__fsub_rn(wf, __fmul_rn(eta, mf)));
}

// Prologue: the new W's header (shift and codebook carried over, status
// cleared, but inheriting an error already latched in W or M) and cleared
// look-back words.
__global__ void __launch_bounds__(256) k_sgd_prologue(DevTensor w_in, DevTensor m, DevTensor w_out,
                                                       uint32_t hash_w, uint32_t hash_m)
{
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

// One CTA (512 threads) per block: threads 0..255 decode W's streams while
// 256..511 decode M's; all 512 update the values; threads 0..255 re-code.
template <int LEVEL>
__global__ void __launch_bounds__(512, 1) k_sgd(const __grid_constant__ SgdArgs a)
{
    using G = Geo<LEVEL>;
    constexpr int EB = Smem<LEVEL>::kExpBytes, SB = Smem<LEVEL>::kSlotBytes;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *eW = smem;
    uint8_t *eM = smem + EB;
    uint32_t *slotW = reinterpret_cast<uint32_t *>(smem + 2 * EB);
    uint32_t *slotM = reinterpret_cast<uint32_t *>(smem + 2 * EB + SB);
    uint32_t *lutW = reinterpret_cast<uint32_t *>(smem + 2 * EB + 2 * SB);
    uint32_t *lutM = lutW + 256;
    uint2 *tbl = reinterpret_cast<uint2 *>(lutM + 256);
    __shared__ uint32_t warp_tot[16];
    __shared__ uint32_t s_err;
    __shared__ unsigned long long s_excl;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int half = tid >> 8;  // 0: W, 1: M
    const uint32_t j = tid & 255;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.w_in.n - base);
    const DevTensor &src = half ? a.m : a.w_in;
    const DevCodebook &cb = half ? a.cbm : a.cbw;
    uint8_t *e_s = half ? eM : eW;
    uint32_t *slot_s = half ? slotM : slotW;
    uint32_t *lut = half ? lutM : lutW;

    if (tid == 0) s_err = 0;
    const lct_header *hs = src.hdr;
    const bool hdr_ok = hs->magic == LCT_MAGIC && hs->n == src.n && hs->level == LEVEL && hs->cb_hash == cb.hash;
    const int delta = hs->delta;
    const int delta_w = a.w_in.hdr->delta;
    lut[j] = dec_entry(cb, delta, (int)j);
    if (half == 0) tbl[j] = enc_entry(a.cbw, delta_w, (int)j);
    {
        const uint4 *sv = reinterpret_cast<const uint4 *>(src.slots + (uint64_t)b * G::W * kStreams);
        uint4 *dv = reinterpret_cast<uint4 *>(slot_s);
#pragma unroll 5
        for (int w = j; w < G::W * kStreams / 4; w += 256) dv[w] = __ldcs(sv + w);
        slot_s[G::W * kStreams + j] = 0u;
    }
    const uint32_t nj = nb > j ? (nb - j + 255) / 256 : 0;
    uint32_t marker = src.markers[(uint64_t)b * kStreams + j];
    bool bad = !hdr_ok || marker > nj;
    marker = min(marker, nj);
    uint32_t spill = nj - marker;
    uint32_t total;
    uint32_t pre = group_exclusive_scan(spill, warp_tot, 8, half * 8, &total);  // syncs
    const uint64_t off0 = src.blk_off[b], off1 = src.blk_off[b + 1];
    const bool ovf_ok = off1 <= src.ovf_cap && off0 <= off1 && off1 - off0 == total;
    bad |= !ovf_ok;

    // ---- decode W (half 0) and M (half 1) side by side
    const uint32_t bits = decode_stream<G::W>(slot_s + j, marker, lut, e_s + j);
    bad |= bits > 32u * G::W;
    if (bad) atomicCAS(&s_err, 0u, (uint32_t)LCT_ERR_CORRUPT);
    if (total > 0 && ovf_ok) {
        const uint8_t *in = src.ovf + off0;
        for (int i = 0; i < 32; ++i) {
            const uint32_t sm = __shfl_sync(0xFFFFFFFFu, marker, i);
            const uint32_t sp = __shfl_sync(0xFFFFFFFFu, spill, i);
            const uint32_t so = __shfl_sync(0xFFFFFFFFu, pre, i);
            const uint32_t sj = (uint32_t)((warp & 7) * 32 + i);
            for (uint32_t l = lane; l < sp; l += 32) e_s[(sm + l) * kRow + sj] = __ldg(in + so + l);
        }
    }
    __syncthreads();

    // ---- update, 8 values per step: new sign-fraction bytes out, new
    //      exponents back into W's staging rows
    {
        const uint2 *sfw = reinterpret_cast<const uint2 *>(a.w_in.sf + base);
        const uint2 *sfm = reinterpret_cast<const uint2 *>(a.m.sf + base);
        uint2 *sfo = reinterpret_cast<uint2 *>(a.w_out.sf + base);
        const uint32_t ng = nb >> 3;
        const float eta = a.eta;
#pragma unroll 2
        for (uint32_t g = tid; g < ng; g += 512) {
            const uint2 sw = __ldcs(sfw + g), sm = __ldcs(sfm + g);
            uint32_t *ew = reinterpret_cast<uint32_t *>(stage_at(eW, g << 3));
            const uint32_t *em = reinterpret_cast<const uint32_t *>(stage_at(eM, g << 3));
            const uint4 vw = join8(sw, make_uint2(ew[0], ew[1]));
            const uint4 vm = join8(sm, make_uint2(em[0], em[1]));
            uint4 r;
            r.x = sgd2(vw.x, vm.x, eta);
            r.y = sgd2(vw.y, vm.y, eta);
            r.z = sgd2(vw.z, vm.z, eta);
            r.w = sgd2(vw.w, vm.w, eta);
            uint2 sf, ex;
            split8(r, sf, ex);
            __stcs(sfo + g, sf);
            ew[0] = ex.x;
            ew[1] = ex.y;
        }
        for (uint32_t i = (ng << 3) + tid; i < nb; i += 512) {
            const uint16_t w = join1(a.w_in.sf[base + i], *stage_at(eW, i));
            const uint16_t m = join1(a.m.sf[base + i], *stage_at(eM, i));
            const uint16_t r = sgd1(w, m, eta);
            a.w_out.sf[base + i] = sf_of(r);
            *stage_at(eW, i) = exp_of(r);
        }
    }
    __syncthreads();

    // ---- re-code W with its codebook and its stored shift
    uint32_t new_marker = 0, new_spill = 0;
    if (half == 0) {
        if (nb == (uint32_t)G::B)
            new_marker = encode_stream<G::W, G::NJ>(eW + j, nj, tbl, slotW + j);
        else
            new_marker = encode_stream<G::W, 0>(eW + j, nj, tbl, slotW + j);
        new_spill = nj - new_marker;
    }
    uint32_t new_total;
    const uint32_t new_pre = group_exclusive_scan(new_spill, warp_tot, 8, 0, &new_total);  // syncs
    {
        const uint4 *sv = reinterpret_cast<const uint4 *>(slotW);
        uint4 *dv = reinterpret_cast<uint4 *>(a.w_out.slots + (uint64_t)b * G::W * kStreams);
        for (int w = tid; w < G::W * kStreams / 4; w += 512) __stcs(dv + w, sv[w]);
        if (half == 0) a.w_out.markers[(uint64_t)b * kStreams + j] = (uint16_t)new_marker;
    }

    // ---- the prologue has cleared W_out's header and look-back words
    pdl_wait();
    if (tid == 0) {
        if (s_err) latch(a.w_out.hdr, s_err);
        bool timed_out;
        const unsigned long long excl = lookback(a.w_out.work, b, new_total, a.wait_ns, &timed_out);
        if (timed_out) latch(a.w_out.hdr, LCT_ERR_TIMEOUT);
        a.w_out.blk_off[b] = excl;
        if (b == a.w_out.nblocks - 1) {
            a.w_out.blk_off[b + 1] = excl + new_total;
            a.w_out.hdr->ovf_used = excl + new_total;
        }
        if (excl + new_total > a.w_out.ovf_cap) latch(a.w_out.hdr, LCT_ERR_OVERFLOW_CAPACITY);
        s_excl = excl;
    }
    __syncthreads();
    const unsigned long long excl = s_excl;
    if (half == 0 && new_total > 0 && excl + new_total <= a.w_out.ovf_cap) {
        uint8_t *out = a.w_out.ovf + excl;
        for (int i = 0; i < 32; ++i) {
            const uint32_t sm = __shfl_sync(0xFFFFFFFFu, new_marker, i);
            const uint32_t sp = __shfl_sync(0xFFFFFFFFu, new_spill, i);
            const uint32_t so = __shfl_sync(0xFFFFFFFFu, new_pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            for (uint32_t l = lane; l < sp; l += 32) out[so + l] = eW[(sm + l) * kRow + sj];
        }
    }
}

template <int LEVEL>
cudaError_t launch_level(const SgdArgs &a, cudaStream_t s)
{
    constexpr int smem = 2 * Smem<LEVEL>::kExpBytes + 2 * Smem<LEVEL>::kSlotBytes + 2 * 256 * 4 + 256 * 8;
    cudaError_t err = cudaFuncSetAttribute(k_sgd<LEVEL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.w_out.nblocks);
    cfg.blockDim = dim3(512);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_sgd<LEVEL>, a);
}

}  // namespace dev

cudaError_t launch_sgd(const SgdArgs &a, cudaStream_t s)
{
    const uint32_t zero_ctas = 1 + a.w_out.nblocks / 8192;
    dev::k_sgd_prologue<<<zero_ctas < 64 ? zero_ctas : 64, 256, 0, s>>>(a.w_in, a.m, a.w_out, a.cbw.hash, a.cbm.hash);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.w_out.nblocks == 0) return err;
    switch (a.w_out.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
