// Encode path of liblct: the scale-shift prologue and the block encoder.
//
// [EXP] "In bits": split every BF16 value into a sign-fraction byte (kept as
// is) and an exponent byte; code the exponent with the precomputed codebook,
// shifted to the tensor's scale from at most 4096 samples.
// [EXP] "Compressing is easy": blocks of 65,536 (CLEAN) or 32,768 values,
// 256 streams per block dealt round-robin, fixed-length slots, uncompressed
// overflow with a per-stream spill marker.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

// Prologue (one launch per encode): CTA 0 estimates the shift and writes the
// tensor header; every CTA zeroes its share of the look-back status words.
// The block encoder is launched as a programmatic dependent and overlaps its
// load/split phase with this kernel.
__global__ void __launch_bounds__(256) k_encode_prologue(const uint16_t *__restrict__ x, DevTensor t,
                                                          int32_t median_exp, uint32_t cb_hash)
{
    pdl_launch_dependents();
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < t.nblocks;
         i += (uint64_t)gridDim.x * blockDim.x)
        t.work[i] = 0ull;
    if (blockIdx.x != 0) return;

    // Shift: m = min(n, 4096) samples at floor(k*n/m); histogram of their
    // exponents in the normal range 1..254; lower median.
    __shared__ uint32_t hist[256];
    __shared__ uint32_t wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    hist[tid] = 0;
    __syncthreads();
    const uint64_t n = t.n;
    const uint32_t m = n < (uint64_t)LCT_SHIFT_SAMPLES ? (uint32_t)n : (uint32_t)LCT_SHIFT_SAMPLES;
    for (uint32_t k = tid; k < m; k += 256) {
        const uint8_t e = exp_of(x[((uint64_t)k * n) / m]);
        if (e >= 1 && e <= 254) atomicAdd(&hist[e], 1u);
    }
    __syncthreads();
    // inclusive scan of the 256 bins (one per thread)
    const uint32_t c = hist[tid];
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    uint32_t before = 0, kept = 0;
    for (int w = 0; w < 8; ++w) {
        if (w < warp) before += wsum[w];
        kept += wsum[w];
    }
    inc += before;
    __shared__ int32_t median;
    if (tid == 0) median = -1;
    __syncthreads();
    if (kept > 0) {
        const uint32_t rank = (kept - 1) / 2;  // lower median, 0-based
        if (inc > rank && inc - c <= rank) median = tid;
    }
    __syncthreads();
    if (tid == 0) {
        int delta = 0;
        if (median >= 0) {
            delta = median - median_exp;
            delta = delta > 127 ? 127 : (delta < -127 ? -127 : delta);
        }
        lct_header *h = t.hdr;
        h->magic = LCT_MAGIC;
        h->version = 1;
        h->n = n;
        h->level = t.level;
        h->delta = delta;
        h->status = 0;
        h->cb_hash = cb_hash;
        h->ovf_used = 0;
        h->ovf_cap = t.ovf_cap;
    }
}

// One CTA per block, one thread per stream.
template <int LEVEL>
__global__ void __launch_bounds__(256, 2) k_encode(const __grid_constant__ EncodeArgs a)
{
    using G = Geo<LEVEL>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *e_s = smem;
    uint32_t *slot_s = reinterpret_cast<uint32_t *>(smem + Smem<LEVEL>::kExpBytes);
    uint2 *tbl = reinterpret_cast<uint2 *>(smem + Smem<LEVEL>::kExpBytes + Smem<LEVEL>::kSlotBytes);
    __shared__ uint32_t warp_tot[8];
    __shared__ unsigned long long s_excl;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.t.n - base);

    // ---- split: sign-fraction bytes straight out, exponents to shared rows
    {
        const uint4 *xv = reinterpret_cast<const uint4 *>(a.x + base);
        uint2 *sfv = reinterpret_cast<uint2 *>(a.t.sf + base);
        const uint32_t ng = nb >> 3;
#pragma unroll 4
        for (uint32_t g = tid; g < ng; g += 256) {
            const uint4 v = __ldcs(xv + g);
            uint2 sf, ex;
            split8(v, sf, ex);
            __stcs(sfv + g, sf);
            uint32_t *dst = reinterpret_cast<uint32_t *>(stage_at(e_s, g << 3));
            dst[0] = ex.x;
            dst[1] = ex.y;
        }
        for (uint32_t i = (ng << 3) + tid; i < nb; i += 256) {
            const uint16_t h = a.x[base + i];
            a.t.sf[base + i] = sf_of(h);
            *stage_at(e_s, i) = exp_of(h);
        }
    }

    // ---- the shift and the cleared look-back words come from the prologue
    pdl_wait();
    const int delta = a.t.hdr->delta;
    tbl[tid] = enc_entry(a.cb, delta, tid);
    __syncthreads();

    // ---- code stream `tid` into its slot
    const uint32_t j = tid;
    const uint32_t nj = nb > j ? (nb - j + 255) / 256 : 0;
    uint32_t marker;
    if (nb == (uint32_t)G::B)
        marker = encode_stream<G::W, G::NJ>(e_s + j, nj, tbl, slot_s + j);
    else
        marker = encode_stream<G::W, 0>(e_s + j, nj, tbl, slot_s + j);
    const uint32_t spill = nj - marker;
    uint32_t total;
    const uint32_t pre = group_exclusive_scan(spill, warp_tot, 8, 0, &total);  // syncs

    // ---- slots and markers out (coalesced)
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(slot_s);
        uint4 *dst = reinterpret_cast<uint4 *>(a.t.slots + (uint64_t)b * G::W * kStreams);
#pragma unroll 5
        for (int w = tid; w < G::W * kStreams / 4; w += 256) __stcs(dst + w, src[w]);
        a.t.markers[(uint64_t)b * kStreams + j] = (uint16_t)marker;
    }

    // ---- overflow offset of this block (single-pass look-back)
    if (tid == 0) {
        bool timed_out;
        const unsigned long long excl = lookback(a.t.work, b, total, a.wait_ns, &timed_out);
        if (timed_out) latch(a.t.hdr, LCT_ERR_TIMEOUT);
        a.t.blk_off[b] = excl;
        if (b == a.t.nblocks - 1) {
            a.t.blk_off[b + 1] = excl + total;
            a.t.hdr->ovf_used = excl + total;
        }
        if (excl + total > a.t.ovf_cap) latch(a.t.hdr, LCT_ERR_OVERFLOW_CAPACITY);
        s_excl = excl;
    }
    __syncthreads();

    // ---- spilled exponents, raw, in (stream, symbol) order: one warp per
    //      stream at a time, lanes over the stream's spilled symbols
    const unsigned long long excl = s_excl;
    if (total > 0 && excl + total <= a.t.ovf_cap) {
        uint8_t *out = a.t.ovf + excl;
        for (int i = 0; i < 32; ++i) {
            const uint32_t sm = __shfl_sync(0xFFFFFFFFu, marker, i);
            const uint32_t sp = __shfl_sync(0xFFFFFFFFu, spill, i);
            const uint32_t so = __shfl_sync(0xFFFFFFFFu, pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            for (uint32_t l = lane; l < sp; l += 32) out[so + l] = e_s[(sm + l) * kRow + sj];
        }
    }
}

template <int LEVEL>
cudaError_t launch_level(const EncodeArgs &a, cudaStream_t s)
{
    constexpr int smem = Smem<LEVEL>::kExpBytes + Smem<LEVEL>::kSlotBytes + 256 * 8;
    cudaError_t err = cudaFuncSetAttribute(k_encode<LEVEL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.t.nblocks);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_encode<LEVEL>, a);
}

}  // namespace dev

cudaError_t launch_encode(const EncodeArgs &a, cudaStream_t s)
{
    const uint32_t zero_ctas = 1 + a.t.nblocks / 8192;
    dev::k_encode_prologue<<<zero_ctas < 64 ? zero_ctas : 64, 256, 0, s>>>(a.x, a.t, a.median_exp, a.cb.hash);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.t.nblocks == 0) return err;
    switch (a.t.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
