// Decode path of liblct: one CTA per block rebuilds the block's BF16 values.
//
// [EXP] "In bits": every value decodes exactly -- the sign-fraction byte is
// copied back and the exponent comes from its code (or the escape literal).
// [EXP] "Compressing is easy": each of the 256 streams decodes independently
// from its fixed-length slot up to its spill marker, then takes its spilled
// exponents from the uncompressed overflow region.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

template <int LEVEL>
__global__ void __launch_bounds__(256, 2) k_decode(const __grid_constant__ DecodeArgs a)
{
    using G = Geo<LEVEL>;
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *e_s = smem;
    uint32_t *slot_s = reinterpret_cast<uint32_t *>(smem + Smem<LEVEL>::kExpBytes);
    uint32_t *lut = reinterpret_cast<uint32_t *>(smem + Smem<LEVEL>::kExpBytes + Smem<LEVEL>::kSlotBytes);
    __shared__ uint32_t warp_tot[8];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.t.n - base);
    lct_header *hdr = a.t.hdr;

    // The header must describe this tensor and this codebook.
    const bool hdr_ok = hdr->magic == LCT_MAGIC && hdr->n == a.t.n && hdr->level == LEVEL &&
                        hdr->cb_hash == a.cb.hash;
    if (!hdr_ok) {
        if (tid == 0) latch(hdr, LCT_ERR_CORRUPT);
        return;
    }
    const int delta = hdr->delta;
    lut[tid] = dec_entry(a.cb, delta, tid);

    // slot image of this block plus one zero guard row
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.t.slots + (uint64_t)b * G::W * kStreams);
        uint4 *dst = reinterpret_cast<uint4 *>(slot_s);
#pragma unroll 5
        for (int w = tid; w < G::W * kStreams / 4; w += 256) dst[w] = __ldcs(src + w);
        slot_s[G::W * kStreams + tid] = 0u;
    }
    const uint32_t j = tid;
    const uint32_t nj = nb > j ? (nb - j + 255) / 256 : 0;
    uint32_t marker = a.t.markers[(uint64_t)b * kStreams + j];
    bool bad = marker > nj;
    marker = min(marker, nj);
    const uint32_t spill = nj - marker;
    uint32_t total;
    const uint32_t pre = group_exclusive_scan(spill, warp_tot, 8, 0, &total);  // syncs

    const uint64_t off0 = a.t.blk_off[b], off1 = a.t.blk_off[b + 1];
    const bool ovf_ok = off1 <= a.t.ovf_cap && off0 <= off1 && off1 - off0 == total;

    const uint32_t bits = decode_stream<G::W>(slot_s + j, marker, lut, e_s + j);
    bad |= bits > 32u * G::W;
    if (bad) latch(hdr, LCT_ERR_CORRUPT);
    if (tid == 0 && !ovf_ok)
        latch(hdr, off1 > a.t.ovf_cap && off0 <= off1 ? LCT_ERR_OVERFLOW_CAPACITY : LCT_ERR_CORRUPT);

    // spilled exponents: one warp per stream at a time
    if (total > 0 && ovf_ok) {
        const uint8_t *in = a.t.ovf + off0;
        for (int i = 0; i < 32; ++i) {
            const uint32_t sm = __shfl_sync(0xFFFFFFFFu, marker, i);
            const uint32_t sp = __shfl_sync(0xFFFFFFFFu, spill, i);
            const uint32_t so = __shfl_sync(0xFFFFFFFFu, pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            for (uint32_t l = lane; l < sp; l += 32) e_s[(sm + l) * kRow + sj] = __ldg(in + so + l);
        }
    }
    __syncthreads();

    // reassemble: sign-fraction bytes + exponents -> BF16, 8 values per step
    const uint2 *sfv = reinterpret_cast<const uint2 *>(a.t.sf + base);
    uint4 *yv = reinterpret_cast<uint4 *>(a.y + base);
    const uint32_t ng = nb >> 3;
#pragma unroll 4
    for (uint32_t g = tid; g < ng; g += 256) {
        const uint2 sf = __ldcs(sfv + g);
        const uint32_t *ep = reinterpret_cast<const uint32_t *>(stage_at(e_s, g << 3));
        __stcs(yv + g, join8(sf, make_uint2(ep[0], ep[1])));
    }
    for (uint32_t i = (ng << 3) + tid; i < nb; i += 256) a.y[base + i] = join1(a.t.sf[base + i], *stage_at(e_s, i));
}

template <int LEVEL>
cudaError_t launch_level(const DecodeArgs &a, cudaStream_t s)
{
    constexpr int smem = Smem<LEVEL>::kExpBytes + Smem<LEVEL>::kSlotBytes + 256 * 4;
    cudaError_t err = cudaFuncSetAttribute(k_decode<LEVEL>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    k_decode<LEVEL><<<a.t.nblocks, 256, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace dev

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t s)
{
    if (a.t.nblocks == 0) return cudaSuccess;
    switch (a.t.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
