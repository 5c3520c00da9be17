// Block offsets of a compressed tensor whose writer deferred them.
//
// [EXP] "Compressing is easy": the spilled exponents of every stream go to
// one uncompressed overflow region; blk_off[b], the exclusive prefix of the
// blocks' overflow byte counts (blk_off[nblocks] being the total), tells a
// reader where block b's bytes begin.  On grids of several waves the writers
// (encode, the fused updates) let a block with nothing to place publish its
// count and leave at once; only blocks with bytes to place wait in the
// look-back.  This kernel, launched after the writer as its programmatic
// dependent, then turns the counts every status word carries into the block
// offsets, the header's ovf_used and the capacity check.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kOffThreads = 1024;
constexpr int kOffPer = 8;  // status words per thread per pass (8192 blocks a pass)

// One CTA per tensor (the two-state update writes two).  Each pass gives every
// thread up to kOffPer consecutive status words, read together; their counts
// are summed, the sums scanned across the CTA, and each thread writes its
// words' offsets from its share of the scan.  One pass covers 8,192 blocks
// (536M values in CLEAN blocks); larger tensors take more passes, the total so
// far carried between them.
__global__ void __launch_bounds__(kOffThreads) k_block_offsets(DevTensor t0, DevTensor t1)
{
    const DevTensor &t = blockIdx.x == 0 ? t0 : t1;
    __shared__ unsigned long long warp_sum[kOffThreads / 32];
    __shared__ uint32_t s_missing;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_missing = 0;
    __syncthreads();
    pdl_wait();  // every block of the writer has published its count
    pdl_launch_dependents();
    const uint64_t nb = t.nblocks;
    unsigned long long carry = 0;
    for (uint64_t pass = 0; pass < nb; pass += (uint64_t)kOffThreads * kOffPer) {
        const uint64_t first = pass + (uint64_t)tid * kOffPer;
        unsigned long long own[kOffPer], sum = 0;
        bool missing = false;
#pragma unroll
        for (int k = 0; k < kOffPer; ++k) {
            own[k] = 0;
            if (first + k < nb) {
                const unsigned long long v = ld_status(&t.work[first + k]);
                missing |= (v >> 62) == 0;  // a block that published nothing
                own[k] = (v >> kOwnShift) & kOwnMask;
            }
            sum += own[k];
        }
        if (missing) s_missing = 1;
        unsigned long long inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long u = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane == 31) warp_sum[warp] = inc;
        __syncthreads();
        unsigned long long before = 0, total = 0;
        for (int w = 0; w < kOffThreads / 32; ++w) {
            const unsigned long long u = warp_sum[w];
            if (w < warp) before += u;
            total += u;
        }
        unsigned long long at = carry + before + inc - sum;
#pragma unroll
        for (int k = 0; k < kOffPer; ++k) {
            if (first + k < nb) t.blk_off[first + k] = at;
            at += own[k];
        }
        carry += total;
        __syncthreads();  // warp_sum is written again by the next pass
    }
    if (tid == 0) {
        t.blk_off[nb] = carry;
        t.hdr->ovf_used = carry;
        if (s_missing) latch(t.hdr, LCT_ERR_CORRUPT);
        if (carry > t.ovf_cap) latch(t.hdr, LCT_ERR_OVERFLOW_CAPACITY);
    }
}

}  // namespace dev

bool deferred_placement(uint32_t nblocks)
{
    int device = 0, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return false;
    return (uint64_t)nblocks >= 4ull * (uint64_t)sms;
}

bool small_grid(uint32_t nblocks)
{
    int device = 0, sms = 0;
    if (cudaGetDevice(&device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return false;
    return (uint64_t)nblocks <= 2ull * (uint64_t)sms;
}

cudaError_t launch_block_offsets(const DevTensor &t, cudaStream_t s)
{
    if (t.nblocks == 0) return cudaSuccess;
    return dev::launch_pdl(dev::k_block_offsets, dim3(1), dim3(dev::kOffThreads), 0, s, t, t);
}

cudaError_t launch_block_offsets2(const DevTensor &t0, const DevTensor &t1, cudaStream_t s)
{
    if (t0.nblocks == 0) return cudaSuccess;
    return dev::launch_pdl(dev::k_block_offsets, dim3(2), dim3(dev::kOffThreads), 0, s, t0, t1);
}

}  // namespace lct
