// Encode path of liblct: the scale-shift prologue and the block encoder.
//
// [EXP] "In bits": split every BF16 value into a sign-fraction byte (kept as
// is) and an exponent byte; code the exponent with the precomputed codebook,
// shifted to the tensor's scale from at most 4096 samples.
// [EXP] "Compressing is easy": blocks of 65,536 (CLEAN) or 32,768 values,
// 256 streams per block dealt round-robin, fixed-length slots, uncompressed
// overflow with a per-stream spill marker.
//
// Thread j of a block's CTA owns stream j.  The BF16 input streams through a
// ring of row chunks filled by TMA bulk copies; each row's values are split,
// their sign-fraction bytes written straight out, and their exponents
// appended to the streams' slot images in shared memory.  A chunk in which
// every stream of a warp has room for all of its codes takes a fast path
// with no per-value fit checks.  Spilled exponents are kept in a 32-row ring; a stream
// that spills more than that has its older spilled exponents read back from
// the input.
#include "codec_dev.cuh"

namespace lct {
namespace dev {

constexpr int kEncThreads = 256;
constexpr int kEncRows = 16;       // rows per input chunk (4 CTAs per SM)
constexpr int kEncRowsSmall = 32;  // rows per input chunk on grids of at most two blocks per SM
constexpr int kEncRing = 2;        // chunks in flight
constexpr int kSpillRows = 32;     // spilled-exponent rows kept

template <int LEVEL, int ROWS>
struct EncodeSmem {
    static constexpr int W = Geo<LEVEL>::W;
    static constexpr int kIn = kEncRing * ROWS * kStreams * 2;
    static constexpr int kSlot = W * kStreams * 4;
    static constexpr int kTbl = 256 * 8;
    static constexpr int kSpill = (kSpillRows * kRow + 127) / 128 * 128;
    static constexpr int kBytes = kIn + kSlot + kTbl + kSpill;
};

// Prologue (one launch per encode, clusters of kSampleCtas CTAs): the first
// cluster estimates the shift and CTA 0 writes the tensor header; every CTA
// zeroes its share of the look-back status words.  The samples are spread
// over the cluster's CTAs (one SM keeps only so many loads in flight) and
// their counts are added up through distributed shared memory.
constexpr int kSampleCtas = 8;

__global__ void __launch_bounds__(256) k_encode_prologue(const uint16_t *__restrict__ x, DevTensor t,
                                                          int32_t median_exp, uint32_t cb_hash)
{
    pdl_wait();               // earlier work in the stream (e.g. what produced x) is done
    pdl_launch_dependents();  // the block encoder may start its input loads now
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < t.nblocks;
         i += (uint64_t)gridDim.x * blockDim.x)
        t.work[i] = 0ull;
    if (blockIdx.x >= kSampleCtas) return;  // not the first cluster

    // Shift: m = min(n, 4096) samples at floor(k*n/m); histogram of their
    // exponents in the normal range 1..254; lower median.  CTA r of the
    // cluster takes k = tid + 256*i for i in [r*kPer, (r+1)*kPer).
    constexpr int kPer = LCT_SHIFT_SAMPLES / 256 / kSampleCtas;
    static_assert(kPer * 256 * kSampleCtas == LCT_SHIFT_SAMPLES, "samples split evenly");
    __shared__ uint32_t hist[8][256];  // one histogram per warp
    __shared__ uint32_t cta_hist[256];
    __shared__ uint32_t wsum[8];
    __shared__ int32_t median;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank();
#pragma unroll
    for (int w = 0; w < 8; ++w) hist[w][tid] = 0;
    if (tid == 0) median = -1;
    __syncthreads();
    const uint64_t n = t.n;
    const uint32_t m = n < (uint64_t)LCT_SHIFT_SAMPLES ? (uint32_t)n : (uint32_t)LCT_SHIFT_SAMPLES;
    // floor(k*n/m): with m = 4096 = 2^12 a shift, with m = n just k
    static_assert(LCT_SHIFT_SAMPLES == 4096, "sample positions use a shift by 12");
    uint16_t v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {  // all loads in flight at once
        const uint32_t k = tid + 256u * (rank * kPer + i);
        const uint64_t at = m == (uint32_t)LCT_SHIFT_SAMPLES ? ((uint64_t)k * n) >> 12 : (uint64_t)k;
        v[i] = k < m ? __ldg(x + at) : 0;
    }
    // Samples concentrate on a few exponents: lanes holding the same one are
    // counted together by one lane, into the warp's own histogram.
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const uint32_t e = exp_of(v[i]);
        const bool keep = tid + 256u * (rank * kPer + i) < m && e >= 1 && e <= 254;
        const uint32_t same = __match_any_sync(kFull, keep ? e : 256u);
        if (keep && lane == __ffs(same) - 1) hist[warp][e] += __popc(same);
    }
    __syncthreads();
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += hist[w][tid];
    cta_hist[tid] = c;
    cluster_sync();  // every CTA's counts are in its shared memory
    if (rank == 0) {
        c = 0;
        for (uint32_t q = 0; q < (uint32_t)kSampleCtas; ++q) c += ld_peer_shared(&cta_hist[tid], q);
        uint32_t inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane == 31) wsum[warp] = inc;
        __syncthreads();
        uint32_t before = 0, kept = 0;
        for (int w = 0; w < 8; ++w) {
            if (w < warp) before += wsum[w];
            kept += wsum[w];
        }
        inc += before;
        if (kept > 0) {
            const uint32_t r = (kept - 1) / 2;  // lower median, 0-based
            if (inc > r && inc - c <= r) median = tid;
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
    cluster_sync();  // CTA 0 has read the other CTAs' counts
}

// ROWS rows of every stream per input chunk.  A grid of at most two blocks per
// SM has no third or fourth CTA on an SM to hide the per-chunk barrier, so it
// takes chunks twice as long (half the barriers, twice the loads in flight per
// thread, 2 CTAs per SM by registers).
template <int LEVEL, int ROWS>
__global__ void __launch_bounds__(kEncThreads, ROWS == kEncRows ? 4 : 2) k_encode(const __grid_constant__ EncodeArgs a)
{
    using G = Geo<LEVEL>;
    using L = EncodeSmem<LEVEL, ROWS>;
    constexpr int W = G::W, R = ROWS, S = kEncRing, SP = kSpillRows;
    constexpr int NW = kEncThreads / 32;
    extern __shared__ __align__(128) uint8_t smem[];
    uint16_t *x_s = reinterpret_cast<uint16_t *>(smem);
    uint32_t *slot_s = reinterpret_cast<uint32_t *>(smem + L::kIn);
    uint2 *tbl = reinterpret_cast<uint2 *>(smem + L::kIn + L::kSlot);
    uint8_t *ring = smem + L::kIn + L::kSlot + L::kTbl;
    __shared__ __align__(8) uint64_t bar[S];
    __shared__ uint32_t warp_tot[NW];
    __shared__ unsigned long long s_excl;
    __shared__ uint32_t s_timeout;

    const int j = threadIdx.x, lane = j & 31, warp = j >> 5;
    const uint32_t b = blockIdx.x;
    const uint64_t base = (uint64_t)b * G::B;
    const uint32_t nb = (uint32_t)min((uint64_t)G::B, a.t.n - base);
    const uint32_t nrows = (nb + 255) >> 8, nbulk = (nb >> 8) / R, nchunks = (nrows + R - 1) / R;
    const uint64_t limit = a.wait_ns;

    if (j == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
        s_timeout = 0;
        // The input was written before the prologue ran, so it can be read
        // before waiting for the prologue.
        for (uint32_t c = 0; c < (uint32_t)S && c < nbulk; ++c) {
            mbar_expect_tx(&bar[c], R * kStreams * 2);
            bulk_load(x_s + c * R * kStreams, a.x + base + (uint64_t)c * R * kStreams, R * kStreams * 2, &bar[c]);
        }
    }
    // the shift and the cleared look-back words come from the prologue
    pdl_wait();
    tbl[j] = enc_entry(a.cb, a.t.hdr->delta, j);
    __syncthreads();

    const uint32_t nj = nb > (uint32_t)j ? (nb - j + 255) / 256 : 0;
    Writer wr;
    wr_init<W>(wr, nj);
    uint32_t *col = slot_s + j;
    uint8_t *sfj = a.t.sf + base + j;
    uint8_t *ringj = ring + j;

    for (uint32_t c = 0; c < nchunks; ++c) {
        const bool bulk = c < nbulk;
        const uint32_t slot = c % S;
        if (bulk && !mbar_wait(&bar[slot], (c / S) & 1u, s_timeout ? 1000000ull : limit)) s_timeout = 1;
        const uint16_t *xc = x_s + slot * R * kStreams + j;
        uint8_t *sfc = sfj + (uint64_t)c * R * kStreams;
        if (bulk) {
            // loads first (inputs, then their code-table entries), stores
            // last, so nothing orders a load behind a store
            uint32_t h[R], need = 0;
            uint2 ent[R];
#pragma unroll
            for (int r = 0; r < R; ++r) h[r] = xc[r * kStreams];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ent[r] = code_of(tbl, h[r]);
                need += ent[r].y;
            }
#pragma unroll
            for (int r = 0; r < R; ++r) sfc[r * kStreams] = sf_of(h[r]);
            if (__all_sync(kFull, wr.alive && need <= wr.rem)) {
                // every stream of the warp keeps the whole chunk in its slot
#pragma unroll
                for (int r = 0; r < R; r += 2) {  // two codes fit the accumulator, then one flush
                    wr_add2(wr, ent[r], ent[r + 1]);
                    wr_flush(wr, col);
                }
                wr.rem -= need;
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const uint32_t k = c * R + r;
                    if (wr_put_checked(wr, ent[r], k, col)) ringj[(k & (SP - 1)) * kRow] = (uint8_t)exp_of(h[r]);
                }
            }
        } else {
            for (int r = 0; r < R; ++r) {
                const uint32_t k = c * R + r;
                if (k >= nj) break;
                const uint32_t h = a.x[base + (uint64_t)k * kStreams + j];
                const uint32_t e = exp_of(h);
                sfc[r * kStreams] = sf_of(h);
                if (wr_put_checked(wr, tbl[e], k, col)) ringj[(k & (SP - 1)) * kRow] = (uint8_t)e;
            }
        }
        __syncthreads();  // every thread is done with this chunk's ring slot
        if (j == 0 && c + S < nbulk) {
            mbar_expect_tx(&bar[slot], R * kStreams * 2);
            bulk_load(x_s + slot * R * kStreams, a.x + base + (uint64_t)(c + S) * R * kStreams, R * kStreams * 2,
                      &bar[slot]);
        }
    }
    wr_finish<W>(wr, col);
    const uint32_t marker = wr.marker, spill = nj - marker;
    uint32_t total;
    const uint32_t pre = group_exclusive_scan(spill, warp_tot, NW, 0, &total);  // syncs: slot image complete

    if (j == 0) {
        fence_proxy_async();
        bulk_store(a.t.slots + (uint64_t)b * W * kStreams, slot_s, W * kStreams * 4);
        bulk_commit();
    }
    a.t.markers[(uint64_t)b * kStreams + j] = (uint16_t)marker;

    // Overflow offset of this block: the single-pass decoupled look-back, or,
    // with deferred placement, a count published without waiting when the
    // block has nothing to place (k_block_offsets writes the offsets after).
    const bool leave = a.deferred && total == 0 && !lookback_leader(b);
    if (warp == 0) {
        if (leave) {
            warp_publish_try(a.t.work, b, 2);
        } else {
            bool timed_out;
            const unsigned long long excl = warp_lookback(a.t.work, b, total, limit, &timed_out);
            if (lane == 0) {
                if (timed_out) latch(a.t.hdr, LCT_ERR_TIMEOUT);
                if (!a.deferred) {
                    a.t.blk_off[b] = excl;
                    if (b == a.t.nblocks - 1) {
                        a.t.blk_off[b + 1] = excl + total;
                        a.t.hdr->ovf_used = excl + total;
                    }
                    if (excl + total > a.t.ovf_cap) latch(a.t.hdr, LCT_ERR_OVERFLOW_CAPACITY);
                }
                s_excl = excl;
            }
        }
    }
    if (!leave) __syncthreads();  // uniform: total is the block's
    const unsigned long long excl = leave ? 0ull : s_excl;

    // spilled exponents, raw, in (stream, symbol) order: a few per stream
    // lane by lane, otherwise one warp per stream at a time with the lanes
    // over the stream's spilled symbols (beyond the capacity nothing is
    // written; the capacity error is latched)
    if (total > 0 && excl + total <= a.t.ovf_cap && __reduce_max_sync(kFull, spill) <= kFewSpills) {
        uint8_t *out = a.t.ovf + excl + pre;
        const uint32_t kept_from = nj > (uint32_t)SP ? nj - SP : 0u;  // older spills were overwritten
        for (uint32_t l = 0; l < spill; ++l) {
            const uint32_t k = marker + l;
            out[l] = k >= kept_from ? ringj[(k & (SP - 1)) * kRow] : exp_of(a.x[base + (uint64_t)k * kStreams + j]);
        }
    } else if (total > 0 && excl + total <= a.t.ovf_cap) {
        uint8_t *out = a.t.ovf + excl;
        for (int i = 0; i < 32; ++i) {
            const uint32_t sm = __shfl_sync(kFull, marker, i);
            const uint32_t sp = __shfl_sync(kFull, spill, i);
            const uint32_t so = __shfl_sync(kFull, pre, i);
            const uint32_t sj = (uint32_t)(warp * 32 + i);
            const uint32_t nj_i = sm + sp;
            const uint32_t kept_from = nj_i > (uint32_t)SP ? nj_i - SP : 0u;  // older spills were overwritten
            for (uint32_t l = lane; l < sp; l += 32) {
                const uint32_t k = sm + l;
                out[so + l] = k >= kept_from ? ring[(k & (SP - 1)) * kRow + sj]
                                             : exp_of(a.x[base + (uint64_t)k * kStreams + sj]);
            }
        }
    }
    pdl_launch_dependents();
    if (j == 0) {
        if (s_timeout) {
            latch(a.t.hdr, LCT_ERR_TIMEOUT);
            for (uint32_t s = 0; s < (uint32_t)S && s < nbulk; ++s) {
                const uint32_t last = s + (nbulk - 1 - s) / S * S;
                mbar_wait(&bar[s], (last / S) & 1u, limit);
            }
        }
        bulk_wait_all();  // the slot image store has read shared memory
    }
}

template <int LEVEL, int ROWS>
cudaError_t launch_kernel(const EncodeArgs &a, cudaStream_t s)
{
    constexpr int smem = EncodeSmem<LEVEL, ROWS>::kBytes;
    cudaError_t err = cudaFuncSetAttribute(k_encode<LEVEL, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    EncodeArgs b = a;
    b.deferred = deferred_placement(a.t.nblocks);
    err = launch_pdl(k_encode<LEVEL, ROWS>, dim3(a.t.nblocks), dim3(kEncThreads), smem, s, b);
    if (err != cudaSuccess || !b.deferred) return err;
    return launch_block_offsets(a.t, s);
}

template <int LEVEL>
cudaError_t launch_level(const EncodeArgs &a, cudaStream_t s)
{
    return small_grid(a.t.nblocks) ? launch_kernel<LEVEL, kEncRowsSmall>(a, s) : launch_kernel<LEVEL, kEncRows>(a, s);
}

}  // namespace dev

cudaError_t launch_encode(const EncodeArgs &a, cudaStream_t s)
{
    // one CTA per 8192 look-back words (at most 64), in whole clusters
    const uint64_t zero_ctas = 1 + a.t.nblocks / 8192;
    const uint32_t k = dev::kSampleCtas, ctas = (uint32_t)((zero_ctas < 64 ? zero_ctas : 64) + k - 1) / k * k;
    cudaError_t err = dev::launch_pdl_cluster(dev::k_encode_prologue, dim3(ctas), dim3(256), 0, s, k, a.x, a.t,
                                              a.median_exp, a.cb.hash);
    if (err != cudaSuccess || a.t.nblocks == 0) return err;
    switch (a.t.level) {
    case LCT_LEVEL_CLEAN: return dev::launch_level<LCT_LEVEL_CLEAN>(a, s);
    case LCT_LEVEL_MEDIUM: return dev::launch_level<LCT_LEVEL_MEDIUM>(a, s);
    default: return dev::launch_level<LCT_LEVEL_HIGH>(a, s);
    }
}

}  // namespace lct
