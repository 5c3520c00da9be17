// Host entry points of liblct (the C ABI declared in include/lct.h):
// argument checks, sizing, and kernel launches.  No device memory is ever
// allocated here; every buffer belongs to the caller.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/lct.h"
#include "../../include/lct_debug.h"
#include "codec_dev.cuh"
#include "internal.h"

namespace lct {
namespace {

uint64_t nblocks_for(uint64_t n, const Geometry &g) { return (n + g.block - 1) / g.block; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
Range range_of(const void *p, uint64_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

void fill_sizes(uint64_t n, const Geometry &g, lct_sizes *s)
{
    std::memset(s, 0, sizeof(*s));
    const uint64_t nb = nblocks_for(n, g);
    s->n = n;
    s->nblocks = nb;
    s->block = g.block;
    s->slot_words = g.slot_words;
    s->header_bytes = LCT_HEADER_BYTES;
    s->sf_bytes = n;
    s->slot_bytes = nb * g.slot_words * kStreams * 4ull;
    s->marker_bytes = nb * kStreams * 2ull;
    s->blk_off_bytes = (nb + 1) * 8ull;
    s->fixed_bytes = s->header_bytes + s->sf_bytes + s->slot_bytes + s->marker_bytes + s->blk_off_bytes;
    s->worst_ovf_bytes = n;
    s->work_bytes = nb * 8ull;
}

// Host-side checks of one tensor descriptor; fills its sizes.
lct_status check_tensor(const lct_tensor *t, bool writer, lct_sizes *s)
{
    Geometry g;
    if (!t || t->n > kMaxN || !level_geometry(t->level, &g)) return LCT_ERR_INVALID_ARG;
    fill_sizes(t->n, g, s);
    if (!t->d_header || !aligned16(t->d_header)) return LCT_ERR_INVALID_ARG;
    if (t->n > 0) {
        if (!t->d_sf || !t->d_slots || !t->d_markers || !t->d_blk_off) return LCT_ERR_INVALID_ARG;
        if (!aligned16(t->d_sf) || !aligned16(t->d_slots) || !aligned16(t->d_markers) ||
            !aligned16(t->d_blk_off))
            return LCT_ERR_INVALID_ARG;
        if (writer && (!t->d_work || !aligned16(t->d_work))) return LCT_ERR_INVALID_ARG;
    }
    if (t->ovf_cap > 0 && !t->d_ovf) return LCT_ERR_INVALID_ARG;
    if (t->d_ovf && !aligned16(t->d_ovf)) return LCT_ERR_INVALID_ARG;
    if (writer && t->n > 0) {
        // the regions a writer fills must not overlap one another
        const void *p[7] = {t->d_header, t->d_sf, t->d_slots, t->d_markers, t->d_blk_off, t->d_ovf, t->d_work};
        const uint64_t len[7] = {s->header_bytes, s->sf_bytes, s->slot_bytes, s->marker_bytes,
                                 s->blk_off_bytes, t->ovf_cap, s->work_bytes};
        for (int i = 0; i < 7; ++i)
            for (int k = i + 1; k < 7; ++k)
                if (p[i] && p[k] && overlap(range_of(p[i], len[i]), range_of(p[k], len[k])))
                    return LCT_ERR_INVALID_ARG;
    }
    return LCT_OK;
}

DevTensor dev_view(const lct_tensor *t, const lct_sizes &s)
{
    DevTensor d;
    d.hdr = static_cast<lct_header *>(t->d_header);
    d.sf = t->d_sf;
    d.slots = t->d_slots;
    d.markers = t->d_markers;
    d.blk_off = t->d_blk_off;
    d.ovf = t->d_ovf;
    d.work = static_cast<unsigned long long *>(t->d_work);
    d.ovf_cap = t->ovf_cap;
    d.n = t->n;
    d.nblocks = static_cast<uint32_t>(s.nblocks);
    d.level = t->level;
    return d;
}

DevCodebook dev_codebook(const lct_codebook &cb)
{
    DevCodebook d;
    std::memcpy(d.len, cb.len, 256);
    std::memcpy(d.code, cb.code, 256);
    std::memcpy(d.dec, cb.dec, sizeof(d.dec));
    d.esc_len = cb.esc_len;
    d.esc_code = cb.esc_code;
    d.zero_atom = static_cast<uint8_t>(cb.zero_atom);
    d.pad = 0;
    d.hash = cb.hash;
    return d;
}

// Every region of a tensor, for overlap checks.
void regions(const lct_tensor *t, const lct_sizes &s, Range out[7])
{
    out[0] = range_of(t->d_header, s.header_bytes);
    out[1] = range_of(t->d_sf, s.sf_bytes);
    out[2] = range_of(t->d_slots, s.slot_bytes);
    out[3] = range_of(t->d_markers, s.marker_bytes);
    out[4] = range_of(t->d_blk_off, s.blk_off_bytes);
    out[5] = range_of(t->d_ovf, t->ovf_cap);
    out[6] = range_of(t->d_work, s.work_bytes);
}

// Aliasing rules of a fused update with nout outputs and nin >= nout inputs,
// output o being the new value of input o (inputs nout.. are read only):
//   - an output may share its header, sign-fraction, slot, marker and offset
//     regions with its own input (in place) but not partly overlap them, and
//     its overflow and scratch are apart from every region of that input;
//   - an output does not touch another input, another output or the dense
//     gradient (grad may be null).
bool aliasing_ok(const Range (*out)[7], int nout, const Range (*in)[7], int nin, const Range *grad)
{
    for (int o = 0; o < nout; ++o) {
        for (int r = 0; r < 7; ++r)
            if (grad && overlap(out[o][r], *grad)) return false;
        for (int i = 0; i < nin; ++i) {
            if (i == o) continue;
            for (int r = 0; r < 7; ++r)
                for (int k = 0; k < 6; ++k)
                    if (overlap(out[o][r], in[i][k])) return false;
        }
        for (int q = 0; q < nout; ++q) {
            if (q == o) continue;
            for (int r = 0; r < 7; ++r)
                for (int k = 0; k < 7; ++k)
                    if (overlap(out[o][r], out[q][k])) return false;
        }
        for (int k = 0; k < 6; ++k)
            if (overlap(out[o][5], in[o][k]) || overlap(out[o][6], in[o][k])) return false;
        for (int r = 0; r < 5; ++r)
            for (int k = 0; k < 6; ++k) {
                const bool same = r == k && out[o][r].lo == in[o][k].lo;
                if (!same && overlap(out[o][r], in[o][k])) return false;
            }
    }
    return true;
}

}  // namespace
}  // namespace lct

using namespace lct;

extern "C" lct_status lct_compressed_size(uint64_t n, int level, const lct_tensor *t, void *stream,
                                          lct_sizes *out)
{
    Geometry g;
    if (!out || n > kMaxN || !level_geometry(level, &g)) return LCT_ERR_INVALID_ARG;
    if (t && (t->n != n || t->level != level)) return LCT_ERR_INVALID_ARG;
    lct_sizes s;
    fill_sizes(n, g, &s);
    if (t) {
        if (!t->d_header || !aligned16(t->d_header)) return LCT_ERR_INVALID_ARG;
        lct_header h;
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if (cudaMemcpyAsync(&h, t->d_header, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
            return LCT_ERR_CUDA;
        if (cudaStreamSynchronize(st) != cudaSuccess) return LCT_ERR_CUDA;
        s.ovf_used = h.ovf_used;
        s.status = h.status;
        s.delta = h.delta;
        if (h.magic != LCT_MAGIC && s.status == 0) s.status = LCT_ERR_CORRUPT;
    }
    *out = s;
    return LCT_OK;
}

extern "C" lct_status lct_encode(const uint16_t *d_x, const lct_codebook *cb, const lct_tensor *t,
                                 void *stream)
{
    lct_sizes s;
    lct_status rc = check_tensor(t, true, &s);
    if (rc != LCT_OK) return rc;
    if (!cb || !codebook_valid(*cb)) return LCT_ERR_INVALID_ARG;
    if (t->n > 0 && (!d_x || !aligned16(d_x))) return LCT_ERR_INVALID_ARG;
    Range r[7];
    regions(t, s, r);
    for (int i = 0; i < 7; ++i)
        if (t->n > 0 && overlap(r[i], range_of(d_x, 2 * t->n))) return LCT_ERR_INVALID_ARG;
    EncodeArgs a;
    a.x = d_x;
    a.t = dev_view(t, s);
    a.cb = dev_codebook(*cb);
    a.median_exp = cb->median_exp;
    a.pad = 0;
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    return launch_encode(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LCT_OK : LCT_ERR_CUDA;
}

extern "C" lct_status lct_decode(const lct_tensor *t, const lct_codebook *cb, uint16_t *d_y, void *stream)
{
    lct_sizes s;
    lct_status rc = check_tensor(t, false, &s);
    if (rc != LCT_OK) return rc;
    if (!cb || !codebook_valid(*cb)) return LCT_ERR_INVALID_ARG;
    if (t->n > 0 && (!d_y || !aligned16(d_y))) return LCT_ERR_INVALID_ARG;
    Range r[7];
    regions(t, s, r);
    for (int i = 0; i < 6; ++i)
        if (t->n > 0 && overlap(r[i], range_of(d_y, 2 * t->n))) return LCT_ERR_INVALID_ARG;
    DecodeArgs a;
    a.t = dev_view(t, s);
    a.y = d_y;
    a.cb = dev_codebook(*cb);
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    a.first_block = 0;
    a.pad = 0;
    return launch_decode(a, a.t.nblocks, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LCT_OK : LCT_ERR_CUDA;
}

extern "C" lct_status lct_decode_blocks(const lct_tensor *t, const lct_codebook *cb, uint64_t first_block,
                                        uint64_t nblocks, uint16_t *d_y, void *stream)
{
    lct_sizes s;
    lct_status rc = check_tensor(t, false, &s);
    if (rc != LCT_OK) return rc;
    if (!cb || !codebook_valid(*cb)) return LCT_ERR_INVALID_ARG;
    if (first_block > s.nblocks || nblocks > s.nblocks - first_block) return LCT_ERR_INVALID_ARG;
    if (nblocks == 0) return LCT_OK;
    const uint64_t lo = first_block * s.block;
    const uint64_t hi = std::min<uint64_t>(t->n, (first_block + nblocks) * s.block);
    if (!d_y || !aligned16(d_y)) return LCT_ERR_INVALID_ARG;
    Range r[7];
    regions(t, s, r);
    for (int i = 0; i < 6; ++i)
        if (overlap(r[i], range_of(d_y, 2 * (hi - lo)))) return LCT_ERR_INVALID_ARG;
    DecodeArgs a;
    a.t = dev_view(t, s);
    a.y = d_y;
    a.cb = dev_codebook(*cb);
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    a.first_block = static_cast<uint32_t>(first_block);
    a.pad = 0;
    return launch_decode(a, static_cast<uint32_t>(nblocks), static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? LCT_OK
               : LCT_ERR_CUDA;
}

extern "C" lct_status lct_sgd_step_fused(const lct_tensor *W_in, const lct_codebook *cbW, const lct_tensor *M,
                                         const lct_codebook *cbM, float eta, const lct_tensor *W_out,
                                         void *stream)
{
    lct_sizes sw, sm, so;
    lct_status rc;
    if ((rc = check_tensor(W_in, false, &sw)) != LCT_OK) return rc;
    if ((rc = check_tensor(M, false, &sm)) != LCT_OK) return rc;
    if ((rc = check_tensor(W_out, true, &so)) != LCT_OK) return rc;
    if (!cbW || !cbM || !codebook_valid(*cbW) || !codebook_valid(*cbM)) return LCT_ERR_INVALID_ARG;
    if (W_in->n != M->n || W_in->n != W_out->n) return LCT_ERR_INVALID_ARG;
    if (W_in->level != M->level || W_in->level != W_out->level) return LCT_ERR_UNSUPPORTED;
    Range ri[2][7], ro[1][7];
    regions(W_in, sw, ri[0]);
    regions(M, sm, ri[1]);
    regions(W_out, so, ro[0]);
    if (W_out->n > 0 && !aliasing_ok(ro, 1, ri, 2, nullptr)) return LCT_ERR_INVALID_ARG;
    UpdateArgs a;
    std::memset(&a, 0, sizeof(a));
    a.in[0] = dev_view(W_in, sw);
    a.in[1] = dev_view(M, sm);
    a.w_out = dev_view(W_out, so);
    a.cb[0] = dev_codebook(*cbW);
    a.cb[1] = dev_codebook(*cbM);
    a.k[0] = eta;
    a.op = OP_SGD;
    a.nin = 2;
    a.in_place = W_out->d_sf == W_in->d_sf ? 1u : 0u;
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    return launch_update(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LCT_OK : LCT_ERR_CUDA;
}

extern "C" lct_status lct_sgd_momentum_step_fused(const lct_tensor *W_in, const lct_codebook *cbW,
                                                  const lct_tensor *M_in, const lct_codebook *cbM,
                                                  const uint16_t *d_g, float eta, float mu, const lct_tensor *W_out,
                                                  const lct_tensor *M_out, void *stream)
{
    lct_sizes sw, sm, sow, som;
    lct_status rc;
    if ((rc = check_tensor(W_in, false, &sw)) != LCT_OK) return rc;
    if ((rc = check_tensor(M_in, false, &sm)) != LCT_OK) return rc;
    if ((rc = check_tensor(W_out, true, &sow)) != LCT_OK) return rc;
    if ((rc = check_tensor(M_out, true, &som)) != LCT_OK) return rc;
    if (!cbW || !cbM || !codebook_valid(*cbW) || !codebook_valid(*cbM)) return LCT_ERR_INVALID_ARG;
    const uint64_t n = W_in->n;
    if (M_in->n != n || W_out->n != n || M_out->n != n) return LCT_ERR_INVALID_ARG;
    if (M_in->level != W_in->level || W_out->level != W_in->level || M_out->level != W_in->level)
        return LCT_ERR_UNSUPPORTED;
    if (n > 0 && (!d_g || !aligned16(d_g))) return LCT_ERR_INVALID_ARG;
    Range ri[2][7], ro[2][7];
    regions(W_in, sw, ri[0]);
    regions(M_in, sm, ri[1]);
    regions(W_out, sow, ro[0]);
    regions(M_out, som, ro[1]);
    if (n > 0) {
        const Range rg = range_of(d_g, 2 * n);
        if (!aliasing_ok(ro, 2, ri, 2, &rg)) return LCT_ERR_INVALID_ARG;
    }
    MomentumArgs a;
    a.w_in = dev_view(W_in, sw);
    a.m_in = dev_view(M_in, sm);
    a.w_out = dev_view(W_out, sow);
    a.m_out = dev_view(M_out, som);
    a.g = d_g;
    a.cbw = dev_codebook(*cbW);
    a.cbm = dev_codebook(*cbM);
    std::memset(a.k, 0, sizeof(a.k));
    a.k[0] = eta;
    a.k[1] = mu;
    a.op = OP2_MOMENTUM;
    a.in_place = (W_out->d_sf == W_in->d_sf || M_out->d_sf == M_in->d_sf) ? 1u : 0u;
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    return launch_momentum(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LCT_OK : LCT_ERR_CUDA;
}

extern "C" lct_status lct_adamw_step_fused(const lct_tensor *W_in, const lct_codebook *cbW, const lct_tensor *M_in,
                                           const lct_codebook *cbM, const lct_tensor *V_in, const lct_codebook *cbV,
                                           const uint16_t *d_g, const lct_adamw_params *p, const lct_tensor *W_out,
                                           const lct_tensor *M_out, const lct_tensor *V_out, void *stream)
{
    const lct_tensor *ins[3] = {W_in, M_in, V_in}, *outs[3] = {W_out, M_out, V_out};
    const lct_codebook *cbs[3] = {cbW, cbM, cbV};
    lct_sizes si[3], so[3];
    lct_status rc;
    for (int i = 0; i < 3; ++i) {
        if ((rc = check_tensor(ins[i], false, &si[i])) != LCT_OK) return rc;
        if ((rc = check_tensor(outs[i], true, &so[i])) != LCT_OK) return rc;
        if (!cbs[i] || !codebook_valid(*cbs[i])) return LCT_ERR_INVALID_ARG;
    }
    if (!p || !(p->step >= 1) || !(p->beta1 >= 0.0 && p->beta1 < 1.0) || !(p->beta2 >= 0.0 && p->beta2 < 1.0) ||
        !(p->eps > 0.0) || !std::isfinite(p->lr) || !std::isfinite(p->weight_decay) || !std::isfinite(p->eps))
        return LCT_ERR_INVALID_ARG;
    const uint64_t n = W_in->n;
    for (int i = 0; i < 3; ++i) {
        if (ins[i]->n != n || outs[i]->n != n) return LCT_ERR_INVALID_ARG;
        if (ins[i]->level != W_in->level || outs[i]->level != W_in->level) return LCT_ERR_UNSUPPORTED;
    }
    if (n > 0 && (!d_g || !aligned16(d_g))) return LCT_ERR_INVALID_ARG;
    Range ri[3][7], ro[3][7];
    for (int i = 0; i < 3; ++i) {
        regions(ins[i], si[i], ri[i]);
        regions(outs[i], so[i], ro[i]);
    }
    if (n > 0) {
        const Range rg = range_of(d_g, 2 * n);
        if (!aliasing_ok(ro, 3, ri, 3, &rg)) return LCT_ERR_INVALID_ARG;
    }
    // the step's constants, rounded to float once
    const double t = static_cast<double>(p->step);
    float k[8];
    k[0] = static_cast<float>(p->beta1);
    k[1] = static_cast<float>(1.0 - p->beta1);
    k[2] = static_cast<float>(p->beta2);
    k[3] = static_cast<float>(1.0 - p->beta2);
    k[4] = static_cast<float>(p->lr / (1.0 - std::pow(p->beta1, t)));
    k[5] = static_cast<float>(1.0 / std::sqrt(1.0 - std::pow(p->beta2, t)));
    k[6] = static_cast<float>(p->eps);
    k[7] = static_cast<float>(p->lr * p->weight_decay);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // pass 1: the moments (M, V and the gradient in, M' and V' out)
    MomentumArgs m;
    m.w_in = dev_view(M_in, si[1]);
    m.m_in = dev_view(V_in, si[2]);
    m.w_out = dev_view(M_out, so[1]);
    m.m_out = dev_view(V_out, so[2]);
    m.g = d_g;
    m.cbw = dev_codebook(*cbM);
    m.cbm = dev_codebook(*cbV);
    std::memcpy(m.k, k, sizeof(k));
    m.op = OP2_ADAM_MOMENTS;
    m.in_place = (M_out->d_sf == M_in->d_sf || V_out->d_sf == V_in->d_sf) ? 1u : 0u;
    m.wait_ns = kDefaultWaitNs;
    set_multipliers(m);
    if (launch_momentum(m, st) != cudaSuccess) return LCT_ERR_CUDA;

    // pass 2: the weight (W, M' and V' in, W' out)
    UpdateArgs a;
    std::memset(&a, 0, sizeof(a));
    a.in[0] = dev_view(W_in, si[0]);
    a.in[1] = dev_view(M_out, so[1]);
    a.in[2] = dev_view(V_out, so[2]);
    a.w_out = dev_view(W_out, so[0]);
    a.cb[0] = dev_codebook(*cbW);
    a.cb[1] = dev_codebook(*cbM);
    a.cb[2] = dev_codebook(*cbV);
    std::memcpy(a.k, k, sizeof(k));
    a.op = OP_ADAMW;
    a.nin = 3;
    a.in_place = W_out->d_sf == W_in->d_sf ? 1u : 0u;
    a.wait_ns = kDefaultWaitNs;
    set_multipliers(a);
    return launch_update(a, st) == cudaSuccess ? LCT_OK : LCT_ERR_CUDA;
}

// ------------------------------------------------------------ test hook

namespace lct {
namespace dev {

// Runs the look-back of block 1 over a status array whose block 0 never
// publishes, in each of its forms (the warp reading every predecessor, the
// warp walking back window by window, the single thread); every bounded wait
// must run out, and only then is LCT_ERR_TIMEOUT latched.  One warp.
__global__ void k_wait_probe(lct_header *hdr, unsigned long long *work, uint64_t wait_ns)
{
    if (threadIdx.x == 0) {
        work[0] = 0ull;
        work[1] = 0ull;
        __threadfence();
    }
    __syncwarp();
    bool t_all = false, t_walk = false, t_one = false;
    warp_lookback_all(work, 1, 0, wait_ns, &t_all);
    warp_lookback_walk(work, 1, 0, wait_ns, &t_walk);
    if (threadIdx.x == 0) {
        lookback(work, 1, 0, wait_ns, &t_one);
        if (t_all && t_walk && t_one) latch(hdr, LCT_ERR_TIMEOUT);
    }
}

}  // namespace dev

cudaError_t launch_wait_probe(lct_header *hdr, unsigned long long *work, uint64_t wait_ns, cudaStream_t s)
{
    dev::k_wait_probe<<<1, 32, 0, s>>>(hdr, work, wait_ns);
    return cudaGetLastError();
}

}  // namespace lct

extern "C" lct_status lct_debug_wait_timeout(void *d_header, void *d_work, uint64_t limit_ns, void *stream)
{
    if (!d_header || !d_work || !aligned16(d_header) || !aligned16(d_work)) return LCT_ERR_INVALID_ARG;
    if (limit_ns == 0 || limit_ns > kDefaultWaitNs) return LCT_ERR_INVALID_ARG;
    return launch_wait_probe(static_cast<lct_header *>(d_header), static_cast<unsigned long long *>(d_work),
                             limit_ns, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? LCT_OK
               : LCT_ERR_CUDA;
}
