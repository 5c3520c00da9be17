// lct_encode_static_scratch: lct_encode for callers that cannot allocate
// device memory at all.
//
// lct_encode needs a little scratch (one 8-byte status word per block, the
// `d_work` region) for the single-pass scan that places each block's
// overflow bytes.  Some callers cannot provide it: a caching allocator or an
// out-of-memory handler that compresses tensors to free space would have to
// re-enter the allocator -- or fail for lack of memory -- to get scratch, and
// some code must avoid cudaMalloc/cudaFree because they can synchronise the
// device.  This entry point takes its scratch from a fixed array that lives
// in the library's own device image instead; the caller still passes the
// input and the compressed tensor's regions, exactly as for lct_encode.
#include <cstdint>

#include "../../include/lct.h"
#include "internal.h"

namespace {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned long long g_static_scan_words[LCT_STATIC_SCRATCH_BLOCKS];

// Device address of the array on the current device, looked up on every
// call: in host code the array's name is only a host-side stand-in, so a
// kernel must be given this address, never the name itself.  Not caching it
// keeps it right after cudaDeviceReset or a new primary context.  The first
// lookup on a device may load the library's device code there.
lct_status scan_words_on_current_device(void **out)
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scan_words) != cudaSuccess || !p) return LCT_ERR_CUDA;
    *out = p;
    return LCT_OK;
}

}  // namespace

extern "C" lct_status lct_encode_static_scratch(const uint16_t *d_x, const lct_codebook *cb, const lct_tensor *t,
                                                void *stream)
{
    lct::Geometry g;
    if (!t || !lct::level_geometry(t->level, &g)) return LCT_ERR_INVALID_ARG;
    const uint64_t nblocks = (t->n + g.block - 1) / g.block;
    if (nblocks > LCT_STATIC_SCRATCH_BLOCKS) return LCT_ERR_UNSUPPORTED;
    void *scan_words = nullptr;
    const lct_status rc = scan_words_on_current_device(&scan_words);
    if (rc != LCT_OK) return rc;
    // Same checks and launches as lct_encode; only the scratch differs.  The
    // encode prologue clears the status words it uses on every call, so the
    // previous call's contents never leak into this one.
    lct_tensor view = *t;
    view.d_work = scan_words;
    return lct_encode(d_x, cb, &view, stream);
}
