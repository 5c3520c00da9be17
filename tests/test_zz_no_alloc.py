"""lct_encode_static_scratch -- the encode entry point for callers that
cannot allocate device memory (an allocator or out-of-memory handler that
compresses tensors to free space, code that must not call cudaMalloc) -- must
write exactly what lct_encode writes.  Called through the C ABI twice in a
row, since every call shares one scratch array inside the library.  This file
is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth


def _regions(ct):
    h = ct.to_host()
    return {k: h[k] for k in ("sf", "slots", "markers", "blk_off", "delta", "status", "ovf_used")} | {
        "ovf": h["ovf"][: h["ovf_used"]]}


@pytest.mark.gpu
def test_static_scratch_encode_matches_lct_encode_twice():
    cases = [(synth.laplace(5 * 65536 + 777, 0.01, seed=21), B.lct_codebook_build(1, 0.01), 0),
             (synth.gelu_sparse(9 * 32768 + 5, seed=22), B.lct_codebook_build(0, 1.0), 2)]
    for x_np, cb, level in cases:          # two calls in a row, different sizes and levels
        x = torch.from_numpy(x_np.view(np.int16)).cuda()
        ref = B.CompressedTensor(x_np.size, level)
        B.lct_encode(x, cb, ref)
        got = B.CompressedTensor(x_np.size, level)
        got.desc.d_work = None              # no caller scratch
        rc = B.library().lct_encode_static_scratch(x.data_ptr(), ctypes.byref(cb), ctypes.byref(got.desc),
                                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == B.LCT_OK
        torch.cuda.synchronize()
        a, b = _regions(ref), _regions(got)
        assert a["status"] == b["status"] == 0
        for k in a:
            assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k
        y = torch.empty_like(x)
        B.lct_decode(got, cb, y)
        torch.cuda.synchronize()
        assert torch.equal(y, x)


@pytest.mark.gpu
def test_static_scratch_rejects_tensors_beyond_its_limit():
    t = B.lct_tensor()
    t.n, t.level = B.LCT_STATIC_SCRATCH_BLOCKS * 65536 + 1, 0
    cb = B.lct_codebook_build(0, 0.02)
    rc = B.library().lct_encode_static_scratch(None, ctypes.byref(cb), ctypes.byref(t), None)
    assert rc == B.LCT_ERR_UNSUPPORTED
