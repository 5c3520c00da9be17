"""Several compressed tensors whose overflow regions are slices of one shared
buffer ([EXP] "Here is the idealized arithmetic": activations, buffers and
the shared overflow buffer also count toward memory).  Each tensor must match
the oracle and decode exactly, the bytes between the slices must stay
untouched, and a tensor whose slice is too small latches its own capacity
error without writing past its slice or disturbing its neighbours."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, gpu_decode, to_device

pytestmark = pytest.mark.gpu

SENTINEL = 0xA5


def _cases():
    """Three spilling tensors at three levels: GELU activations under a
    Gaussian(1) model (HIGH), and uniformly random bit patterns (nearly every
    exponent escapes) in CLEAN and in MEDIUM blocks."""
    return [
        (synth.gelu_sparse(3 * 32768 + 11, seed=41), (0, 1.0, 0.0), 2),
        (synth.random_bits(2 * 65536 + 5, seed=42), (1, 0.01, 0.0), 0),
        (synth.random_bits(4 * 32768 + 3, seed=43), (2, 1e-3, 3.0), 1),
    ]


def _carve(sizes, gap=256):
    """Slice offsets for the given capacities, each start 256-byte aligned and
    followed by at least `gap` sentinel bytes."""
    offs, at = [], 0
    for s in sizes:
        offs.append(at)
        at = (at + s + gap + 255) // 256 * 256
    return offs, at


def _encode_into_shared(cases, caps):
    offs, total = _carve(caps)
    shared = torch.full((total,), SENTINEL, dtype=torch.uint8, device="cuda")
    cts = []
    for (x, (m, s, sh), lv), o, c in zip(cases, offs, caps):
        cb = B.lct_codebook_build(m, s, sh)
        ct = B.CompressedTensor(x.size, lv, ovf=shared[o:o + c])
        B.lct_encode(to_device(x), cb, ct)
        cts.append((ct, cb))
    torch.cuda.synchronize()
    return shared, offs, cts


def test_three_tensors_share_one_overflow_buffer():
    cases = _cases()
    refs = [oracle.encode(x, oracle.codebook_build(m, s, sh), lv) for x, (m, s, sh), lv in cases]
    assert all(r.ovf_used > 1000 for r in refs)  # every tensor spills
    caps = [r.ovf_used for r in refs]           # exact fit
    shared, offs, cts = _encode_into_shared(cases, caps)
    host = shared.cpu().numpy()
    for (ct, cb), ref, (x, _, _), o, c in zip(cts, refs, cases, offs, caps):
        got = ct.to_host()
        assert got["status"] == 0
        assert_same_format(got, ref)
        assert np.array_equal(host[o:o + c], ref.overflow_bytes())
        assert np.array_equal(gpu_decode(ct, cb), x)
    # nothing was written outside the slices
    inside = np.zeros(host.size, bool)
    for o, c in zip(offs, caps):
        inside[o:o + c] = True
    assert (host[~inside] == SENTINEL).all()


def test_overrun_in_one_slice_latches_only_that_tensor():
    cases = _cases()
    refs = [oracle.encode(x, oracle.codebook_build(m, s, sh), lv) for x, (m, s, sh), lv in cases]
    caps = [r.ovf_used for r in refs]
    caps[1] -= 1                                # the middle tensor is one byte short
    shared, offs, cts = _encode_into_shared(cases, caps)
    host = shared.cpu().numpy()
    short = oracle.encode(cases[1][0], oracle.codebook_build(*cases[1][1]), cases[1][2], ovf_cap=caps[1])
    assert short.status == oracle.CAPACITY
    for i, ((ct, cb), ref, (x, _, _), o, c) in enumerate(zip(cts, refs, cases, offs, caps)):
        st = ct.state()
        if i == 1:
            assert st.status == B.LCT_ERR_OVERFLOW_CAPACITY and st.ovf_used == ref.ovf_used
            assert_same_format(ct.to_host(), short)  # the blocks that fit are written as the oracle writes them
        else:
            assert st.status == 0
            assert np.array_equal(host[o:o + c], ref.overflow_bytes())
            assert np.array_equal(gpu_decode(ct, cb), x)
    inside = np.zeros(host.size, bool)
    for o, c in zip(offs, caps):
        inside[o:o + c] = True
    assert (host[~inside] == SENTINEL).all()      # in particular the byte right after the short slice
