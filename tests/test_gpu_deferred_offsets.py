"""Block offsets written after the writer, on grids of many blocks.

[EXP] "Compressing is easy": every stream's spilled exponents go to one
uncompressed overflow region, and a block's bytes are found through the
prefix of the blocks' byte counts.  On a grid of at least four blocks per SM
the writers let a block with no overflow bytes publish its count and leave,
blocks with bytes to place still wait for their prefix, and a small kernel
writes the block offsets, ovf_used and the capacity check afterwards.  The
tensors below have 4 * SMs + 50 blocks or more, so they take that path; every
region must still equal the oracle's: spilling blocks among many that spill
nothing, every block spilling under a too-small overflow capacity, and
a fused SGD step and an in-place momentum step writing such a tensor."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, codebooks, gpu_decode, gpu_encode, to_device, workload

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A
ETA = float(np.float32(1e-3))


def _grid_blocks():
    return 4 * torch.cuda.get_device_properties(0).multi_processor_count + 50


def _mixed_laplace(seed=21):
    """Laplace(0.01) weights over many CLEAN blocks and a ragged tail, with
    20,000 random bit patterns written into four of the blocks: those spill
    (about 78 escaped exponents per stream); of the others most place nothing
    and some (a stream's Laplace tail) a few bytes."""
    nblocks = _grid_blocks()
    n = nblocks * 65536 + 777
    x = synth.laplace(n, 0.01, seed=seed)
    for i, b in enumerate((3, nblocks // 2, nblocks // 2 + 1, nblocks)):
        at = b * 65536
        x[at:at + min(20000, n - at)] = synth.random_bits(min(20000, n - at), seed=seed + i)
    return x


def test_mixed_spill_encode_and_decode():
    x = _mixed_laplace()
    cb, ocb = codebooks(1, 0.01)
    ct = gpu_encode(x, cb, 0)
    ref = oracle.encode(x, ocb, 0)
    assert ref.nblocks >= _grid_blocks()
    spilling = np.nonzero(np.diff(ref.blk_off))[0]
    assert {3, ref.nblocks // 2} <= set(spilling.tolist())  # the blocks given random bits spill
    assert spilling.size < ref.nblocks // 2  # most blocks place nothing
    got = ct.to_host()
    assert got["status"] == 0
    assert_same_format(got, ref)
    assert np.array_equal(gpu_decode(ct, cb), x)


def test_capacity_latched_with_deferred_offsets():
    """GELU activations in HIGH blocks (every block spills) with half the
    overflow capacity they need: CAPACITY latched, ovf_used the full need,
    every block offset and the bytes of the blocks that fit as the oracle
    writes them, and not one byte written past the capacity."""
    nblocks = _grid_blocks()
    x, m, s, sh, lv = workload("gelu_act", nblocks * 32768 + 5)
    cb, ocb = codebooks(m, s, sh)
    full = oracle.encode(x, ocb, lv)
    cap = int(full.ovf_used) // 2
    short = oracle.encode(x, ocb, lv, ovf_cap=cap)
    assert short.status == oracle.CAPACITY
    buf = torch.full((cap + 4096,), SENTINEL, dtype=torch.uint8, device="cuda")
    ct = B.CompressedTensor(x.size, lv, ovf=buf[:cap])
    B.lct_encode(to_device(x), cb, ct)
    torch.cuda.synchronize()
    st = ct.state()
    assert st.status == B.LCT_ERR_OVERFLOW_CAPACITY and st.ovf_used == full.ovf_used
    assert_same_format(ct.to_host(), short)
    assert (buf[cap:].cpu().numpy() == SENTINEL).all()


def test_sgd_step_on_mixed_tensor():
    w = _mixed_laplace(seed=23)
    n = w.size
    m = synth.laplace(n, 1e-3, seed=24)
    cbw, ocbw = codebooks(1, 0.01)
    cbm, ocbm = codebooks(1, 1e-3)
    W, M = gpu_encode(w, cbw, 0), gpu_encode(m, cbm, 0)
    out = B.CompressedTensor(n, 0)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    ref = oracle.sgd_step(oracle.encode(w, ocbw, 0), ocbw, oracle.encode(m, ocbm, 0), ocbm, ETA)
    got = out.to_host()
    assert got["status"] == ref.status == 0
    assert np.diff(ref.blk_off).any()  # the new W still has spilling blocks
    assert_same_format(got, ref)


def test_momentum_step_in_place_on_mixed_tensor():
    w = _mixed_laplace(seed=25)
    n = w.size
    m = synth.laplace(n, 1e-3, seed=26)
    g = synth.normal(n, 1e-4, seed=27)
    cbw, ocbw = codebooks(1, 0.01)
    cbm, ocbm = codebooks(1, 1e-3)
    W, M = gpu_encode(w, cbw, 0), gpu_encode(m, cbm, 0)
    W2, M2 = B.CompressedTensor(n, 0, like=W), B.CompressedTensor(n, 0, like=M)
    eta, mu = float(np.float32(1e-3)), float(np.float32(0.9))
    B.lct_sgd_momentum_step_fused(W, cbw, M, cbm, to_device(g), eta, mu, W2, M2)
    torch.cuda.synchronize()
    ref_w, ref_m = oracle.sgd_momentum_step(oracle.encode(w, ocbw, 0), ocbw, oracle.encode(m, ocbm, 0), ocbm, g,
                                            eta, mu)
    for t, r in ((W2, ref_w), (M2, ref_m)):
        got = t.to_host()
        assert got["status"] == r.status == 0
        assert_same_format(got, r)
