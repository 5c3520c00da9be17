"""GPU parity of the fused compressed SGD step W <- W - eta*M against the CPU
oracle: every region of the new compressed W must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, codebooks, gpu_decode, gpu_encode

pytestmark = pytest.mark.gpu

ETA = float(np.float32(1e-3))


def _setup(w, m, level, wmodel=(0, 0.02, 0.0), mmodel=(0, 1e-3, 0.0)):
    cbw, ocbw = codebooks(*wmodel)
    cbm, ocbm = codebooks(*mmodel)
    W = gpu_encode(w, cbw, level)
    M = gpu_encode(m, cbm, level)
    oW = oracle.encode(w, ocbw, level)
    oM = oracle.encode(m, ocbm, level)
    return W, M, cbw, cbm, oW, oM, ocbw, ocbm


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 300, 65536, 2 * 65536 + 777])
def test_sgd_step_matches_oracle(level, n):
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, level)
    out = B.CompressedTensor(n, level)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, ETA)
    got = out.to_host()
    assert got["status"] == ref.status == 0
    assert_same_format(got, ref)
    rc, yref = oracle.decode(ref, ocbw)
    assert np.array_equal(gpu_decode(out, cbw), yref)


def test_sgd_in_place_equals_out_of_place():
    n = 3 * 65536 + 1001
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 0)
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, ETA)
    # W_out shares W's header, sign-fraction, slots, markers and offsets;
    # only the overflow and the scratch are its own.
    out = B.CompressedTensor(n, 0, like=W)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    assert_same_format(out.to_host(), ref)


def test_sgd_with_spill_and_special_values():
    """Activation-like W that spills (HIGH), with zeros, subnormals, infinities
    and NaNs among the values."""
    n = 4 * 32768 + 123
    w = synth.gelu_sparse(n, seed=5)
    m = synth.normal(n, 1e-3, 4)
    w[:6] = [0x0001, 0x8001, 0x7F80, 0xFF80, 0x7FC1, 0x0000]
    m[:6] = [0x3F80, 0x0001, 0x7F80, 0x3F80, 0x0000, 0x7FA0]
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 2, wmodel=(0, 1.0, 0.0))
    assert oW.ovf_used > 0
    out = B.CompressedTensor(n, 2)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, ETA)
    assert_same_format(out.to_host(), ref)


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("in_place", [False, True])
def test_sgd_worst_case_spill(level, in_place):
    """Every new exponent of the first block is 255 (W is NaN there), which no
    codebook codes: each of its streams keeps exactly 2W escapes (16 bits
    each) in its slot and spills all the rest, the most an in-place step has
    to keep.  The other blocks hold uniformly random bit patterns (mostly
    escapes too), so an out-of-place step spills far beyond its kept rows."""
    bsz = 65536 if level == 0 else 32768
    words = {0: 25, 1: 16, 2: 20}[level]
    n = 2 * bsz + 999
    w = synth.random_bits(n, 21)
    w[:bsz] = 0x7FC1
    m = synth.normal(n, 1e-3, 4)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, level)
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, ETA)
    assert (ref.markers[:256] == 2 * words).all()
    out = B.CompressedTensor(n, level, like=W) if in_place else B.CompressedTensor(n, level)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    got = out.to_host()
    assert got["status"] == ref.status == 0
    assert_same_format(got, ref)


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("in_place", [False, True])
def test_sgd_spill_on_a_grid_of_more_than_two_blocks_per_sm(level, in_place):
    """The worst-case spill data above on a grid of 2 * SMs + 40 blocks, which
    runs the SGD kernel built for throughput (three CTAs per SM out of place)
    instead of the software-pipelined one the small tests above reach; the
    blocks that spill are spread over the grid."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bsz = 65536 if level == 0 else 32768
    nblocks = 2 * sms + 40
    n = nblocks * bsz - 777
    w = synth.normal(n, 0.02, 31)
    for b in (0, nblocks // 3, nblocks - 1):  # blocks of NaN and of random bit patterns
        w[b * bsz:b * bsz + bsz // 2] = synth.random_bits(bsz // 2, 32 + b)
    w[bsz // 2:bsz] = 0x7FC1
    m = synth.normal(n, 1e-3, 4)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, level)
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, ETA)
    assert ref.ovf_used > 0
    out = B.CompressedTensor(n, level, like=W) if in_place else B.CompressedTensor(n, level)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    got = out.to_host()
    assert got["status"] == ref.status == 0
    assert_same_format(got, ref)


def test_sgd_162m_step_one_full_and_sampled_steps():
    """162,000,000-value W ~ N(0, 0.02) and M ~ N(0, 1e-3), CLEAN, eta = 1e-3,
    100 steps on the GPU with ping-pong overflow buffers.  Step 1 is compared
    in full with the oracle; after steps 2, 10 and 100 a sample of blocks
    (first, middle, last partial) is compared with the oracle run on those
    blocks alone (blocks are independent given the fixed shift), and the block
    offsets with the markers."""
    name = "sgd_162m"
    wl = synth.WORKLOADS[name]
    n = wl["n"]
    w = synth.generate(name)
    m = synth.momentum(name)
    cbw, ocbw = codebooks(0, wl["scale"])
    cbm, ocbm = codebooks(0, wl["momentum"]["scale"])
    W = gpu_encode(w, cbw, 0)
    M = gpu_encode(m, cbm, 0)
    delta_w = W.to_host()["delta"]
    assert delta_w == oracle.shift(w, ocbw.median_exp)
    A, Bt = W, B.CompressedTensor(n, 0, like=W)     # in place, overflow ping-pong
    Bt2 = B.CompressedTensor(n, 0, like=W)
    bufs = [Bt, Bt2]
    nb = A.nblocks
    sample = [0, 1, nb // 2, nb - 2, nb - 1]
    block = 65536
    oM_delta = M.to_host()["delta"]

    def oracle_blocks(step):
        out = {}
        for b in sample:
            s = slice(b * block, min((b + 1) * block, n))
            ow = oracle.encode(w[s], ocbw, 0, delta=delta_w)
            om = oracle.encode(m[s], ocbm, 0, delta=oM_delta)
            for _ in range(step):
                ow = oracle.sgd_step(ow, ocbw, om, ocbm, ETA)
            out[b] = ow
        return out

    cur = A
    for step in range(1, 101):
        nxt = bufs[step % 2]
        B.lct_sgd_step_fused(cur, cbw, M, cbm, ETA, nxt)
        cur = nxt
        if step == 1:
            torch.cuda.synchronize()
            ref = oracle.sgd_step(oracle.encode(w, ocbw, 0), ocbw, oracle.encode(m, ocbm, 0), ocbm, ETA)
            assert_same_format(cur.to_host(), ref)
            del ref
        if step in (2, 10, 100):
            torch.cuda.synchronize()
            got = cur.to_host()
            assert got["status"] == 0 and got["delta"] == delta_w
            refs = oracle_blocks(step)
            for b, ob in refs.items():
                W_ = 25 * 256
                s = slice(b * block, min((b + 1) * block, n))
                assert np.array_equal(got["sf"][s], ob.sf), (step, b)
                assert np.array_equal(got["slots"][b * W_:(b + 1) * W_], ob.slots), (step, b)
                assert np.array_equal(got["markers"][b * 256:(b + 1) * 256], ob.markers), (step, b)
                o0, o1 = int(got["blk_off"][b]), int(got["blk_off"][b + 1])
                assert o1 - o0 == ob.ovf_used and np.array_equal(got["ovf"][o0:o1], ob.ovf[:ob.ovf_used])
            # offsets = prefix of the per-block spill implied by the markers
            nj = np.full(nb * 256, 256, np.int64)
            last = n - (nb - 1) * block
            nj[(nb - 1) * 256:] = [max(0, -(-(last - j) // 256)) for j in range(256)]
            spill = (nj - got["markers"].astype(np.int64)).reshape(nb, 256).sum(1)
            assert np.array_equal(got["blk_off"], np.concatenate([[0], np.cumsum(spill)]).astype(np.uint64))


@pytest.mark.parametrize("eta", [0.0, -1e-3, 0.5, 3.0e4, 1e-40, float("inf"), float("-inf"), float("nan")])
@pytest.mark.parametrize("large", [False, True])
def test_sgd_eta_edge_cases(eta, large):
    """eta zero, negative, large (the exponents move, so few groups keep their
    old codes and many values escape and spill), subnormal in float32, and
    infinite or NaN (every new value infinite or NaN, exponent 255, which no
    codebook codes).  The step is W' = bf16(fl32(w - fl32(eta*m))) for any
    float32 eta ([EXP] "Training adds a second problem"), with NaN written as
    0x7FC0; the new W must equal the oracle's bit for bit, both on a small grid
    (the software-pipelined kernel) and on a grid of more than two blocks per
    SM (the throughput kernel, which canonicalises NaN everywhere only when
    eta is not finite)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nblocks = 2 * sms + 3 if large else 3
    n = nblocks * 65536 - 555
    w = synth.normal(n, 0.02, 41)
    m = synth.normal(n, 1e-3, 42)
    w[:4] = [0x0000, 0x8000, 0x0001, 0x7F80]  # +0, -0, a subnormal, +inf
    m[:4] = [0x3F80, 0x0000, 0xBF80, 0x3F80]
    eta32 = float(np.float32(eta))
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 0)
    ref = oracle.sgd_step(oW, ocbw, oM, ocbm, eta32)
    out = B.CompressedTensor(n, 0)
    B.lct_sgd_step_fused(W, cbw, M, cbm, eta32, out)
    torch.cuda.synchronize()
    got = out.to_host()
    assert got["status"] == ref.status == 0
    assert_same_format(got, ref)
    rc, yref = oracle.decode(ref, ocbw)
    assert np.array_equal(gpu_decode(out, cbw), yref)
