"""GPU parity of the fused compressed SGD-with-momentum step
M <- bf16(mu*M + g), W <- bf16(W - eta*M) against the CPU oracle: every region
of both new compressed tensors must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, codebooks, gpu_decode, gpu_encode, to_device

pytestmark = pytest.mark.gpu

ETA = float(np.float32(1e-3))
MU = float(np.float32(0.9))


def _setup(w, m, level, wmodel=(0, 0.02, 0.0), mmodel=(0, 1e-3, 0.0)):
    cbw, ocbw = codebooks(*wmodel)
    cbm, ocbm = codebooks(*mmodel)
    return (gpu_encode(w, cbw, level), gpu_encode(m, cbm, level), cbw, cbm,
            oracle.encode(w, ocbw, level), oracle.encode(m, ocbm, level), ocbw, ocbm)


def _run(W, M, cbw, cbm, g, ow, om, mu=MU):
    B.lct_sgd_momentum_step_fused(W, cbw, M, cbm, to_device(g), ETA, mu, ow, om)
    torch.cuda.synchronize()
    return ow.to_host(), om.to_host()


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 300, 65536, 2 * 65536 + 777])
def test_momentum_step_matches_oracle(level, n):
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    g = synth.normal(n, 1e-4, 6)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, level)
    gw, gm = _run(W, M, cbw, cbm, g, B.CompressedTensor(n, level), B.CompressedTensor(n, level))
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, ETA, MU)
    assert gw["status"] == rw.status == 0 and gm["status"] == rm.status == 0
    assert_same_format(gw, rw)
    assert_same_format(gm, rm)


@pytest.mark.parametrize("which", ["both", "w", "m"])
def test_momentum_in_place_equals_oracle(which):
    """Outputs sharing their input's header, sign-fraction bytes, slots,
    markers and offsets (only overflow and scratch are their own)."""
    n = 3 * 65536 + 1001
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    g = synth.normal(n, 1e-4, 6)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 0)
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, ETA, MU)
    ow = B.CompressedTensor(n, 0, like=W) if which in ("both", "w") else B.CompressedTensor(n, 0)
    om = B.CompressedTensor(n, 0, like=M) if which in ("both", "m") else B.CompressedTensor(n, 0)
    gw, gm = _run(W, M, cbw, cbm, g, ow, om)
    assert_same_format(gw, rw)
    assert_same_format(gm, rm)


@pytest.mark.parametrize("level", [0, 2])
@pytest.mark.parametrize("in_place", [False, True])
def test_momentum_heavy_spill_and_special_values(level, in_place):
    """Momentum with exponents spread over the whole range (nearly every new
    M exponent escapes, whatever the shift, so every stream spills most of
    its rows: more than the rows an out-of-place step keeps), an
    activation-like W that spills too, and zeros, subnormals, infinities and
    NaNs among the values."""
    bsz = 65536 if level == 0 else 32768
    n = 3 * bsz + 4321
    w = synth.gelu_sparse(n, seed=5)
    m = synth.random_bits(n, 8)
    g = synth.normal(n, 0.1, 9)
    w[:6] = [0x0001, 0x8001, 0x7F80, 0xFF80, 0x7FC1, 0x0000]
    m[:6] = [0x3F80, 0x0001, 0x7F80, 0x3F80, 0x0000, 0x7FA0]
    g[:6] = [0x8000, 0x0001, 0xFF80, 0x0000, 0x7FC0, 0x3F80]
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, level, wmodel=(0, 1.0, 0.0))
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, ETA, MU)
    nj = 256 if level == 0 else 128
    assert (rm.markers.astype(int) < nj - 40).mean() > 0.9   # beyond the 32 kept rows
    assert rw.ovf_used > 0
    ow = B.CompressedTensor(n, level, like=W) if in_place else B.CompressedTensor(n, level)
    om = B.CompressedTensor(n, level, like=M) if in_place else B.CompressedTensor(n, level)
    gw, gm = _run(W, M, cbw, cbm, g, ow, om)
    assert gw["status"] == 0 and gm["status"] == 0
    assert_same_format(gw, rw)
    assert_same_format(gm, rm)


def test_momentum_capacity_is_per_output():
    """Too little overflow room for the new momentum: M' latches capacity,
    W' is unaffected and still exact."""
    n = 2 * 65536 + 99
    w = synth.normal(n, 0.02, 3)
    m = synth.random_bits(n, 8)
    g = synth.normal(n, 0.1, 9)
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 0)
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, ETA, MU, ovf_cap_m=1000)
    assert rm.status == oracle.CAPACITY and rw.status == 0
    gw, gm = _run(W, M, cbw, cbm, g, B.CompressedTensor(n, 0), B.CompressedTensor(n, 0, ovf_cap=1000))
    assert gw["status"] == 0 and gm["status"] == B.LCT_ERR_OVERFLOW_CAPACITY
    assert gm["ovf_used"] == rm.ovf_used
    assert_same_format(gw, rw)


def test_momentum_corrupt_input_latches_both_outputs():
    n = 65536
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    g = synth.normal(n, 1e-4, 6)
    W, M, cbw, cbm, *_ = _setup(w, m, 0)
    M.regions["markers"].fill_(0xFF)             # markers beyond the stream length
    gw, gm = _run(W, M, cbw, cbm, g, B.CompressedTensor(n, 0), B.CompressedTensor(n, 0))
    assert gw["status"] == B.LCT_ERR_CORRUPT and gm["status"] == B.LCT_ERR_CORRUPT


def test_momentum_162m_step_one_full_and_sampled_steps():
    """162,000,000 values, CLEAN, both outputs in place with ping-pong
    overflow buffers, ten steps with alternating seeded gradients.  Step 1 is
    compared in full with the oracle; after step 10 a sample of blocks (first,
    middle, last partial) is compared with the oracle run on those blocks
    alone (blocks are independent given the fixed shifts)."""
    name = "momentum_162m"
    wl = synth.WORKLOADS[name]
    n = wl["n"]
    w = synth.generate(name)
    m = synth.momentum(name)
    grads = [synth.gradient(name, 1), synth.gradient(name, 2)]
    eta, mu = float(np.float32(wl["eta"])), float(np.float32(wl["mu"]))
    cbw, ocbw = codebooks(0, wl["scale"])
    cbm, ocbm = codebooks(0, wl["momentum"]["scale"])
    W = gpu_encode(w, cbw, 0)
    M = gpu_encode(m, cbm, 0)
    dw, dm = W.to_host()["delta"], M.to_host()["delta"]
    gdev = [to_device(g) for g in grads]
    wbufs = [B.CompressedTensor(n, 0, like=W), B.CompressedTensor(n, 0, like=W)]
    mbufs = [B.CompressedTensor(n, 0, like=M), B.CompressedTensor(n, 0, like=M)]
    cw, cm = W, M
    for step in range(1, 11):
        nw, nm = wbufs[step % 2], mbufs[step % 2]
        B.lct_sgd_momentum_step_fused(cw, cbw, cm, cbm, gdev[(step - 1) % 2], eta, mu, nw, nm)
        cw, cm = nw, nm
        if step == 1:
            torch.cuda.synchronize()
            rw, rm = oracle.sgd_momentum_step(oracle.encode(w, ocbw, 0), ocbw, oracle.encode(m, ocbm, 0), ocbm,
                                              grads[0], eta, mu)
            assert_same_format(cw.to_host(), rw)
            assert_same_format(cm.to_host(), rm)
            del rw, rm
    torch.cuda.synchronize()
    gw, gm = cw.to_host(), cm.to_host()
    assert gw["status"] == 0 and gm["status"] == 0 and gw["delta"] == dw and gm["delta"] == dm
    nb, block, W_ = W.nblocks, 65536, 25 * 256
    for b in [0, 1, nb // 2, nb - 2, nb - 1]:
        s = slice(b * block, min((b + 1) * block, n))
        ow = oracle.encode(w[s], ocbw, 0, delta=dw)
        om = oracle.encode(m[s], ocbm, 0, delta=dm)
        for step in range(1, 11):
            ow, om = oracle.sgd_momentum_step(ow, ocbw, om, ocbm, grads[(step - 1) % 2][s], eta, mu)
        for got, ref in ((gw, ow), (gm, om)):
            assert np.array_equal(got["sf"][s], ref.sf), b
            assert np.array_equal(got["slots"][b * W_:(b + 1) * W_], ref.slots), b
            assert np.array_equal(got["markers"][b * 256:(b + 1) * 256], ref.markers), b
            o0, o1 = int(got["blk_off"][b]), int(got["blk_off"][b + 1])
            assert o1 - o0 == ref.ovf_used and np.array_equal(got["ovf"][o0:o1], ref.ovf[:ref.ovf_used])
    # the decoded weights agree with the oracle's on the sampled blocks
    y = gpu_decode(cw, cbw)
    rc, yref = oracle.decode(ow, ocbw)
    assert rc == 0 and np.array_equal(y[(nb - 1) * block:], yref)


@pytest.mark.parametrize("eta, mu", [(0.0, 0.9), (1e-3, 0.0), (1e-3, -0.5), (0.75, 1.5), (1e-3, 1e-40),
                                     (float("inf"), 0.9), (1e-3, float("inf")), (1e-3, float("nan")),
                                     (float("nan"), 0.9)])
@pytest.mark.parametrize("large", [False, True])
def test_momentum_hyperparameter_edge_cases(eta, mu, large):
    """eta and mu zero, negative, above one, subnormal in float32, infinite
    and NaN.  Both new states follow M' = bf16(fl32(fl32(mu*m) + g)) and
    W' = bf16(fl32(w - fl32(eta*M'))) for any float32 eta and mu, NaN written
    as 0x7FC0; both must equal the oracle's bit for bit on a small grid and on
    a grid of more than two blocks per SM."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nblocks = 2 * sms + 3 if large else 3
    n = nblocks * 65536 - 555
    w = synth.normal(n, 0.02, 43)
    m = synth.normal(n, 1e-3, 44)
    g = synth.normal(n, 1e-4, 45)
    w[:4] = [0x0000, 0x8000, 0x0001, 0x7F80]  # +0, -0, a subnormal, +inf
    m[:4] = [0x3F80, 0x0000, 0xBF80, 0x0000]
    eta32, mu32 = float(np.float32(eta)), float(np.float32(mu))
    W, M, cbw, cbm, oW, oM, ocbw, ocbm = _setup(w, m, 0)
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, eta32, mu32)
    ow, om = B.CompressedTensor(n, 0), B.CompressedTensor(n, 0)
    B.lct_sgd_momentum_step_fused(W, cbw, M, cbm, to_device(g), eta32, mu32, ow, om)
    torch.cuda.synchronize()
    gw, gm = ow.to_host(), om.to_host()
    assert gw["status"] == rw.status == 0 and gm["status"] == rm.status == 0
    assert_same_format(gw, rw)
    assert_same_format(gm, rm)
