"""GPU parity of coding with a zero-atom codebook (a point mass at exponent 0
that is never shifted) against the CPU oracle: encode, decode, the fused SGD
and the fused momentum step, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, gpu_decode, gpu_encode, to_device, workload

pytestmark = pytest.mark.gpu

ETA = float(np.float32(1e-3))


def _books(model=0, scale=1.0, shape=0.0, zf=0.3):
    return (B.lct_codebook_build_zero_atom(model, scale, shape, zf),
            oracle.codebook_build_zero_atom(model, scale, shape, zf))


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 300, 2 * 65536 + 777])
def test_zero_atom_roundtrip_matches_oracle(level, n):
    x = synth.gelu_sparse(n, seed=5)
    cb, ocb = _books()
    ct = gpu_encode(x, cb, level)
    ref = oracle.encode(x, ocb, level)
    got = ct.to_host()
    assert got["status"] == ref.status == 0
    assert_same_format(got, ref)
    assert np.array_equal(gpu_decode(ct, cb), x)


@pytest.mark.parametrize("level", [0, 2])
def test_zero_atom_every_bf16_pattern(level):
    x = synth.all_bf16_patterns()
    for k in (-20, 0, 20):          # move the shift, and with it the collision with symbol 0
        xk = synth.scale_pow2(x, k) if k else x
        cb, ocb = _books()
        ct = gpu_encode(xk, cb, level)
        assert_same_format(ct.to_host(), oracle.encode(xk, ocb, level))
        assert np.array_equal(gpu_decode(ct, cb), xk)


def test_zero_atom_gelu_pow2_rounds_full_size():
    """[8, 4096, 3072] GELU activations with 30% zeros under a zero-atom
    Gaussian(1) codebook, scaled by 2^k: parity on three rounds; on all nine
    the markers and overflow size stay put, and the overflow is a fraction of
    the plain codebook's."""
    x0, m, s, sh, lv = workload("gelu_act")
    cb, ocb = _books(m, s, sh, 0.3)
    plain = B.lct_codebook_build(m, s, sh)
    used_plain = gpu_encode(x0, plain, lv).state().ovf_used
    markers0 = used0 = None
    for k in range(-4, 5):
        xk = synth.scale_pow2(x0, k)
        ct = gpu_encode(xk, cb, lv)
        got = ct.to_host()
        assert got["status"] == 0
        if k in (-4, 0, 4):
            assert_same_format(got, oracle.encode(xk, ocb, lv))
        if markers0 is None:
            markers0, used0 = got["markers"].copy(), got["ovf_used"]
        assert np.array_equal(got["markers"], markers0) and got["ovf_used"] == used0
        assert np.array_equal(gpu_decode(ct, cb), xk)
        del ct
    assert used0 < used_plain / 4


@pytest.mark.parametrize("in_place", [False, True])
def test_zero_atom_sgd_and_momentum(in_place):
    """Activation-like W (30% zeros) under a zero-atom codebook through the
    fused SGD and momentum steps; M with its own zero-atom codebook."""
    n = 3 * 32768 + 4321
    w = synth.gelu_sparse(n, seed=5)
    m = synth.normal(n, 1e-3, 4)
    m[::3] = 0
    g = synth.normal(n, 1e-4, 6)
    cbw, ocbw = _books(0, 1.0, 0.0, 0.3)
    cbm, ocbm = _books(0, 1e-3, 0.0, 0.33)
    W, M = gpu_encode(w, cbw, 2), gpu_encode(m, cbm, 2)
    oW, oM = oracle.encode(w, ocbw, 2), oracle.encode(m, ocbm, 2)
    out = B.CompressedTensor(n, 2, like=W) if in_place else B.CompressedTensor(n, 2)
    B.lct_sgd_step_fused(W, cbw, M, cbm, ETA, out)
    torch.cuda.synchronize()
    assert_same_format(out.to_host(), oracle.sgd_step(oW, ocbw, oM, ocbm, ETA))
    W, M = gpu_encode(w, cbw, 2), gpu_encode(m, cbm, 2)
    ow = B.CompressedTensor(n, 2, like=W) if in_place else B.CompressedTensor(n, 2)
    om = B.CompressedTensor(n, 2, like=M) if in_place else B.CompressedTensor(n, 2)
    B.lct_sgd_momentum_step_fused(W, cbw, M, cbm, to_device(g), ETA, 0.9, ow, om)
    torch.cuda.synchronize()
    rw, rm = oracle.sgd_momentum_step(oW, ocbw, oM, ocbm, g, ETA, float(np.float32(0.9)))
    assert_same_format(ow.to_host(), rw)
    assert_same_format(om.to_host(), rm)
