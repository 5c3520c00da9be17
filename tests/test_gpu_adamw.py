"""GPU parity of the fused AdamW step (moments pass, then weight pass) on
compressed W, M and V against the CPU oracle: every region of the three new
compressed tensors must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, codebooks, gpu_encode, to_device

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def _inputs(n, seed=0):
    w = synth.normal(n, 0.02, 3 + seed)
    m = synth.normal(n, 1e-4, 4 + seed)
    v = synth.bf16_bits(np.abs(synth.bits_to_f32(synth.normal(n, 1e-8, 5 + seed))))
    g = synth.normal(n, 1e-4, 6 + seed)
    return w, m, v, g


MODELS = ((0, 0.02, 0.0), (0, 1e-4, 0.0), (1, 1e-8, 0.0))


def _setup(w, m, v, level):
    books = [codebooks(*md) for md in MODELS]
    gpu = [gpu_encode(x, cb, level) for x, (cb, _) in zip((w, m, v), books)]
    ref = [oracle.encode(x, ocb, level) for x, (_, ocb) in zip((w, m, v), books)]
    return gpu, ref, [cb for cb, _ in books], [ocb for _, ocb in books]


def _step(gpu, cbs, g, t, outs):
    B.lct_adamw_step_fused(gpu[0], cbs[0], gpu[1], cbs[1], gpu[2], cbs[2], to_device(g), HP["lr"], HP["beta1"],
                           HP["beta2"], HP["eps"], HP["weight_decay"], t, *outs)
    torch.cuda.synchronize()
    return [o.to_host() for o in outs]


def _k(t):
    return oracle.adamw_constants(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], t)


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 300, 2 * 65536 + 777])
def test_adamw_matches_oracle(level, n):
    w, m, v, g = _inputs(n)
    gpu, ref, cbs, ocbs = _setup(w, m, v, level)
    outs = [B.CompressedTensor(n, level) for _ in range(3)]
    got = _step(gpu, cbs, g, 3, outs)
    exp = oracle.adamw_step(ref[0], ocbs[0], ref[1], ocbs[1], ref[2], ocbs[2], g, _k(3))
    for gt, rf in zip(got, exp):
        assert gt["status"] == rf.status == 0
        assert_same_format(gt, rf)


@pytest.mark.parametrize("which", ["all", "w", "mv"])
def test_adamw_in_place(which):
    n = 3 * 65536 + 1001
    w, m, v, g = _inputs(n, 1)
    gpu, ref, cbs, ocbs = _setup(w, m, v, 0)
    exp = oracle.adamw_step(ref[0], ocbs[0], ref[1], ocbs[1], ref[2], ocbs[2], g, _k(1))
    place = {"all": (True, True, True), "w": (True, False, False), "mv": (False, True, True)}[which]
    outs = [B.CompressedTensor(n, 0, like=x) if p else B.CompressedTensor(n, 0) for x, p in zip(gpu, place)]
    got = _step(gpu, cbs, g, 1, outs)
    for gt, rf in zip(got, exp):
        assert_same_format(gt, rf)


@pytest.mark.parametrize("in_place", [False, True])
def test_adamw_heavy_spill_and_special_values(in_place):
    """Moments whose exponents fit no model (every stream spills most of its
    rows), an activation-like weight, and zeros, subnormals, infinities and
    NaNs among the values (a negative second moment gives sqrt -> NaN)."""
    n = 3 * 32768 + 4321
    w = synth.gelu_sparse(n, seed=5)
    m = synth.random_bits(n, 8)
    v = synth.random_bits(n, 9)
    g = synth.normal(n, 0.1, 10)
    w[:6] = [0x0001, 0x8001, 0x7F80, 0xFF80, 0x7FC1, 0x0000]
    g[:6] = [0x8000, 0x0001, 0xFF80, 0x0000, 0x7FC0, 0x3F80]
    gpu, ref, cbs, ocbs = _setup(w, m, v, 2)
    exp = oracle.adamw_step(ref[0], ocbs[0], ref[1], ocbs[1], ref[2], ocbs[2], g, _k(5))
    assert exp[1].ovf_used > 0 and exp[2].ovf_used > 0
    outs = [B.CompressedTensor(n, 2, like=x) if in_place else B.CompressedTensor(n, 2) for x in gpu]
    got = _step(gpu, cbs, g, 5, outs)
    for gt, rf in zip(got, exp):
        assert gt["status"] == rf.status == 0
        assert_same_format(gt, rf)


def test_adamw_ten_steps_in_place():
    """Ten steps with a fresh gradient each, all three tensors updated in
    place with ping-pong overflow regions; compared with the oracle after
    every step."""
    n = 2 * 65536 + 123
    w, m, v, _ = _inputs(n, 2)
    gpu, ref, cbs, ocbs = _setup(w, m, v, 0)
    bufs = [[B.CompressedTensor(n, 0, like=x) for x in gpu] for _ in range(2)]
    cur = gpu
    for t in range(1, 11):
        g = synth.normal(n, 1e-4, 100 + t)
        nxt = bufs[t % 2]
        got = _step(cur, cbs, g, t, nxt)
        ref = list(oracle.adamw_step(ref[0], ocbs[0], ref[1], ocbs[1], ref[2], ocbs[2], g, _k(t)))
        for gt, rf in zip(got, ref):
            assert gt["status"] == rf.status == 0
            assert_same_format(gt, rf)
        cur = nxt


EDGES = [dict(lr=0.0), dict(lr=-1e-3), dict(beta1=0.0), dict(beta2=0.0), dict(beta1=0.9999999, beta2=0.9999999),
         dict(eps=1e-30), dict(weight_decay=0.0), dict(weight_decay=1e3), dict(t=1), dict(t=10 ** 6)]


@pytest.mark.parametrize("edge", EDGES, ids=lambda e: ",".join("%s=%g" % kv for kv in e.items()))
@pytest.mark.parametrize("in_place", [False, True])
def test_adamw_hyperparameter_edge_cases(edge, in_place):
    """Hyperparameters at the edges of what the ABI accepts: a zero or
    negative learning rate, beta1 or beta2 zero or just below one, a tiny eps,
    no or a large weight decay, the first step and a step far enough that the
    bias corrections round to one.  The step constants come from the same
    hyperparameters on both sides; every region of the three new tensors must
    equal the oracle's."""
    hp = dict(HP, t=3)
    hp.update(edge)
    n = 3 * 65536 - 555
    w, m, v, g = _inputs(n, 7)
    gpu, ref, cbs, ocbs = _setup(w, m, v, 0)
    k = oracle.adamw_constants(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], hp["t"])
    exp = oracle.adamw_step(ref[0], ocbs[0], ref[1], ocbs[1], ref[2], ocbs[2], g, k)
    outs = [B.CompressedTensor(n, 0, like=x) if in_place else B.CompressedTensor(n, 0) for x in gpu]
    B.lct_adamw_step_fused(gpu[0], cbs[0], gpu[1], cbs[1], gpu[2], cbs[2], to_device(g), hp["lr"], hp["beta1"],
                           hp["beta2"], hp["eps"], hp["weight_decay"], hp["t"], *outs)
    torch.cuda.synchronize()
    for o, rf in zip(outs, exp):
        gt = o.to_host()
        assert gt["status"] == rf.status == 0
        assert_same_format(gt, rf)
