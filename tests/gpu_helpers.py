"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare every region of the format with the CPU oracle, element by
element (integer data: bit-exact)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

MODEL_ID = {"gaussian": 0, "laplace": 1, "powerlaw": 2}
LEVEL_ID = {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}


def to_device(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


def from_device(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def codebooks(model: int, scale: float, shape: float = 0.0):
    return B.lct_codebook_build(model, scale, shape), oracle.codebook_build(model, scale, shape)


def gpu_encode(x: np.ndarray, cb, level: int, ovf_cap=None) -> B.CompressedTensor:
    ct = B.CompressedTensor(x.size, level, ovf_cap=ovf_cap)
    B.lct_encode(to_device(x), cb, ct)
    torch.cuda.synchronize()
    return ct


def gpu_decode(ct: B.CompressedTensor, cb) -> np.ndarray:
    y = torch.empty(ct.n, dtype=torch.int16, device="cuda")
    B.lct_decode(ct, cb, y)
    torch.cuda.synchronize()
    return from_device(y)


def assert_same_format(gpu: dict, ref: oracle.Compressed, blocks=None):
    """Bit-exact comparison of a GPU tensor (to_host() dict) with the oracle's
    encoding; `blocks` restricts the comparison to those block indices."""
    assert gpu["delta"] == ref.delta, ("delta", gpu["delta"], ref.delta)
    assert gpu["ovf_used"] == ref.ovf_used, ("ovf_used", gpu["ovf_used"], ref.ovf_used)
    assert np.array_equal(gpu["blk_off"], ref.blk_off)
    W, Bk = ref.slot_words, ref.block
    if blocks is None:
        assert np.array_equal(gpu["sf"], ref.sf)
        _eq(gpu["slots"], ref.slots, "slots")
        _eq(gpu["markers"], ref.markers, "markers")
        used = min(ref.ovf_used, ref.ovf.size)
        fit = [b for b in range(ref.nblocks) if ref.blk_off[b + 1] <= ref.ovf.size]
        hi = int(ref.blk_off[fit[-1] + 1]) if fit else 0
        _eq(gpu["ovf"][:hi], ref.ovf[:hi], "overflow")
        assert used >= hi
    else:
        for b in blocks:
            s = slice(b * Bk, min((b + 1) * Bk, ref.n))
            assert np.array_equal(gpu["sf"][s], ref.sf[s]), ("sf", b)
            _eq(gpu["slots"][b * W * 256:(b + 1) * W * 256], ref.slots[b * W * 256:(b + 1) * W * 256], "slots %d" % b)
            _eq(gpu["markers"][b * 256:(b + 1) * 256], ref.markers[b * 256:(b + 1) * 256], "markers %d" % b)
            o0, o1 = int(ref.blk_off[b]), int(ref.blk_off[b + 1])
            _eq(gpu["ovf"][o0:o1], ref.ovf[o0:o1], "overflow %d" % b)


def _eq(a, b, what):
    if not np.array_equal(a, b):
        bad = np.nonzero(a != b)[0]
        raise AssertionError("%s differs at %d places, first %d: gpu %r oracle %r" % (
            what, bad.size, bad[0], a[bad[0]], b[bad[0]]))


def workload(name: str, n=None):
    w = synth.WORKLOADS[name]
    x = synth.generate(name, n)
    return x, MODEL_ID[w["model"]], w["scale"], w["shape"], LEVEL_ID[w["level"]]
