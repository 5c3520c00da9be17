"""Encode and decode on both sides of the small-grid switch.

[EXP] "Compressing is easy": each block of 256 streams is encoded and decoded
on its own, so the result cannot depend on how many blocks a launch has.  The
library picks its kernels by grid size all the same: a grid of at most two
blocks per SM takes the encoder with 32-row input chunks and the decoder that
keeps slot words in registers; a larger grid takes the four-CTA kernels.
These tests encode tensors of exactly 2 * SMs and 2 * SMs + 1 blocks (the last
one ragged), with spilling blocks among ones that spill nothing, and compare
every region with the oracle's encoding and the decoded values with the input."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import assert_same_format, codebooks, gpu_decode, gpu_encode

pytestmark = pytest.mark.gpu

BLOCK = {0: 65536, 1: 32768}


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _tensor(nblocks, level, seed):
    """Laplace(0.01) values over `nblocks` blocks, the last one 777 values
    short, with random bit patterns written into the first 20,000 values of
    three blocks (those spill; most others spill nothing)."""
    bk = BLOCK[level]
    n = nblocks * bk - 777
    x = synth.laplace(n, 0.01, seed=seed)
    for i, b in enumerate((0, nblocks // 2, nblocks - 1)):
        at = b * bk
        m = min(20000, n - at)
        x[at:at + m] = synth.random_bits(m, seed=seed + 10 + i)
    return x


@pytest.mark.parametrize("extra", [0, 1])
@pytest.mark.parametrize("level", [0, 1])
def test_encode_decode_at_the_small_grid_boundary(level, extra):
    nblocks = 2 * _sms() + extra
    x = _tensor(nblocks, level, seed=31 + 2 * level + extra)
    cb, ocb = codebooks(1, 0.01)
    ct = gpu_encode(x, cb, level)
    ref = oracle.encode(x, ocb, level)
    assert ref.nblocks == nblocks
    spilling = set(np.nonzero(np.diff(ref.blk_off))[0].tolist())
    assert {0, nblocks // 2, nblocks - 1} <= spilling
    got = ct.to_host()
    assert got["status"] == 0
    assert_same_format(got, ref)
    assert np.array_equal(gpu_decode(ct, cb), x)
