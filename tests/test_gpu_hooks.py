"""GPU checks of the two pieces built on the codec for training: saved
activations kept compressed between forward and backward (gradients must be
bit for bit those of the uncompressed run), and a linear layer whose weight
is decoded tile by tile from its compressed form."""
import numpy as np
import pytest
import torch

from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth
from lossless_bf16_tensor_gb300.activations import compressed_activations
from lossless_bf16_tensor_gb300.matmul import compressed_linear

from gpu_helpers import to_device

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy()


def _mlp_grads(x, w1, w2, hook=None):
    x = x.clone().requires_grad_(True)
    a, b = w1.clone().requires_grad_(True), w2.clone().requires_grad_(True)
    if hook is None:
        y = torch.nn.functional.gelu(x @ a.t()) @ b.t()
    else:
        with hook:
            y = torch.nn.functional.gelu(x @ a.t()) @ b.t()
    (y.float() ** 2).sum().backward()
    return [_bits(t) for t in (y, x.grad, a.grad, b.grad)]


def _mlp_inputs(seed=0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = (torch.randn(2048, 1024, generator=g) * 0.5).to(torch.bfloat16).cuda()
    w1 = (torch.randn(4096, 1024, generator=g) * 0.02).to(torch.bfloat16).cuda()
    w2 = (torch.randn(1024, 4096, generator=g) * 0.02).to(torch.bfloat16).cuda()
    return x, w1, w2


def test_compressed_activations_give_identical_gradients():
    x, w1, w2 = _mlp_inputs()
    ref = _mlp_grads(x, w1, w2)
    cb = B.lct_codebook_build_zero_atom(0, 0.5, 0.0, 0.0)
    hook = compressed_activations(cb, level="CLEAN")
    got = _mlp_grads(x, w1, w2, hook)
    for r, g in zip(ref, got):
        assert np.array_equal(r, g)
    assert hook.stats["compressed"] >= 2 and hook.stats["fallback"] == 0
    assert hook.stats["stored_bytes"] < 0.8 * hook.stats["raw_bytes"]


def test_compressed_activations_fall_back_when_overflow_does_not_fit():
    """Activations whose exponents fit no model spill far beyond a tiny
    overflow allowance: those tensors keep their BF16 original and the
    gradients are still exact."""
    x, w1, w2 = _mlp_inputs(1)
    bits = synth.random_bits(x.numel(), 3)
    bits[(bits & 0x7F80) == 0x7F80] &= 0xBFFF          # no infinities or NaNs
    x = to_device(bits).view(torch.bfloat16).reshape(x.shape)
    ref = _mlp_grads(x, w1, w2)
    cb = B.lct_codebook_build(0, 0.5, 0.0)
    hook = compressed_activations(cb, level="CLEAN", ovf_frac=0.001, max_pending=1)
    got = _mlp_grads(x, w1, w2, hook)
    for r, g in zip(ref, got):
        assert np.array_equal(r, g)
    assert hook.stats["fallback"] >= 1


@pytest.mark.parametrize("tile_blocks", [1, 4, 16])
def test_compressed_linear_matches_dense_tiles(tile_blocks):
    """y = x W^T with W [4096, 1024] decoded 16 rows per block: equal, bit for
    bit, to cuBLAS on the same dense row tiles, and close to the one-shot
    dense product."""
    out_f, in_f = 4096, 1024
    w = synth.normal(out_f * in_f, 0.02, 11)
    x = to_device(synth.normal(512 * in_f, 1.0, 12)).view(torch.bfloat16).reshape(512, in_f)
    cb = B.lct_codebook_build(0, 0.02)
    ct = B.CompressedTensor(w.size, 0)
    B.lct_encode(to_device(w), cb, ct)
    wd = to_device(w).view(torch.bfloat16).reshape(out_f, in_f)
    y = compressed_linear(x, ct, cb, out_f, in_f, tile_blocks=tile_blocks)
    torch.cuda.synchronize()
    rows = tile_blocks * 65536 // in_f
    ref = torch.cat([(wd[r:r + rows] @ x.t()) for r in range(0, out_f, rows)], 0).t()
    assert np.array_equal(_bits(y), _bits(ref))
    full = x @ wd.t()
    assert torch.allclose(y.float(), full.float(), rtol=1e-2, atol=1e-2)
    assert ct.state().status == 0


def test_compressed_linear_default_tile():
    """Without a tile size the weight is decoded one wave of decode CTAs at a
    time (here all 64 blocks at once): bit for bit the dense product on the
    whole weight."""
    out_f, in_f = 4096, 1024
    w = synth.normal(out_f * in_f, 0.02, 13)
    x = to_device(synth.normal(256 * in_f, 1.0, 14)).view(torch.bfloat16).reshape(256, in_f)
    cb = B.lct_codebook_build(0, 0.02)
    ct = B.CompressedTensor(w.size, 0)
    B.lct_encode(to_device(w), cb, ct)
    wd = to_device(w).view(torch.bfloat16).reshape(out_f, in_f)
    y = compressed_linear(x, ct, cb, out_f, in_f)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y), _bits((wd @ x.t()).t()))
