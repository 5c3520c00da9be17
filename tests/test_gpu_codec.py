"""GPU parity of the encode/decode path against the CPU oracle, through the C
ABI: shift, sign-fraction bytes, slot words, markers, block offsets, overflow
bytes and decoded values must all be identical (0 ULP, bit for bit)."""
import numpy as np
import pytest
import torch

import oracle
from lossless_bf16_tensor_gb300 import binding as B
from lossless_bf16_tensor_gb300 import synth

from gpu_helpers import (assert_same_format, codebooks, from_device, gpu_decode, gpu_encode, to_device,
                         workload)

pytestmark = pytest.mark.gpu


def _roundtrip(x, model, scale, shape, level, ovf_cap=None):
    cb, ocb = codebooks(model, scale, shape)
    ct = gpu_encode(x, cb, level, ovf_cap=ovf_cap)
    ref = oracle.encode(x, ocb, level, ovf_cap=ovf_cap)
    got = ct.to_host()
    assert got["status"] == ref.status
    assert_same_format(got, ref)
    if ref.status == oracle.OK:
        y = gpu_decode(ct, cb)
        assert np.array_equal(y, x)
        assert ct.state().status == B.LCT_OK
    return ct, ref, cb, ocb


def test_one_clean_block_gaussian():
    """65,536 values ~ N(0, 0.02), Gaussian codebook, CLEAN: one block."""
    x, m, s, sh, lv = workload("gauss_block")
    ct, ref, cb, _ = _roundtrip(x, m, s, sh, lv)
    assert ref.delta == 0 and ref.ovf_used == 0
    st = ct.state()
    assert st.delta == 0 and st.ovf_used == 0


@pytest.mark.parametrize("level", [0, 1, 2])
@pytest.mark.parametrize("n", [1, 7, 8, 255, 256, 257, 4097, 32767, 32768, 32769, 65535, 65536, 65537,
                               3 * 65536 + 1234])
def test_ragged_sizes(level, n):
    x = synth.laplace(n, 0.01, seed=n)
    _roundtrip(x, 1, 0.01, 0.0, level)


@pytest.mark.parametrize("level", [0, 1, 2])
def test_every_bf16_pattern(level):
    """Zeros, subnormals, infinities and every NaN payload survive exactly."""
    x = synth.all_bf16_patterns()
    for model, scale, shape in [(0, 0.02, 0.0), (2, 1e-3, 3.0), (1, 1e10, 0.0)]:
        _roundtrip(x, model, scale, shape, level)


@pytest.mark.parametrize("name,n", [("heavy_64m", 5 * 32768 + 17), ("gelu_act", 6 * 32768 - 5)])
def test_spilling_workloads_small(name, n):
    x, m, s, sh, lv = workload(name, n)
    _, ref, _, _ = _roundtrip(x, m, s, sh, lv)
    if name == "gelu_act":
        assert ref.ovf_used > 0


def test_forced_spill_every_stream():
    """Every value escapes (exponents far from the codebook): each stream
    spills, offsets run over every block."""
    rng = np.random.default_rng(3)
    e = rng.integers(1, 40, size=3 * 65536 + 99).astype(np.uint16)
    x = (e << 7) | rng.integers(0, 128, size=e.size).astype(np.uint16)
    x[::2] |= 0x8000
    _, ref, _, _ = _roundtrip(x, 0, 1.0, 0.0, 0)
    assert ref.ovf_used > x.size // 2


def test_laplace_16m_full():
    x, m, s, sh, lv = workload("laplace_16m")
    _roundtrip(x, m, s, sh, lv)


def test_heavy_tail_64m_full():
    x, m, s, sh, lv = workload("heavy_64m")
    _roundtrip(x, m, s, sh, lv)


def test_gelu_activation_pow2_rounds():
    """[8, 4096, 3072] GELU activations with 30% zeros, scaled by 2^k for
    k = -4..4; the shift is re-estimated every round.  Full-size parity on
    three rounds; on all nine, the shift moves by k and the markers and
    overflow size do not move at all."""
    x0, m, s, sh, lv = workload("gelu_act")
    cb, ocb = codebooks(m, s, sh)
    markers0 = d0 = used0 = None
    for k in range(-4, 5):
        xk = synth.scale_pow2(x0, k)
        ct = gpu_encode(xk, cb, lv)
        got = ct.to_host()
        assert got["status"] == 0
        if k in (-4, 0, 4):
            assert_same_format(got, oracle.encode(xk, ocb, lv))
        if markers0 is None:
            markers0, d0, used0 = got["markers"].copy(), got["delta"] - k, got["ovf_used"]
        assert got["delta"] == d0 + k
        assert np.array_equal(got["markers"], markers0)
        assert got["ovf_used"] == used0
        assert np.array_equal(gpu_decode(ct, cb), xk)
        del ct


def test_decode_of_oracle_encoding():
    """The GPU decoder reads streams written by the oracle (not by the GPU)."""
    x, m, s, sh, lv = workload("heavy_64m", 4 * 32768 + 1000)
    cb, ocb = codebooks(0, 1.0, 0.0)
    ref = oracle.encode(x, ocb, 2, block=32768, slot_words=20)
    ct = gpu_encode(np.zeros_like(x), cb, 2)           # a valid header for this n
    torch.cuda.synchronize()
    r = ct.regions
    r["sf"].copy_(torch.from_numpy(ref.sf))
    r["slots"].copy_(torch.from_numpy(ref.slots.view(np.uint8)))
    r["markers"].copy_(torch.from_numpy(ref.markers.view(np.uint8)))
    r["blk_off"].copy_(torch.from_numpy(ref.blk_off.view(np.uint8)))
    r["ovf"][: ref.ovf_used].copy_(torch.from_numpy(ref.ovf[: ref.ovf_used]))
    hdr = r["header"].cpu().numpy().copy()
    hdr[20:24] = np.array([ref.delta], np.int32).view(np.uint8)
    r["header"].copy_(torch.from_numpy(hdr))
    assert np.array_equal(gpu_decode(ct, cb), x)


def test_empty_tensor():
    cb = B.lct_codebook_build(0, 0.02)
    ct = B.CompressedTensor(0, 0)
    B.lct_encode(torch.empty(0, dtype=torch.int16, device="cuda"), cb, ct)
    y = torch.empty(0, dtype=torch.int16, device="cuda")
    B.lct_decode(ct, cb, y)
    st = ct.state()
    assert st.status == 0 and st.ovf_used == 0


def test_overflow_capacity_is_latched():
    x, m, s, sh, lv = workload("gelu_act", 3 * 32768)
    cb, ocb = codebooks(m, s, sh)
    full = oracle.encode(x, ocb, lv)
    cap = int(full.blk_off[1]) + 3
    ct, ref, _, _ = _roundtrip(x, m, s, sh, lv, ovf_cap=cap)
    assert ref.status == oracle.CAPACITY
    st = ct.state()
    assert st.status == B.LCT_ERR_OVERFLOW_CAPACITY and st.ovf_used == full.ovf_used
    y = torch.empty(ct.n, dtype=torch.int16, device="cuda")
    B.lct_decode(ct, cb, y)
    assert ct.state().status == B.LCT_ERR_OVERFLOW_CAPACITY


def _encoded(n=3 * 65536 + 5):
    x = synth.laplace(n, 0.01, seed=9)
    cb = B.lct_codebook_build(1, 0.01)
    return x, cb, gpu_encode(x, cb, 0)


def test_corrupt_marker_is_latched_not_faulted():
    x, cb, ct = _encoded()
    mk = ct.regions["markers"].view(torch.int16)
    mk[300] = 1000                                 # beyond the stream's 256 symbols
    gpu_decode(ct, cb)
    assert ct.state().status == B.LCT_ERR_CORRUPT


def test_corrupt_slots_are_latched_not_faulted():
    """Garbage slot words decode without reading outside the slot image; an
    all-ones slot (every window reads as the longest code) overruns and is
    reported."""
    x, cb, ct = _encoded()
    g = torch.Generator(device="cpu").manual_seed(5)
    ct.regions["slots"].copy_(torch.randint(0, 256, (ct.regions["slots"].numel(),), generator=g,
                                            dtype=torch.uint8))
    gpu_decode(ct, cb)
    ct.state()
    x, cb, ct = _encoded()
    ct.regions["slots"].fill_(0xFF)
    gpu_decode(ct, cb)
    assert ct.state().status == B.LCT_ERR_CORRUPT


def test_bad_magic_and_wrong_codebook():
    x, cb, ct = _encoded()
    other = B.lct_codebook_build(0, 0.02)
    gpu_decode(ct, other)
    assert ct.state().status == B.LCT_ERR_CORRUPT
    x, cb, ct = _encoded()
    ct.regions["header"][0] = 0
    gpu_decode(ct, cb)
    assert ct.state().status == B.LCT_ERR_CORRUPT


def test_bounded_wait_runs_out():
    """A block waiting for a predecessor that never publishes gives up after
    the limit in every form of the wait (all predecessors at once, window by
    window, single thread) and latches LCT_ERR_TIMEOUT; the context stays
    usable."""
    hdr = torch.zeros(64, dtype=torch.uint8, device="cuda")
    work = torch.zeros(64, dtype=torch.uint8, device="cuda")
    B.lct_debug_wait_timeout(hdr, work, 2_000_000)
    torch.cuda.synchronize()
    assert int(hdr[24:28].cpu().numpy().view(np.uint32)[0]) == B.LCT_ERR_TIMEOUT
    x, cb, ct = _encoded(70000)
    assert np.array_equal(gpu_decode(ct, cb), x)


def test_async_on_side_stream():
    """Calls run on the stream given (here a non-default one)."""
    x = synth.laplace(2 * 65536 + 3, 0.01, seed=4)
    cb = B.lct_codebook_build(1, 0.01)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd = to_device(x)
        ct = B.CompressedTensor(x.size, 0)
        y = torch.empty(x.size, dtype=torch.int16, device="cuda")
        B.lct_encode(xd, cb, ct, stream=s)
        B.lct_decode(ct, cb, y, stream=s)
    s.synchronize()
    assert np.array_equal(from_device(y), x)


@pytest.mark.parametrize("level", [0, 2])
def test_decode_blocks_equals_full_decode(level):
    """Decoding any block range, the ragged last block included, gives the
    same values as the full decode of those positions."""
    x, m, s, sh, _ = workload("gelu_act", n=5 * 65536 + 1234)
    cb, ocb = codebooks(m, s, sh)
    ct = gpu_encode(x, cb, level)
    block = 65536 if level == 0 else 32768
    nb = ct.nblocks
    for first, count in [(0, 1), (1, 2), (nb - 1, 1), (0, nb), (nb - 3, 3)]:
        lo, hi = first * block, min(x.size, (first + count) * block)
        y = torch.empty(hi - lo, dtype=torch.int16, device="cuda")
        B.lct_decode_blocks(ct, cb, first, count, y)
        torch.cuda.synchronize()
        assert np.array_equal(from_device(y), x[lo:hi]), (first, count)
    assert ct.state().status == 0


def test_compressed_tensor_moves_through_host_memory():
    """A compressed tensor is self-describing (its header holds no pointer):
    copied to host memory and back into fresh device buffers, it decodes to
    the same values, and the fused SGD reads it like the original."""
    x, m, s, sh, lv = workload("heavy_64m", n=3 * 32768 + 555)
    cb, ocb = codebooks(m, s, sh)
    ct = gpu_encode(x, cb, lv)
    saved = ct.buffer.cpu()                      # checkpoint
    back = B.CompressedTensor(x.size, lv, zero_fill=False)
    assert back.buffer.numel() == saved.numel()
    back.buffer.copy_(saved)                     # resume into other device memory
    torch.cuda.synchronize()
    assert np.array_equal(gpu_decode(back, cb), x)
    assert_same_format(back.to_host(), oracle.encode(x, ocb, lv))


def test_more_than_two_to_the_32_values():
    """4,294,979,641 values (past 2^32, so every 32-bit element index would
    wrap): encode, decode checked in full on the device, fused SGD; blocks at
    the start, across the 2^32 boundary and at the ragged end compared with
    the oracle run on those blocks alone (blocks are independent given the
    shift).  Values tile a seeded 2^20-value Laplace draw."""
    n = (1 << 32) + 12345
    period = 1 << 20
    xb = synth.laplace(period, 0.01, seed=11)
    mb = synth.laplace(period, 1e-3, seed=12)
    reps = n // period + 1
    x = torch.from_numpy(xb.view(np.int16)).cuda().repeat(reps)[:n]
    m = torch.from_numpy(mb.view(np.int16)).cuda().repeat(reps)[:n]
    cb, ocb = codebooks(1, 0.01)
    cbm, ocbm = codebooks(1, 1e-3)
    X = B.CompressedTensor(n, 0)
    Mc = B.CompressedTensor(n, 0)
    B.lct_encode(x, cb, X)
    B.lct_encode(m, cbm, Mc)
    y = torch.empty_like(x)
    B.lct_decode(X, cb, y)
    Wn = B.CompressedTensor(n, 0)
    B.lct_sgd_step_fused(X, cb, Mc, cbm, float(np.float32(1e-3)), Wn)
    torch.cuda.synchronize()
    assert torch.equal(y, x)
    del y
    sx, sm_, sw = X.state(), Mc.state(), Wn.state()
    assert sx.status == sm_.status == sw.status == 0
    block, nb = 65536, X.nblocks
    hx, hm, hw = (t.regions for t in (X, Mc, Wn))
    for b in (0, (1 << 32) // block - 1, (1 << 32) // block, nb - 1):
        lo, hi = b * block, min(n, (b + 1) * block)
        idx = np.arange(lo, hi, dtype=np.int64) % period
        xs, ms = xb[idx], mb[idx]
        rx = oracle.encode(xs, ocb, 0, delta=sx.delta)
        rm = oracle.encode(ms, ocbm, 0, delta=sm_.delta)
        rw = oracle.sgd_step(rx, ocb, rm, ocbm, float(np.float32(1e-3)))
        for regs, ref in ((hx, rx), (hw, rw)):
            assert np.array_equal(regs["sf"][lo:hi].cpu().numpy(), ref.sf), b
            sl = regs["slots"].view(torch.int32)[b * 25 * 256:(b + 1) * 25 * 256].cpu().numpy().view(np.uint32)
            assert np.array_equal(sl, ref.slots), b
            mk = regs["markers"].view(torch.int16)[b * 256:(b + 1) * 256].cpu().numpy().view(np.uint16)
            assert np.array_equal(mk, ref.markers), b
            off = regs["blk_off"].view(torch.int64)[b:b + 2].cpu().numpy()
            assert off[1] - off[0] == ref.ovf_used, b


def test_package_level_usage():
    """The package-level calls a user starts from: build a codebook, encode,
    decode, fused SGD into a new tensor; checked against the oracle's SGD."""
    import lossless_bf16_tensor_gb300 as L
    torch.manual_seed(0)
    n = 4 * 65536
    w = (torch.randn(n, device="cuda") * 0.02).to(torch.bfloat16)
    m = (torch.randn(n, device="cuda") * 1e-3).to(torch.bfloat16)
    cb, cbm = L.lct_codebook_build("gaussian", 0.02), L.lct_codebook_build("gaussian", 1e-3)
    W, M, W2 = (L.CompressedTensor(n, "CLEAN") for _ in range(3))
    L.lct_encode(w.view(torch.int16), cb, W)
    L.lct_encode(m.view(torch.int16), cbm, M)
    assert 1.40 < W.compression_ratio() < 1.44
    y = torch.empty_like(w)
    L.lct_decode(W, cb, y.view(torch.int16))
    assert torch.equal(y, w)
    eta = float(np.float32(1e-3))
    L.lct_sgd_step_fused(W, cb, M, cbm, eta, W2)
    torch.cuda.synchronize()
    w_np, m_np = (t.view(torch.int16).cpu().numpy().view(np.uint16) for t in (w, m))
    ocb, ocbm = oracle.codebook_build(0, 0.02), oracle.codebook_build(0, 1e-3)
    ref = oracle.sgd_step(oracle.encode(w_np, ocb, 0), ocb, oracle.encode(m_np, ocbm, 0), ocbm, eta)
    assert W2.state().status == B.LCT_OK
    assert_same_format(W2.to_host(), ref)


def test_step_captured_in_a_cuda_graph():
    """The calls enqueue work only (no host synchronisation, no allocation),
    so a step of encode, decode and fused SGD can be captured in a CUDA graph
    and replayed on new inputs copied into the captured buffers; every replay
    matches the oracle."""
    n = 2 * 65536 + 4097
    cb, ocb = codebooks(1, 0.01, 0.0)
    cbm, ocbm = codebooks(1, 1e-3, 0.0)
    m = synth.laplace(n, 1e-3, seed=2)
    M = gpu_encode(m, cbm, 0)
    X, Wn = B.CompressedTensor(n, 0), B.CompressedTensor(n, 0)
    x = torch.empty(n, dtype=torch.int16, device="cuda")
    y = torch.empty_like(x)
    eta = float(np.float32(1e-3))
    s = torch.cuda.Stream()
    x.copy_(to_device(synth.laplace(n, 0.01, seed=40)))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):  # one step outside the capture (loads the kernels)
        B.lct_encode(x, cb, X, s)
        B.lct_decode(X, cb, y, s)
        B.lct_sgd_step_fused(X, cb, M, cbm, eta, Wn, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.lct_encode(x, cb, X, s)
        B.lct_decode(X, cb, y, s)
        B.lct_sgd_step_fused(X, cb, M, cbm, eta, Wn, s)
    ref_m = oracle.encode(m, ocbm, 0)
    for seed in (41, 42, 43):
        xh = synth.laplace(n, 0.01, seed=seed)
        x.copy_(to_device(xh))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        ref = oracle.encode(xh, ocb, 0)
        assert_same_format(X.to_host(), ref)
        assert np.array_equal(from_device(y), xh)
        assert_same_format(Wn.to_host(), oracle.sgd_step(ref, ocb, ref_m, ocbm, eta))
