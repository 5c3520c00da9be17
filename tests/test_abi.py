"""C-ABI checks that need no GPU: the library loads and exports every entry
point its headers declare, the host-side codebook builder reproduces the
oracle's tables, region sizes follow the format, and host-detectable argument
errors come back as status codes without touching the device."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MODELS = [(0, 0.02, 0.0), (0, 1.0, 0.0), (0, 1e-3, 0.0), (0, 3e-30, 0.0), (0, 1e20, 0.0),
          (1, 0.01, 0.0), (1, 3e-5, 0.0), (1, 7.0, 0.0), (2, 1e-3, 3.0), (2, 0.5, 1.5), (2, 1e-6, 0.7),
          (2, 2.0, 12.0)]


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"^lct_status\s+(lct_\w+)\s*\(", text, flags=re.M))
    return names


def test_library_exports_every_declared_entry_point(lct_lib):
    names = declared_functions()
    assert {"lct_codebook_build", "lct_encode", "lct_decode", "lct_sgd_step_fused",
            "lct_compressed_size"} <= names
    lib = lct_lib.library()
    for n in names:
        assert hasattr(lib, n), n


@pytest.mark.parametrize("model,scale,shape", MODELS)
def test_codebook_matches_oracle(lct_lib, orc, model, scale, shape):
    cb = lct_lib.lct_codebook_build(model, scale, shape)
    ref = orc.codebook_build(model, scale, shape)
    assert bytes(cb.len) == bytes(ref.len)
    assert list(cb.code) == [int(c) for c in ref.code]
    assert cb.esc_len == ref.esc_len and cb.esc_code == ref.esc_code
    assert cb.nsym == ref.k and cb.median_exp == ref.median_exp
    for v in range(256):
        assert cb.dec[v] & 0x1FF == ref.lut_sym[v]
        assert cb.dec[v] >> 12 == ref.lut_len[v]


def test_codebook_rejects_bad_parameters(lct_lib):
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook()
    for args in [(0, 0.0, 0.0), (1, -1.0, 0.0), (2, 1.0, 0.0), (0, float("inf"), 0.0), (3, 1.0, 1.0),
                 (2, 1.0, float("nan")), (0, float("nan"), 0.0)]:
        assert lib.lct_codebook_build(args[0], args[1], args[2], ctypes.byref(cb)) == lct_lib.LCT_ERR_INVALID_ARG
    assert lib.lct_codebook_build(0, 1.0, 0.0, None) == lct_lib.LCT_ERR_INVALID_ARG


@pytest.mark.parametrize("n", [0, 1, 255, 65536, 65537, 162_000_000, 1 << 26])
@pytest.mark.parametrize("level", [0, 1, 2])
def test_region_sizes(lct_lib, orc, n, level):
    block, words = orc.geometry(level)
    nb = -(-n // block)
    s = lct_lib.lct_compressed_size(n, level)
    assert (s.block, s.slot_words, s.nblocks) == (block, words, nb)
    assert s.sf_bytes == n and s.slot_bytes == nb * words * 256 * 4
    assert s.marker_bytes == nb * 512 and s.blk_off_bytes == 8 * (nb + 1)
    assert s.fixed_bytes == 64 + s.sf_bytes + s.slot_bytes + s.marker_bytes + s.blk_off_bytes
    assert s.worst_ovf_bytes == n and s.work_bytes == 8 * nb


def test_clean_all_in_ratio(lct_lib):
    """All-in ratio of a CLEAN tensor with no spill: 2n over the fixed bytes
    (slots, markers and offsets included), just under the 1.4382x payload bound."""
    n = 1 << 24
    s = lct_lib.lct_compressed_size(n, 0)
    assert abs(2 * n / s.fixed_bytes - 1.4301) < 5e-4


def test_sizes_reject_bad_arguments(lct_lib):
    lib = lct_lib.library()
    out = lct_lib.lct_sizes()
    assert lib.lct_compressed_size(10, 3, None, None, ctypes.byref(out)) == lct_lib.LCT_ERR_INVALID_ARG
    assert lib.lct_compressed_size((1 << 40) + 1, 0, None, None, ctypes.byref(out)) == lct_lib.LCT_ERR_INVALID_ARG
    assert lib.lct_compressed_size(10, 0, None, None, None) == lct_lib.LCT_ERR_INVALID_ARG


def _fake_tensor(lct_lib, n=1000, level=0, base=0x10000000):
    t = lct_lib.lct_tensor()
    t.n, t.level = n, level
    t.d_header, t.d_sf, t.d_slots = base, base + 0x1000, base + 0x100000
    t.d_markers, t.d_blk_off, t.d_ovf = base + 0x200000, base + 0x300000, base + 0x400000
    t.ovf_cap, t.d_work = n, base + 0x500000
    return t


def test_host_argument_errors_never_reach_the_device(lct_lib):
    """Each call below fails a host check, so no CUDA call is made (this
    machine has no GPU; reaching the device would give LCT_ERR_CUDA)."""
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook_build(0, 0.02)
    bad_cb = lct_lib.lct_codebook_build(0, 0.02)
    bad_cb.len[120] = 9
    x = 0x20000000
    E = lct_lib.LCT_ERR_INVALID_ARG

    def enc(t, c=cb, xp=x):
        return lib.lct_encode(xp, ctypes.byref(c), ctypes.byref(t), None)

    t = _fake_tensor(lct_lib)
    assert enc(t, c=bad_cb) == E                        # malformed codebook
    assert lib.lct_encode(x, None, ctypes.byref(t), None) == E
    assert enc(t, xp=None) == E                         # NULL input
    assert enc(t, xp=x + 2) == E                        # misaligned input
    for field in ("d_header", "d_sf", "d_slots", "d_markers", "d_blk_off", "d_work"):
        u = _fake_tensor(lct_lib)
        setattr(u, field, None)
        assert enc(u) == E, field
        setattr(u, field, getattr(_fake_tensor(lct_lib), field) + 4)
        assert enc(u) == E, field
    u = _fake_tensor(lct_lib)
    u.level = 7
    assert enc(u) == E
    u = _fake_tensor(lct_lib)
    u.d_ovf = u.d_slots                                # overlapping regions
    assert enc(u) == E
    u = _fake_tensor(lct_lib)
    assert enc(u, xp=u.d_sf) == E                      # input overlaps the output
    # decode
    y = 0x30000000
    assert lib.lct_decode(ctypes.byref(t), ctypes.byref(bad_cb), y, None) == E
    assert lib.lct_decode(ctypes.byref(t), ctypes.byref(cb), y + 8, None) == E
    assert lib.lct_decode(ctypes.byref(t), ctypes.byref(cb), t.d_sf, None) == E
    # sgd
    w, m, o = _fake_tensor(lct_lib), _fake_tensor(lct_lib, base=0x40000000), _fake_tensor(lct_lib, base=0x50000000)

    def sgd(w, m, o):
        return lib.lct_sgd_step_fused(ctypes.byref(w), ctypes.byref(cb), ctypes.byref(m), ctypes.byref(cb),
                                      ctypes.c_float(1e-3), ctypes.byref(o), None)

    m2 = _fake_tensor(lct_lib, n=999, base=0x40000000)
    assert sgd(w, m2, o) == E                           # n mismatch
    m3 = _fake_tensor(lct_lib, level=1, base=0x40000000)
    assert sgd(w, m3, o) == lct_lib.LCT_ERR_UNSUPPORTED  # level mismatch
    o2 = _fake_tensor(lct_lib, base=0x50000000)
    o2.d_ovf = w.d_ovf                                  # shares W_in's overflow
    assert sgd(w, m, o2) == E
    o3 = _fake_tensor(lct_lib, base=0x10000000)          # fully aliases W_in, overflow included
    assert sgd(w, m, o3) == E
    o4 = _fake_tensor(lct_lib, base=0x40000000)          # writes into M
    assert sgd(w, m, o4) == E
    # the debug hook checks its arguments too
    assert lib.lct_debug_wait_timeout(None, 0x10000000, 1000, None) == E
    assert lib.lct_debug_wait_timeout(0x10000000, 0x10000000 + 4, 1000, None) == E
    assert lib.lct_debug_wait_timeout(0x10000000, 0x10000010, 0, None) == E


def test_momentum_host_argument_errors_never_reach_the_device(lct_lib):
    """Host checks of lct_sgd_momentum_step_fused: sizes, levels, gradient
    pointer and the aliasing rules between the two inputs, the two outputs
    and the gradient (no CUDA call is made on any of these)."""
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook_build(0, 0.02)
    E = lct_lib.LCT_ERR_INVALID_ARG
    g = 0x60000000

    def mom(w, m, ow, om, gp=g, c=cb):
        return lib.lct_sgd_momentum_step_fused(ctypes.byref(w), ctypes.byref(c), ctypes.byref(m), ctypes.byref(c),
                                               gp, ctypes.c_float(1e-3), ctypes.c_float(0.9), ctypes.byref(ow),
                                               ctypes.byref(om), None)

    def four():
        return (_fake_tensor(lct_lib), _fake_tensor(lct_lib, base=0x40000000),
                _fake_tensor(lct_lib, base=0x50000000), _fake_tensor(lct_lib, base=0x70000000))

    w, m, ow, om = four()
    bad_cb = lct_lib.lct_codebook_build(0, 0.02)
    bad_cb.len[3] = 9
    assert mom(w, m, ow, om, c=bad_cb) == E             # malformed codebook
    assert mom(w, m, ow, om, gp=None) == E               # NULL gradient
    assert mom(w, m, ow, om, gp=g + 2) == E              # misaligned gradient
    assert mom(w, m, ow, om, gp=ow.d_sf) == E            # gradient overlaps an output
    m2 = _fake_tensor(lct_lib, n=999, base=0x40000000)
    assert mom(w, m2, ow, om) == E                       # n mismatch
    om2 = _fake_tensor(lct_lib, level=1, base=0x70000000)
    assert mom(w, m, ow, om2) == lct_lib.LCT_ERR_UNSUPPORTED
    w, m, ow, om = four()
    om.d_ovf = ow.d_ovf                                  # the outputs share an overflow region
    assert mom(w, m, ow, om) == E
    w, m, ow, om = four()
    ow2 = _fake_tensor(lct_lib, base=0x40000000)         # W' written into M
    assert mom(w, m, ow2, om) == E
    om3 = _fake_tensor(lct_lib, base=0x10000000)         # M' written into W
    assert mom(w, m, ow, om3) == E
    ow4 = _fake_tensor(lct_lib, base=0x10000000)         # W' fully aliases W_in, overflow included
    assert mom(w, m, ow4, om) == E
    ow5 = _fake_tensor(lct_lib, base=0x50000000)
    ow5.d_sf = w.d_sf + 16                               # partly overlaps W_in's bytes
    assert mom(w, m, ow5, om) == E


ZERO_ATOM_MODELS = [(0, 1.0, 0.0, 0.3), (0, 0.02, 0.0, 0.0), (1, 0.01, 0.0, 0.5), (2, 1e-3, 3.0, 0.1),
                    (0, 1.0, 0.0, 0.95)]


@pytest.mark.parametrize("model,scale,shape,zf", ZERO_ATOM_MODELS)
def test_zero_atom_codebook_matches_oracle(lct_lib, orc, model, scale, shape, zf):
    cb = lct_lib.lct_codebook_build_zero_atom(model, scale, shape, zf)
    ref = orc.codebook_build_zero_atom(model, scale, shape, zf)
    assert cb.zero_atom == 1 and ref.zero_atom == 1 and cb.zero_frac == zf
    assert bytes(cb.len) == bytes(ref.len)
    assert list(cb.code) == [int(c) for c in ref.code]
    assert cb.esc_len == ref.esc_len and cb.esc_code == ref.esc_code
    assert cb.nsym == ref.k and cb.median_exp == ref.median_exp
    for v in range(256):
        assert cb.dec[v] & 0x1FF == ref.lut_sym[v] and cb.dec[v] >> 12 == ref.lut_len[v]
    # the flag is part of the codebook's identity: the plain model's codes
    # with zero_frac = 0 hash differently
    if zf == 0.0:
        plain = lct_lib.lct_codebook_build(model, scale, shape)
        assert bytes(plain.len) == bytes(cb.len) and plain.hash != cb.hash


def test_zero_atom_rejects_bad_parameters(lct_lib):
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook()
    E = lct_lib.LCT_ERR_INVALID_ARG
    for zf in (-0.1, 1.0, 1.5, float("nan")):
        assert lib.lct_codebook_build_zero_atom(0, 1.0, 0.0, zf, ctypes.byref(cb)) == E
    assert lib.lct_codebook_build_zero_atom(0, -1.0, 0.0, 0.3, ctypes.byref(cb)) == E
    assert lib.lct_codebook_build_zero_atom(0, 1.0, 0.0, 0.3, None) == E
    # a codebook whose flag is neither 0 nor 1 is refused by every entry point
    good = lct_lib.lct_codebook_build_zero_atom(0, 1.0, 0.0, 0.3)
    good.zero_atom = 2
    t = _fake_tensor(lct_lib)
    assert lib.lct_encode(0x20000000, ctypes.byref(good), ctypes.byref(t), None) == E


def test_decode_blocks_host_checks(lct_lib):
    """lct_decode_blocks refuses ranges past the last block and output that
    overlaps the tensor; an empty range enqueues nothing and succeeds."""
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook_build(0, 0.02)
    E = lct_lib.LCT_ERR_INVALID_ARG
    t = _fake_tensor(lct_lib, n=3 * 65536 + 5)          # 4 blocks
    y = 0x60000000

    def dec(first, count, yp=y):
        return lib.lct_decode_blocks(ctypes.byref(t), ctypes.byref(cb), first, count, yp, None)

    assert dec(0, 5) == E and dec(4, 1) == E and dec(5, 0) == E and dec(2, (1 << 64) - 1) == E
    assert dec(1, 1, yp=y + 2) == E                      # misaligned
    assert dec(1, 1, yp=None) == E
    assert dec(1, 1, yp=t.d_sf) == E                     # overlaps the tensor
    assert dec(4, 0) == lct_lib.LCT_OK and dec(0, 0) == lct_lib.LCT_OK


def test_adamw_host_argument_errors_never_reach_the_device(lct_lib):
    """Host checks of lct_adamw_step_fused: parameters, sizes, levels, the
    gradient pointer and the aliasing rules (no CUDA call is made)."""
    lib = lct_lib.library()
    cb = lct_lib.lct_codebook_build(0, 0.02)
    E = lct_lib.LCT_ERR_INVALID_ARG
    g = 0x6A000000
    bases = [0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000, 0x70000000]

    def six():
        return [_fake_tensor(lct_lib, base=x) for x in bases]

    def adam(ts, p=None, gp=g):
        p = p or lct_lib.lct_adamw_params(1e-3, 0.9, 0.999, 1e-8, 0.01, 1)
        w, m, v, ow, om, ov = ts
        return lib.lct_adamw_step_fused(ctypes.byref(w), ctypes.byref(cb), ctypes.byref(m), ctypes.byref(cb),
                                        ctypes.byref(v), ctypes.byref(cb), gp, ctypes.byref(p), ctypes.byref(ow),
                                        ctypes.byref(om), ctypes.byref(ov), None)

    P = lct_lib.lct_adamw_params
    for bad in (P(1e-3, 0.9, 0.999, 1e-8, 0.0, 0), P(1e-3, 1.0, 0.999, 1e-8, 0.0, 1),
                P(1e-3, 0.9, -0.1, 1e-8, 0.0, 1), P(1e-3, 0.9, 0.999, 0.0, 0.0, 1),
                P(float("nan"), 0.9, 0.999, 1e-8, 0.0, 1), P(1e-3, 0.9, 0.999, 1e-8, float("inf"), 1)):
        assert adam(six(), p=bad) == E
    assert adam(six(), gp=None) == E
    assert adam(six(), gp=g + 4) == E
    ts = six()
    assert adam(ts, gp=ts[3].d_sf) == E                   # gradient overlaps an output
    ts = six()
    ts[1] = _fake_tensor(lct_lib, n=999, base=bases[1])
    assert adam(ts) == E                                  # n mismatch
    ts = six()
    ts[5] = _fake_tensor(lct_lib, level=2, base=bases[5])
    assert adam(ts) == lct_lib.LCT_ERR_UNSUPPORTED
    ts = six()
    ts[4] = _fake_tensor(lct_lib, base=bases[2])          # M' written into V
    assert adam(ts) == E
    ts = six()
    ts[3].d_ovf = ts[4].d_ovf                              # two outputs share an overflow region
    assert adam(ts) == E
    ts = six()
    ts[3] = _fake_tensor(lct_lib, base=bases[0])          # W' fully aliases W, overflow included
    assert adam(ts) == E


@pytest.mark.parametrize("level,per_value", [(0, 3.3985), (1, 3.5157), (2, 3.6407)])
def test_roofline_bytes_are_the_format_bytes(lct_lib, level, per_value):
    """bench.py's roofline numerator: an encode or decode of n values moves the
    2n uncompressed bytes plus the compressed form (sign-fraction bytes, full
    fixed slots, markers, block offsets, used overflow), 3.3985 / 3.5157 /
    3.6407 bytes per value for CLEAN / MEDIUM / HIGH before overflow."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    n = 1 << 24
    sizes = lct_lib.lct_compressed_size(n, level)
    one = bench.algorithmic_bytes(sizes, 0)
    assert abs((2 * n + one) / n - per_value) < 3e-4  # the figures are rounded to 4 places
    assert bench.algorithmic_bytes(sizes, 12345) == one + 12345
    # the fused SGD reads two compressed tensors and writes one
    assert 3 * one / n == pytest.approx(3 * (per_value - 2), abs=9e-4)
