"""CPU oracle for the LCT BF16 exponent-Huffman codec -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does: it has
no CPU fallback, and nothing here is shared with it.

The arithmetic lives in ``lct_oracle.c`` (plain single-threaded C, built with
floating-point contraction off); this module only builds it, loads it with
ctypes and moves numpy arrays in and out.  See ``lct_oracle.h`` for what each
function follows on the pages and what pins it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lct_oracle.c")
_HDR = os.path.join(_HERE, "lct_oracle.h")
_LIB = os.path.join(_HERE, "liblct_oracle.so")

GAUSSIAN, LAPLACE, POWERLAW = 0, 1, 2
CLEAN, MEDIUM, HIGH = 0, 1, 2
ESC = 256
OK, BAD_ARG, CAPACITY, CORRUPT = 0, 1, 3, 4
STREAMS = 256


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library beside its source."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB)
    return _LIB


class Codebook(ctypes.Structure):
    _fields_ = [
        ("weight", ctypes.c_uint64 * 256),
        ("len", ctypes.c_uint8 * 256),
        ("code", ctypes.c_uint16 * 256),
        ("esc_len", ctypes.c_uint8),
        ("pad0", ctypes.c_uint8),
        ("esc_code", ctypes.c_uint16),
        ("k", ctypes.c_int32),
        ("median_exp", ctypes.c_int32),
        ("lut_sym", ctypes.c_uint16 * 256),
        ("lut_len", ctypes.c_uint8 * 256),
        ("zero_atom", ctypes.c_int32),
    ]

    def lengths(self) -> np.ndarray:
        return np.frombuffer(bytes(self.len), dtype=np.uint8).copy()

    def codes(self) -> np.ndarray:
        return np.frombuffer(bytes(self.code), dtype=np.uint16).copy()


class _Tensor(ctypes.Structure):
    _fields_ = [
        ("n", ctypes.c_uint64),
        ("block", ctypes.c_uint32),
        ("slot_words", ctypes.c_uint32),
        ("delta", ctypes.c_int32),
        ("pad0", ctypes.c_uint32),
        ("sf", ctypes.c_void_p),
        ("slots", ctypes.c_void_p),
        ("markers", ctypes.c_void_p),
        ("blk_off", ctypes.c_void_p),
        ("ovf", ctypes.c_void_p),
        ("ovf_cap", ctypes.c_uint64),
        ("ovf_used", ctypes.c_uint64),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        l = ctypes.CDLL(build())
        P = ctypes.c_void_p
        l.orc_level_geometry.argtypes = [ctypes.c_int, P, P]
        l.orc_model_pmf.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, P]
        l.orc_weights_from_pmf.argtypes = [P, P]
        l.orc_weights_from_pmf.restype = None
        l.orc_package_merge.argtypes = [ctypes.c_int, P, P, ctypes.c_int, P]
        l.orc_codebook_from_weights.argtypes = [P, P]
        l.orc_codebook_build.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, P]
        l.orc_codebook_build_zero_atom.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                                   ctypes.c_double, P]
        l.orc_codebook_assign_codes.argtypes = [P]
        l.orc_shift.argtypes = [P, ctypes.c_uint64, ctypes.c_int]
        l.orc_encode.argtypes = [P, P, P]
        l.orc_decode.argtypes = [P, P, P]
        l.orc_bf16_rne.argtypes = [ctypes.c_float]
        l.orc_bf16_rne.restype = ctypes.c_uint16
        l.orc_sgd_step.argtypes = [P, P, P, P, ctypes.c_float, P]
        l.orc_sgd_momentum_step.argtypes = [P, P, P, P, P, ctypes.c_float, ctypes.c_float, P, P, P]
        l.orc_adamw_constants.argtypes = [ctypes.c_double] * 5 + [ctypes.c_uint32, P]
        l.orc_adamw_constants.restype = None
        l.orc_adamw_step.argtypes = [P] * 7 + [P, P, P, P, P]
        _lib = l
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def geometry(level: int) -> tuple[int, int]:
    b, w = ctypes.c_uint32(), ctypes.c_uint32()
    rc = lib().orc_level_geometry(level, ctypes.byref(b), ctypes.byref(w))
    if rc != OK:
        raise ValueError("bad level %r" % level)
    return b.value, w.value


def model_pmf(model: int, scale: float, shape: float = 0.0) -> np.ndarray:
    p = np.zeros(256, dtype=np.float64)
    rc = lib().orc_model_pmf(model, scale, shape, _ptr(p))
    if rc != OK:
        raise ValueError("bad model parameters")
    return p


def weights_from_pmf(p: np.ndarray) -> np.ndarray:
    p = np.ascontiguousarray(p, dtype=np.float64)
    w = np.zeros(256, dtype=np.uint64)
    lib().orc_weights_from_pmf(_ptr(p), _ptr(w))
    return w


def package_merge(weights, L: int, ids=None) -> np.ndarray:
    w = np.ascontiguousarray(weights, dtype=np.uint64)
    n = len(w)
    idv = np.ascontiguousarray(np.arange(n) if ids is None else ids, dtype=np.int32)
    out = np.zeros(n, dtype=np.uint8)
    rc = lib().orc_package_merge(n, _ptr(w), _ptr(idv), L, _ptr(out))
    if rc != OK:
        raise ValueError("package-merge rejected n=%d L=%d" % (n, L))
    return out


def codebook_from_weights(w) -> Codebook:
    w = np.ascontiguousarray(w, dtype=np.uint64)
    cb = Codebook()
    rc = lib().orc_codebook_from_weights(_ptr(w), ctypes.byref(cb))
    if rc != OK:
        raise ValueError("codebook construction failed")
    return cb


def codebook_build(model: int, scale: float, shape: float = 0.0) -> Codebook:
    cb = Codebook()
    rc = lib().orc_codebook_build(model, scale, shape, ctypes.byref(cb))
    if rc != OK:
        raise ValueError("bad model parameters")
    return cb


def codebook_build_zero_atom(model: int, scale: float, shape: float, zero_frac: float) -> Codebook:
    """A model with a point mass of zero_frac at exponent 0 (zeros), coded
    as an unshifted symbol 0."""
    cb = Codebook()
    rc = lib().orc_codebook_build_zero_atom(model, scale, shape, zero_frac, ctypes.byref(cb))
    if rc != OK:
        raise ValueError("bad model parameters")
    return cb


def codebook_from_lengths(lengths, esc_len: int, median_exp: int = 127) -> Codebook:
    """A hand-made codebook: given lengths, canonical codes assigned."""
    cb = Codebook()
    for s, l in enumerate(lengths):
        cb.len[s] = int(l)
    cb.esc_len = esc_len
    cb.median_exp = median_exp
    rc = lib().orc_codebook_assign_codes(ctypes.byref(cb))
    if rc != OK:
        raise ValueError("lengths violate the Kraft inequality or the cap")
    return cb


def shift(x: np.ndarray, median_exp: int) -> int:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    return int(lib().orc_shift(_ptr(x), x.size, median_exp))


def bf16_rne(f: float) -> int:
    return int(lib().orc_bf16_rne(f))


@dataclass
class Compressed:
    """One compressed tensor as host arrays (the oracle's view of the format)."""
    n: int
    block: int
    slot_words: int
    delta: int
    sf: np.ndarray
    slots: np.ndarray
    markers: np.ndarray
    blk_off: np.ndarray
    ovf: np.ndarray
    ovf_used: int = 0
    status: int = OK

    @property
    def nblocks(self) -> int:
        return (self.n + self.block - 1) // self.block

    @classmethod
    def empty(cls, n: int, block: int, slot_words: int, ovf_cap: int | None = None):
        nb = (n + block - 1) // block
        cap = n if ovf_cap is None else ovf_cap
        return cls(n, block, slot_words, 0,
                   np.zeros(n, np.uint8),
                   np.zeros(nb * slot_words * STREAMS, np.uint32),
                   np.zeros(nb * STREAMS, np.uint16),
                   np.zeros(nb + 1, np.uint64),
                   np.zeros(max(cap, 1), np.uint8)[:cap] if cap > 0 else np.zeros(0, np.uint8))

    def _struct(self) -> _Tensor:
        t = _Tensor()
        t.n = self.n
        t.block = self.block
        t.slot_words = self.slot_words
        t.delta = self.delta
        t.sf = _ptr(self.sf).value
        t.slots = _ptr(self.slots).value
        t.markers = _ptr(self.markers).value
        t.blk_off = _ptr(self.blk_off).value
        t.ovf = _ptr(self.ovf).value if self.ovf.size else None
        t.ovf_cap = self.ovf.size
        t.ovf_used = self.ovf_used
        return t

    def overflow_bytes(self) -> np.ndarray:
        return self.ovf[: min(self.ovf_used, self.ovf.size)]


def encode(x: np.ndarray, cb: Codebook, level: int | None = None, *, block=None,
           slot_words=None, delta=None, ovf_cap=None) -> Compressed:
    """Shift estimate (unless ``delta`` is given) and encode."""
    x = np.ascontiguousarray(x, dtype=np.uint16).reshape(-1)
    if level is not None:
        block, slot_words = geometry(level)
    if delta is None:
        delta = shift(x, cb.median_exp)
    c = Compressed.empty(x.size, block, slot_words, ovf_cap)
    c.delta = delta
    t = c._struct()
    c.status = lib().orc_encode(_ptr(x), ctypes.byref(cb), ctypes.byref(t))
    c.ovf_used = int(t.ovf_used)
    return c


def decode(c: Compressed, cb: Codebook) -> tuple[int, np.ndarray]:
    y = np.zeros(c.n, dtype=np.uint16)
    t = c._struct()
    rc = lib().orc_decode(ctypes.byref(t), ctypes.byref(cb), _ptr(y) if c.n else None)
    return int(rc), y


def sgd_step(W: Compressed, cbW: Codebook, M: Compressed, cbM: Codebook, eta: float,
             ovf_cap=None) -> Compressed:
    out = Compressed.empty(W.n, W.block, W.slot_words, ovf_cap)
    tw, tm, to = W._struct(), M._struct(), out._struct()
    out.status = lib().orc_sgd_step(ctypes.byref(tw), ctypes.byref(cbW), ctypes.byref(tm),
                                    ctypes.byref(cbM), ctypes.c_float(eta), ctypes.byref(to))
    out.delta = int(to.delta)
    out.ovf_used = int(to.ovf_used)
    return out


def sgd_momentum_step(W: Compressed, cbW: Codebook, M: Compressed, cbM: Codebook, g: np.ndarray,
                      eta: float, mu: float, ovf_cap_w=None, ovf_cap_m=None) -> tuple[Compressed, Compressed]:
    """Heavy-ball momentum step on compressed W and M with a dense BF16
    gradient (uint16 bit patterns): returns the new (W, M)."""
    g = np.ascontiguousarray(g, dtype=np.uint16).reshape(-1)
    if g.size != W.n:
        raise ValueError("gradient size differs from W")
    w_out = Compressed.empty(W.n, W.block, W.slot_words, ovf_cap_w)
    m_out = Compressed.empty(M.n, M.block, M.slot_words, ovf_cap_m)
    tw, tm, tow, tom = W._struct(), M._struct(), w_out._struct(), m_out._struct()
    rc = (ctypes.c_int * 2)()
    lib().orc_sgd_momentum_step(ctypes.byref(tw), ctypes.byref(cbW), ctypes.byref(tm), ctypes.byref(cbM),
                                _ptr(g) if g.size else None, ctypes.c_float(eta), ctypes.c_float(mu),
                                ctypes.byref(tow), ctypes.byref(tom), rc)
    for out, t, st in ((w_out, tow, rc[0]), (m_out, tom, rc[1])):
        out.status = int(st)
        out.delta = int(t.delta)
        out.ovf_used = int(t.ovf_used)
    return w_out, m_out


def adamw_constants(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, t: int) -> np.ndarray:
    """The eight float constants of one AdamW step (see orc_adamw_constants)."""
    k = np.zeros(8, np.float32)
    lib().orc_adamw_constants(lr, beta1, beta2, eps, weight_decay, t, _ptr(k))
    return k


def adamw_step(W: Compressed, cbW: Codebook, M: Compressed, cbM: Codebook, V: Compressed, cbV: Codebook,
               g: np.ndarray, k: np.ndarray, caps=(None, None, None)):
    """One AdamW step on compressed W, M, V with a dense BF16 gradient:
    returns the new (W, M, V)."""
    g = np.ascontiguousarray(g, dtype=np.uint16).reshape(-1)
    k = np.ascontiguousarray(k, dtype=np.float32)
    if g.size != W.n or k.size != 8:
        raise ValueError("gradient size differs from W, or k is not 8 floats")
    outs = [Compressed.empty(t.n, t.block, t.slot_words, cap) for t, cap in zip((W, M, V), caps)]
    ts = [t._struct() for t in (W, M, V)]
    tos = [o._struct() for o in outs]
    rc = (ctypes.c_int * 3)()
    lib().orc_adamw_step(ctypes.byref(ts[0]), ctypes.byref(cbW), ctypes.byref(ts[1]), ctypes.byref(cbM),
                         ctypes.byref(ts[2]), ctypes.byref(cbV), _ptr(g) if g.size else None, _ptr(k),
                         ctypes.byref(tos[0]), ctypes.byref(tos[1]), ctypes.byref(tos[2]), rc)
    for o, t, st in zip(outs, tos, rc):
        o.status = int(st)
        o.delta = int(t.delta)
        o.ovf_used = int(t.ovf_used)
    return tuple(outs)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
