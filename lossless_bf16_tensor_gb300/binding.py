"""ctypes binding of liblct.so with the C ABI's names (argument marshalling only).

Every step of the codec runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.  There is no CPU fallback:
importing this module fails if the library has not been built
(``python -m lossless_bf16_tensor_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblct.so")

if not os.path.exists(LIB_PATH):
    raise ImportError("liblct.so is not built (run `python -m lossless_bf16_tensor_gb300.build`); "
                      "the codec has no CPU fallback")

_lib = ctypes.CDLL(LIB_PATH)

# ------------------------------------------------------------ constants

LCT_OK, LCT_ERR_INVALID_ARG, LCT_ERR_UNSUPPORTED, LCT_ERR_OVERFLOW_CAPACITY, LCT_ERR_CORRUPT, \
    LCT_ERR_TIMEOUT, LCT_ERR_CUDA = range(7)
STATUS_NAMES = {0: "LCT_OK", 1: "LCT_ERR_INVALID_ARG", 2: "LCT_ERR_UNSUPPORTED",
                3: "LCT_ERR_OVERFLOW_CAPACITY", 4: "LCT_ERR_CORRUPT", 5: "LCT_ERR_TIMEOUT",
                6: "LCT_ERR_CUDA"}
LCT_MODEL_GAUSSIAN, LCT_MODEL_LAPLACE, LCT_MODEL_POWERLAW = 0, 1, 2
LCT_LEVEL_CLEAN, LCT_LEVEL_MEDIUM, LCT_LEVEL_HIGH = 0, 1, 2
LCT_HEADER_BYTES = 64
LCT_STATIC_SCRATCH_BLOCKS = 16384
LCT_MAGIC = 0x3154434C
MODELS = {"gaussian": 0, "laplace": 1, "powerlaw": 2}
LEVELS = {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}


class LctError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s" % (what, STATUS_NAMES.get(status, status)))
        self.status = status


# ------------------------------------------------------------ structures

class lct_codebook(ctypes.Structure):
    _fields_ = [("len", ctypes.c_uint8 * 256), ("code", ctypes.c_uint8 * 256),
                ("dec", ctypes.c_uint16 * 256), ("esc_len", ctypes.c_uint8),
                ("esc_code", ctypes.c_uint8), ("nsym", ctypes.c_uint16),
                ("median_exp", ctypes.c_int32), ("model", ctypes.c_int32),
                ("hash", ctypes.c_uint32), ("scale", ctypes.c_double), ("shape", ctypes.c_double),
                ("zero_frac", ctypes.c_double), ("zero_atom", ctypes.c_uint32), ("reserved", ctypes.c_uint32)]


class lct_adamw_params(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("step", ctypes.c_uint64)]


class lct_tensor(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("level", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("d_header", ctypes.c_void_p), ("d_sf", ctypes.c_void_p), ("d_slots", ctypes.c_void_p),
                ("d_markers", ctypes.c_void_p), ("d_blk_off", ctypes.c_void_p), ("d_ovf", ctypes.c_void_p),
                ("ovf_cap", ctypes.c_uint64), ("d_work", ctypes.c_void_p)]


class lct_sizes(ctypes.Structure):
    _fields_ = [("n", ctypes.c_uint64), ("nblocks", ctypes.c_uint64), ("block", ctypes.c_uint32),
                ("slot_words", ctypes.c_uint32), ("header_bytes", ctypes.c_uint64),
                ("sf_bytes", ctypes.c_uint64), ("slot_bytes", ctypes.c_uint64),
                ("marker_bytes", ctypes.c_uint64), ("blk_off_bytes", ctypes.c_uint64),
                ("fixed_bytes", ctypes.c_uint64), ("worst_ovf_bytes", ctypes.c_uint64),
                ("work_bytes", ctypes.c_uint64), ("ovf_used", ctypes.c_uint64),
                ("status", ctypes.c_uint32), ("delta", ctypes.c_int32)]


_P = ctypes.c_void_p
_lib.lct_codebook_build.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.POINTER(lct_codebook)]
_lib.lct_codebook_build_zero_atom.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                              ctypes.POINTER(lct_codebook)]
_lib.lct_compressed_size.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.POINTER(lct_tensor), _P,
                                     ctypes.POINTER(lct_sizes)]
_lib.lct_encode.argtypes = [_P, ctypes.POINTER(lct_codebook), ctypes.POINTER(lct_tensor), _P]
_lib.lct_decode.argtypes = [ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook), _P, _P]
_lib.lct_decode_blocks.argtypes = [ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook), ctypes.c_uint64,
                                   ctypes.c_uint64, _P, _P]
_lib.lct_sgd_step_fused.argtypes = [ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook),
                                    ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook), ctypes.c_float,
                                    ctypes.POINTER(lct_tensor), _P]
_lib.lct_sgd_momentum_step_fused.argtypes = [ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook),
                                             ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook), _P,
                                             ctypes.c_float, ctypes.c_float, ctypes.POINTER(lct_tensor),
                                             ctypes.POINTER(lct_tensor), _P]
_lib.lct_adamw_step_fused.argtypes = [ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_codebook)] * 3 + [
    _P, ctypes.POINTER(lct_adamw_params), ctypes.POINTER(lct_tensor), ctypes.POINTER(lct_tensor),
    ctypes.POINTER(lct_tensor), _P]
_lib.lct_debug_wait_timeout.argtypes = [_P, _P, ctypes.c_uint64, _P]
_lib.lct_encode_static_scratch.argtypes = [_P, ctypes.POINTER(lct_codebook), ctypes.POINTER(lct_tensor), _P]
for _fn in ("lct_codebook_build", "lct_codebook_build_zero_atom", "lct_compressed_size", "lct_encode", "lct_decode",
            "lct_decode_blocks", "lct_sgd_step_fused",
            "lct_sgd_momentum_step_fused", "lct_adamw_step_fused", "lct_debug_wait_timeout",
            "lct_encode_static_scratch"):
    getattr(_lib, _fn).restype = ctypes.c_int


def library() -> ctypes.CDLL:
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != LCT_OK:
        raise LctError(rc, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _model(m) -> int:
    return MODELS[m] if isinstance(m, str) else int(m)


def _level(lv) -> int:
    return LEVELS[lv] if isinstance(lv, str) else int(lv)


# ------------------------------------------------------------ entry points

def lct_codebook_build(model, scale: float, shape: float = 0.0) -> lct_codebook:
    cb = lct_codebook()
    _check(_lib.lct_codebook_build(_model(model), float(scale), float(shape), ctypes.byref(cb)),
           "lct_codebook_build")
    return cb


def lct_codebook_build_zero_atom(model, scale: float, shape: float, zero_frac: float) -> lct_codebook:
    cb = lct_codebook()
    _check(_lib.lct_codebook_build_zero_atom(_model(model), float(scale), float(shape), float(zero_frac),
                                             ctypes.byref(cb)), "lct_codebook_build_zero_atom")
    return cb


def lct_compressed_size(n: int, level, t: "CompressedTensor | None" = None, stream=None) -> lct_sizes:
    s = lct_sizes()
    desc = ctypes.byref(t.desc) if t is not None else None
    _check(_lib.lct_compressed_size(int(n), _level(level), desc, _stream(stream) if t is not None else None,
                                    ctypes.byref(s)), "lct_compressed_size")
    return s


def _dev_ptr(x: torch.Tensor, n: int) -> int:
    if not x.is_cuda or x.element_size() != 2 or not x.is_contiguous() or x.numel() != n:
        raise ValueError("expected a contiguous CUDA tensor of %d 16-bit values" % n)
    return x.data_ptr()


def lct_encode(x: torch.Tensor, cb: lct_codebook, t: "CompressedTensor", stream=None) -> None:
    ptr = _dev_ptr(x, t.n) if t.n else None
    _check(_lib.lct_encode(ptr, ctypes.byref(cb), ctypes.byref(t.desc), _stream(stream)), "lct_encode")


def lct_encode_static_scratch(x: torch.Tensor, cb: lct_codebook, t: "CompressedTensor", stream=None) -> None:
    """lct_encode without caller-provided scratch: for callers that cannot
    allocate device memory (e.g. an allocator compressing tensors to free
    space); the library's fixed scratch array is used instead of t's."""
    ptr = _dev_ptr(x, t.n) if t.n else None
    _check(_lib.lct_encode_static_scratch(ptr, ctypes.byref(cb), ctypes.byref(t.desc), _stream(stream)),
           "lct_encode_static_scratch")


def lct_decode(t: "CompressedTensor", cb: lct_codebook, y: torch.Tensor, stream=None) -> None:
    ptr = _dev_ptr(y, t.n) if t.n else None
    _check(_lib.lct_decode(ctypes.byref(t.desc), ctypes.byref(cb), ptr, _stream(stream)), "lct_decode")


def lct_decode_blocks(t: "CompressedTensor", cb: lct_codebook, first_block: int, nblocks: int, y: torch.Tensor,
                      stream=None) -> None:
    """Decode blocks first_block .. first_block+nblocks-1 into y (a CUDA
    16-bit tensor holding exactly those blocks' values)."""
    block = int(t.sizes.block)
    lo = int(first_block) * block
    hi = min(t.n, (int(first_block) + int(nblocks)) * block)
    ptr = _dev_ptr(y, max(hi - lo, 0)) if nblocks else None
    _check(_lib.lct_decode_blocks(ctypes.byref(t.desc), ctypes.byref(cb), int(first_block), int(nblocks), ptr,
                                  _stream(stream)), "lct_decode_blocks")


def lct_sgd_step_fused(W_in: "CompressedTensor", cbW: lct_codebook, M: "CompressedTensor", cbM: lct_codebook,
                       eta: float, W_out: "CompressedTensor", stream=None) -> None:
    _check(_lib.lct_sgd_step_fused(ctypes.byref(W_in.desc), ctypes.byref(cbW), ctypes.byref(M.desc),
                                   ctypes.byref(cbM), ctypes.c_float(eta), ctypes.byref(W_out.desc),
                                   _stream(stream)), "lct_sgd_step_fused")


def lct_sgd_momentum_step_fused(W_in: "CompressedTensor", cbW: lct_codebook, M_in: "CompressedTensor",
                                cbM: lct_codebook, g: torch.Tensor, eta: float, mu: float,
                                W_out: "CompressedTensor", M_out: "CompressedTensor", stream=None) -> None:
    ptr = _dev_ptr(g, W_in.n) if W_in.n else None
    _check(_lib.lct_sgd_momentum_step_fused(ctypes.byref(W_in.desc), ctypes.byref(cbW), ctypes.byref(M_in.desc),
                                            ctypes.byref(cbM), ptr, ctypes.c_float(eta), ctypes.c_float(mu),
                                            ctypes.byref(W_out.desc), ctypes.byref(M_out.desc), _stream(stream)),
           "lct_sgd_momentum_step_fused")


def lct_adamw_step_fused(W_in: "CompressedTensor", cbW: lct_codebook, M_in: "CompressedTensor", cbM: lct_codebook,
                         V_in: "CompressedTensor", cbV: lct_codebook, g: torch.Tensor, lr: float, beta1: float,
                         beta2: float, eps: float, weight_decay: float, step: int, W_out: "CompressedTensor",
                         M_out: "CompressedTensor", V_out: "CompressedTensor", stream=None) -> None:
    ptr = _dev_ptr(g, W_in.n) if W_in.n else None
    p = lct_adamw_params(float(lr), float(beta1), float(beta2), float(eps), float(weight_decay), int(step))
    _check(_lib.lct_adamw_step_fused(ctypes.byref(W_in.desc), ctypes.byref(cbW), ctypes.byref(M_in.desc),
                                     ctypes.byref(cbM), ctypes.byref(V_in.desc), ctypes.byref(cbV), ptr,
                                     ctypes.byref(p), ctypes.byref(W_out.desc), ctypes.byref(M_out.desc),
                                     ctypes.byref(V_out.desc), _stream(stream)), "lct_adamw_step_fused")


def lct_debug_wait_timeout(header: torch.Tensor, work: torch.Tensor, limit_ns: int, stream=None) -> None:
    _check(_lib.lct_debug_wait_timeout(header.data_ptr(), work.data_ptr(), int(limit_ns), _stream(stream)),
           "lct_debug_wait_timeout")


# ------------------------------------------------------------ allocation

def _round_up(v: int, a: int = 256) -> int:
    return (v + a - 1) // a * a


class CompressedTensor:
    """Device regions of one compressed tensor, carved from one torch buffer.

    ``ovf_cap`` defaults to the worst case (n bytes); pass a smaller value or
    an external ``ovf`` (a uint8 CUDA tensor, e.g. a slice of a shared
    overflow buffer) to share overflow space between tensors.
    """

    def __init__(self, n: int, level, ovf_cap: int | None = None, device="cuda", ovf: torch.Tensor | None = None,
                 like: "CompressedTensor | None" = None, zero_fill: bool = True):
        self.n = int(n)
        self.level = _level(level)
        self.sizes = lct_compressed_size(self.n, self.level)
        s = self.sizes
        if ovf is not None:
            ovf_cap = ovf.numel()
        elif ovf_cap is None:
            ovf_cap = s.worst_ovf_bytes
        self.ovf_cap = int(ovf_cap)
        parts = [("header", s.header_bytes), ("sf", s.sf_bytes), ("slots", s.slot_bytes),
                 ("markers", s.marker_bytes), ("blk_off", s.blk_off_bytes), ("work", s.work_bytes)]
        if like is not None:
            # share everything but the overflow and the scratch (in-place SGD)
            parts = [("work", s.work_bytes)]
        if ovf is None:
            parts.append(("ovf", self.ovf_cap))
        offs, total = {}, 0
        for name, size in parts:
            offs[name] = (total, int(size))
            total = _round_up(total + int(size))
        # a writer fills every region it owns (header, sign-fraction bytes,
        # slots, markers, offsets, the used overflow) and clears its scratch,
        # so zero filling is only for tidiness
        alloc = torch.zeros if zero_fill else torch.empty
        self.buffer = alloc(max(total, 256), dtype=torch.uint8, device=device)
        self.regions = {name: self.buffer[o:o + sz] for name, (o, sz) in offs.items()}
        if like is not None:
            for name in ("header", "sf", "slots", "markers", "blk_off"):
                self.regions[name] = like.regions[name]
        if ovf is not None:
            self.regions["ovf"] = ovf
        d = lct_tensor()
        d.n = self.n
        d.level = self.level
        d.d_header = self.regions["header"].data_ptr()
        d.d_sf = self.regions["sf"].data_ptr() if self.n else None
        d.d_slots = self.regions["slots"].data_ptr() if self.n else None
        d.d_markers = self.regions["markers"].data_ptr() if self.n else None
        d.d_blk_off = self.regions["blk_off"].data_ptr() if self.n else None
        d.d_ovf = self.regions["ovf"].data_ptr() if self.ovf_cap else None
        d.ovf_cap = self.ovf_cap
        d.d_work = self.regions["work"].data_ptr() if self.n else None
        self.desc = d

    @property
    def nblocks(self) -> int:
        return int(self.sizes.nblocks)

    def state(self, stream=None) -> lct_sizes:
        """Synchronise and read the header (ovf_used, status, delta)."""
        return lct_compressed_size(self.n, self.level, self, stream)

    def compression_ratio(self, stream=None) -> float:
        st = self.state(stream)
        return 2.0 * self.n / (self.sizes.fixed_bytes + st.ovf_used) if self.n else 1.0

    def to_host(self) -> dict:
        """Copy every region to host numpy arrays (unsigned views)."""
        def cpu(name, dt):
            return self.regions[name].cpu().numpy().view(dt)
        out = {"sf": cpu("sf", np.uint8), "slots": cpu("slots", np.uint32), "markers": cpu("markers", np.uint16),
               "blk_off": cpu("blk_off", np.uint64), "ovf": cpu("ovf", np.uint8)}
        hdr = self.regions["header"].cpu().numpy()
        out["header"] = hdr
        out["delta"] = int(hdr[20:24].view(np.int32)[0])
        out["status"] = int(hdr[24:28].view(np.uint32)[0])
        out["ovf_used"] = int(hdr[32:40].view(np.uint64)[0])
        return out
