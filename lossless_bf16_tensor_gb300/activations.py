"""Saved activations kept compressed between forward and backward.

The pages compress a network's activations during training (the NanoGPT row
"activations compressed" of [EXP] "LCT paper -- Lossless Huffman coding of
BF16 training tensors -- What does it mean?", results table): each tensor
autograd saves for the backward pass is encoded when it is saved and decoded
when backward needs it.  Because the codec is lossless the gradients are bit
for bit those of the uncompressed run.

This module only orchestrates calls through the C ABI (``lct_encode`` /
``lct_decode``); the coding runs in liblct's kernels.

Overflow room is bounded: a saved tensor gets ``ovf_frac * n`` bytes of
overflow.  Whether a tensor fitted is known only when its encode has run, so
the BF16 original is kept until then.  The check is asynchronous (a pinned
copy of the header and a CUDA event per tensor): finished encodes are
checked at every later save, and at most ``max_pending`` tensors wait
unchecked before the oldest is waited for.  A tensor that did not fit keeps
its original and drops the compressed copy.
"""
from __future__ import annotations

import math

import torch

from . import binding as B

_STATUS_OFFSET = 24  # lct_header.status


class _Saved:
    __slots__ = ("ct", "shape", "original", "event", "hdr", "checked")

    def __init__(self, ct, shape, original, event, hdr):
        self.ct = ct
        self.shape = shape
        self.original = original
        self.event = event
        self.hdr = hdr
        self.checked = False


class compressed_activations:
    """Context manager: while active, BF16 CUDA tensors that autograd saves
    for backward (at least ``min_numel`` values, not parameters) are stored
    LCT-compressed with codebook ``cb`` at ``level``.

    ``stats`` counts the tensors and bytes: raw (2 bytes per value) and
    compressed (the regions a compressed tensor holds, overflow capacity
    included) for the tensors that stayed compressed, and the tensors that
    fell back to their original because the overflow did not fit.
    """

    def __init__(self, cb: B.lct_codebook, level="CLEAN", min_numel: int = 65536, ovf_frac: float = 0.125,
                 max_pending: int = 4):
        if not 0.0 <= ovf_frac <= 1.0:
            raise ValueError("ovf_frac must be within [0, 1]")
        self.cb = cb
        self.level = B._level(level)
        self.min_numel = int(min_numel)
        self.ovf_frac = float(ovf_frac)
        self.max_pending = int(max_pending)
        self._pending: list[_Saved] = []
        self._ctx = None
        self.stats = {"compressed": 0, "fallback": 0, "raw_bytes": 0, "stored_bytes": 0}

    # ---------------------------------------------------------- context
    def __enter__(self):
        self._ctx = torch.autograd.graph.saved_tensors_hooks(self._pack, self._unpack)
        self._ctx.__enter__()
        return self

    def __exit__(self, *exc):
        self._ctx.__exit__(*exc)
        self._ctx = None
        return False

    def flush(self) -> None:
        """Wait for every pending encode and settle it (drop originals that
        are no longer needed)."""
        for e in self._pending:
            self._settle(e, wait=True)
        self._pending = []

    # ------------------------------------------------------------ hooks
    def _eligible(self, t: torch.Tensor) -> bool:
        return (t.is_cuda and t.dtype == torch.bfloat16 and t.numel() >= self.min_numel
                and not isinstance(t, torch.nn.Parameter))

    def _pack(self, t: torch.Tensor):
        if not self._eligible(t):
            return t
        self._poll()
        n = t.numel()
        src = t.contiguous().view(torch.int16).reshape(-1)
        ct = B.CompressedTensor(n, self.level, ovf_cap=int(math.ceil(n * self.ovf_frac)), device=t.device,
                                zero_fill=False)
        stream = torch.cuda.current_stream(t.device)
        B.lct_encode(src, self.cb, ct, stream)
        hdr = torch.empty(64, dtype=torch.uint8, pin_memory=True)
        hdr.copy_(ct.regions["header"], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream)
        e = _Saved(ct, t.shape, t, ev, hdr)
        self._pending.append(e)
        return e

    def _unpack(self, e):
        if not isinstance(e, _Saved):
            return e
        if not e.checked:
            self._settle(e, wait=True)
            self._pending = [p for p in self._pending if p is not e]
        if e.original is not None:
            return e.original
        y = torch.empty(e.shape, dtype=torch.bfloat16, device=e.ct.buffer.device)
        stream = torch.cuda.current_stream(y.device)
        e.ct.buffer.record_stream(stream)  # backward may run on another stream than the save
        B.lct_decode(e.ct, self.cb, y.view(torch.int16).reshape(-1), stream)
        return y

    # ---------------------------------------------------- async checks
    def _poll(self) -> None:
        keep = []
        for i, e in enumerate(self._pending):
            must_wait = len(self._pending) - i > self.max_pending
            if must_wait or e.event.query():
                self._settle(e, wait=must_wait)
            else:
                keep.append(e)
        self._pending = keep

    def _settle(self, e: _Saved, wait: bool) -> None:
        if e.checked:
            return
        if wait:
            e.event.synchronize()
        status = int(e.hdr[_STATUS_OFFSET:_STATUS_OFFSET + 4].view(torch.int32).item())
        n = e.ct.n
        if status == B.LCT_OK:
            e.original = None
            self.stats["compressed"] += 1
            self.stats["raw_bytes"] += 2 * n
            self.stats["stored_bytes"] += e.ct.buffer.numel()
        else:
            e.ct = None
            self.stats["fallback"] += 1
        e.checked = True
