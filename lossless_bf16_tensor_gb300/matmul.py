"""Matmul with a compressed operand, decoded one tile at a time.

[EXP] "LCT paper -- Lossless Huffman coding of BF16 training tensors -- What
does it mean?", paragraph "Read the 3.5x longer context claim carefully":
decoding inside matmul kernels is named as future work.  Here the compressed
weight is decoded tile by tile (``lct_decode_blocks``) into a double buffer
on a side stream while cuBLAS (torch.mm) consumes the previous tile on the
caller's stream, so only two tiles of the weight are ever dense.

Only orchestration lives here: decoding runs in liblct's kernels, the GEMM in
cuBLAS.
"""
from __future__ import annotations

import torch

from . import binding as B


_SIDE_STREAMS: dict = {}


def _side_stream(device: torch.device) -> torch.cuda.Stream:
    """One decode stream per device, made on first use and kept: a new stream
    per call would cost a driver call each time."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    if idx not in _SIDE_STREAMS:
        _SIDE_STREAMS[idx] = torch.cuda.Stream(device=idx)
    return _SIDE_STREAMS[idx]


def tile_rows(ct: B.CompressedTensor, in_features: int, tile_blocks: int) -> int:
    """Rows of a row-major [out, in] weight that `tile_blocks` blocks hold."""
    vals = tile_blocks * int(ct.sizes.block)
    if vals % in_features:
        raise ValueError("a tile of %d blocks (%d values) does not hold whole rows of %d" %
                         (tile_blocks, vals, in_features))
    return vals // in_features


def default_tile_blocks(w: B.CompressedTensor, in_features: int, device: torch.device) -> int:
    """A tile of about four blocks per SM (one full wave of decode CTAs),
    rounded down to whole rows, or the whole weight if that is smaller.  A
    block's streams decode serially (a decode launch of one block takes about
    19 us on a GB300, of 608 blocks about 40 us), so a tile of a few blocks
    leaves most SMs idle and small tiles cost far more than the GEMM they
    feed."""
    idx = device.index if device.index is not None else torch.cuda.current_device()
    want = 4 * torch.cuda.get_device_properties(idx).multi_processor_count
    if want >= w.nblocks:
        return w.nblocks
    block = int(w.sizes.block)
    step = 1
    while (step * block) % in_features:  # smallest block count holding whole rows
        step += 1
    return max(step, want // step * step)


def compressed_linear(x: torch.Tensor, w: B.CompressedTensor, cb: B.lct_codebook, out_features: int,
                      in_features: int, tile_blocks: int | None = None) -> torch.Tensor:
    """y = x @ W^T for a BF16 weight W [out_features, in_features], stored
    compressed in row-major order; x [..., in_features] BF16 on CUDA.  W is
    decoded `tile_blocks` blocks (a whole number of rows) at a time; by default
    one wave of decode CTAs (default_tile_blocks)."""
    if w.n != out_features * in_features:
        raise ValueError("weight size does not match its shape")
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.shape[-1] != in_features:
        raise ValueError("x must be a CUDA BF16 tensor [..., in_features]")
    if tile_blocks is None:
        tile_blocks = default_tile_blocks(w, in_features, x.device)
    x2 = x.reshape(-1, in_features)
    if tile_blocks >= w.nblocks:
        # one tile: decode the whole weight on the caller's stream, one GEMM
        dense = torch.empty(w.n, dtype=torch.bfloat16, device=x.device)
        B.lct_decode(w, cb, dense.view(torch.int16), torch.cuda.current_stream(x.device))
        return torch.mm(x2, dense.view(out_features, in_features).t()).reshape(*x.shape[:-1], out_features)
    rows = tile_rows(w, in_features, tile_blocks)
    main = torch.cuda.current_stream(x.device)
    side = _side_stream(x.device)
    nbuf = 2
    bufs = [torch.empty(rows * in_features, dtype=torch.bfloat16, device=x.device) for _ in range(nbuf)]
    decoded = [torch.cuda.Event() for _ in range(nbuf)]
    consumed = [torch.cuda.Event() for _ in range(nbuf)]
    x2t = x2.t()
    # y^T [out, M]: the rows of one weight tile give contiguous rows of y^T
    yt = torch.empty(out_features, x2t.shape[1], dtype=torch.bfloat16, device=x.device)
    ntiles = (w.nblocks + tile_blocks - 1) // tile_blocks
    side.wait_stream(main)  # x, w and the buffers are ready
    for t in range(ntiles):
        k = t % nbuf
        first = t * tile_blocks
        count = min(tile_blocks, w.nblocks - first)
        r0 = t * rows
        r1 = min(out_features, r0 + rows)
        tile = bufs[k][:(r1 - r0) * in_features]
        if t >= nbuf:
            side.wait_event(consumed[k])  # the GEMM nbuf tiles back has read this buffer
        B.lct_decode_blocks(w, cb, first, count, tile.view(torch.int16), side)
        decoded[k].record(side)
        main.wait_event(decoded[k])
        torch.mm(tile.view(r1 - r0, in_features), x2t, out=yt[r0:r1])
        consumed[k].record(main)
    # every decode on the side stream finished before the main stream's last
    # GEMM, so the buffers (allocated on the main stream) can be freed as usual
    return yt.t().contiguous().reshape(*x.shape[:-1], out_features)
