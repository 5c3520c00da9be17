"""Lossless BF16 tensor compression on GB300 (sm_103a): LCT's exponent-Huffman
codec, the fused compressed SGD / SGD-with-momentum / AdamW steps, and the
pieces built on them for training (saved activations kept compressed,
a linear layer whose weight is decoded tile by tile).

The work happens in ``liblct.so`` (CUDA kernels behind a C ABI, declared in
``include/lct.h``); ``binding`` is its thin ctypes binding, re-exported here:

    from lossless_bf16_tensor_gb300 import (lct_codebook_build, lct_codebook_build_zero_atom,
                                            lct_encode, lct_decode, lct_decode_blocks,
                                            lct_sgd_step_fused, lct_sgd_momentum_step_fused,
                                            lct_adamw_step_fused, lct_compressed_size,
                                            CompressedTensor)

``activations.compressed_activations`` and ``matmul.compressed_linear`` are
imported from their modules.  The binding is loaded on first attribute access
and raises if the library is not built; nothing falls back to the CPU.
"""

_BINDING_NAMES = {"lct_codebook_build", "lct_codebook_build_zero_atom", "lct_encode", "lct_decode",
                  "lct_decode_blocks", "lct_sgd_step_fused", "lct_sgd_momentum_step_fused",
                  "lct_adamw_step_fused", "lct_encode_static_scratch", "lct_compressed_size",
                  "lct_debug_wait_timeout", "CompressedTensor", "LctError", "library"}


def __getattr__(name):
    if name in _BINDING_NAMES:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
