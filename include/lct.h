/*
 * lct.h -- C ABI of liblct.so: lossless BF16 tensor compression on the GPU
 * (exponent-Huffman coding with fixed-length streams) and the fused
 * compressed SGD step, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow two pages describing LCT (Losslessly Compressed
 * Tensors), cited by title and paragraph:
 *   [ABS] "LCT: Losslessly Compressed Tensors with GPU friendly execution for
 *         Training" (Zhu, Sun, Lio, Yu), abstract page;
 *   [EXP] "LCT paper -- Lossless Huffman coding of BF16 training tensors --
 *         What does it mean?", explainer page; paragraphs are named by their
 *         opening words ("In bits", "Compressing is easy", "Training adds a
 *         second problem", "Here is the idealized arithmetic").
 *
 * Conventions shared by every entry point
 *   - Every function returns an lct_status and never throws.
 *   - The library never allocates device memory.  All device buffers are
 *     owned by the caller and named by plain device pointers ("d_" prefix);
 *     every other pointer is a host pointer.
 *   - GPU work is enqueued asynchronously on `stream` (a cudaStream_t passed
 *     as void*; NULL is the legacy default stream).  Nothing synchronises
 *     except lct_compressed_size() with a tensor.
 *   - Errors the host can see (NULL or misaligned pointers, size mismatches,
 *     bad levels, malformed codebooks, overlapping buffers) return at once
 *     and enqueue nothing.  Errors only the GPU can see (overflow capacity
 *     exceeded, corrupt stream data, an overflow-offset wait that ran out)
 *     are latched into the tensor's device header; read them back with
 *     lct_compressed_size().  Device-side checks never fault: every index
 *     into caller memory is bounds-checked and skipped on failure.
 *   - Device pointers must be 16-byte aligned.
 *   - Launches report CUDA launch errors as LCT_ERR_CUDA.
 */
#ifndef LCT_H
#define LCT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LCT_OK = 0,
    LCT_ERR_INVALID_ARG = 1,       /* host-side argument check failed */
    LCT_ERR_UNSUPPORTED = 2,       /* valid request the library does not implement */
    LCT_ERR_OVERFLOW_CAPACITY = 3, /* device: the overflow bytes did not fit d_ovf */
    LCT_ERR_CORRUPT = 4,           /* device: header, markers or offsets inconsistent */
    LCT_ERR_TIMEOUT = 5,           /* device: a wait for an earlier block's offset ran out */
    LCT_ERR_CUDA = 6               /* a CUDA runtime call failed */
} lct_status;

/* Exponent distribution models the user picks from ([EXP] "In bits"). */
typedef enum {
    LCT_MODEL_GAUSSIAN = 0, /* |x| half-normal, scale = sigma */
    LCT_MODEL_LAPLACE = 1,  /* |x| exponential, scale = b */
    LCT_MODEL_POWERLAW = 2  /* |x| Lomax (Pareto II), scale = s, shape = alpha */
} lct_model;

/* Block levels ([EXP] "Compressing is easy"): CLEAN blocks hold 65,536
 * exponents, MEDIUM and HIGH 32,768.  Each stream's slot is 800 bits in
 * CLEAN (3.125 bits/exponent; the pages' 1.4382x CLEAN bound,
 * [EXP] "Here is the idealized arithmetic"), 512 bits in MEDIUM and 640 bits
 * in HIGH (4 and 5 bits/exponent: sizes the pages do not print). */
typedef enum { LCT_LEVEL_CLEAN = 0, LCT_LEVEL_MEDIUM = 1, LCT_LEVEL_HIGH = 2 } lct_level;

#define LCT_STREAMS 256        /* streams per block, dealt round-robin */
#define LCT_MAX_CODE_BITS 8    /* code length cap ([EXP] "In bits") */
#define LCT_LITERAL_BITS 8     /* raw exponent after the escape prefix */
#define LCT_SHIFT_SAMPLES 4096 /* at most this many samples set the shift */
#define LCT_HEADER_BYTES 64
#define LCT_MAGIC 0x3154434Cu  /* "LCT1" */

/* A precomputed codebook ([EXP] "In bits": built ahead of time from the
 * chosen model, codes at most 8 bits, rare exponents under one escape prefix
 * followed by an 8-bit literal).  Plain host data, about 1 KB; it is copied
 * into kernel parameters on every call.
 *
 * Symbols are shifted exponents s = e - delta (delta from the tensor header).
 * Codes are canonical: ordered by (length, symbol), escape last among equal
 * lengths; code values are right-aligned in `len` bits, sent most significant
 * bit first. */
typedef struct {
    uint8_t len[256];     /* code length of symbol s (1..8), 0 = sent as escape */
    uint8_t code[256];    /* code of symbol s, right-aligned */
    uint16_t dec[256];    /* 8-bit window -> bits 0..8 symbol (256 = escape), bits 12..15 length */
    uint8_t esc_len;      /* escape prefix length (1..8) */
    uint8_t esc_code;     /* escape prefix, right-aligned */
    uint16_t nsym;        /* symbols with their own code */
    int32_t median_exp;   /* the model's median biased exponent (1..254) */
    int32_t model;        /* lct_model it was built from */
    uint32_t hash;        /* 32-bit FNV-1a of len, code, esc_len, esc_code, zero_atom */
    double scale, shape;  /* model parameters it was built from */
    double zero_frac;     /* point mass at zero it was built with (0 = none) */
    uint32_t zero_atom;   /* 1: exponent 0 always codes as symbol 0, unshifted;
                             a nonzero exponent the shift maps to symbol 0 escapes */
    uint32_t reserved;
} lct_codebook;

/* Device header, LCT_HEADER_BYTES at t->d_header.  Written by lct_encode and
 * lct_sgd_step_fused; read by lct_decode and lct_compressed_size. */
typedef struct {
    uint32_t magic;    /* LCT_MAGIC */
    uint32_t version;  /* 1 */
    uint64_t n;        /* BF16 values */
    int32_t level;     /* lct_level */
    int32_t delta;     /* scale shift: symbol = exponent - delta */
    uint32_t status;   /* first device-side error latched (an lct_status), 0 = none */
    uint32_t cb_hash;  /* codebook hash the streams were written with */
    uint64_t ovf_used; /* overflow bytes the last write needed (may exceed ovf_cap) */
    uint64_t ovf_cap;  /* capacity the last write was given */
    uint64_t reserved[2];
} lct_header;

/* A compressed tensor: caller-owned device regions (sizes from
 * lct_compressed_size).  Layout, with nblocks = ceil(n / block):
 *   d_sf       n bytes: sign in bit 7, fraction in bits 0..6, element order
 *              ([EXP] "In bits": the sign-fraction byte is stored as is);
 *   d_slots    nblocks * slot_words * 256 uint32, index [block][word][stream]:
 *              stream j of a block holds its positions i with i mod 256 = j
 *              ([EXP] "Compressing is easy": neighbours go to different
 *              streams), codes packed MSB-first from bit 31 of word 0, unused
 *              bits zero;
 *   d_markers  nblocks * 256 uint16: symbols held in each slot; the stream's
 *              later symbols are in the overflow (the spill-start marker);
 *   d_blk_off  nblocks + 1 uint64: exclusive prefix of the blocks' overflow
 *              byte counts; entry nblocks is the total;
 *   d_ovf      ovf_cap bytes: spilled exponents, uncompressed, in (block,
 *              stream, symbol) order; may be a slice of a buffer shared by
 *              many tensors ([EXP] "Here is the idealized arithmetic");
 *   d_work     work_bytes of scratch for the blocks' overflow-offset scan
 *              (not part of the compressed data; needed by writers only). */
typedef struct {
    uint64_t n;
    int32_t level;
    int32_t reserved;
    void *d_header;
    uint8_t *d_sf;
    uint32_t *d_slots;
    uint16_t *d_markers;
    uint64_t *d_blk_off;
    uint8_t *d_ovf;
    uint64_t ovf_cap;
    void *d_work;
} lct_tensor;

typedef struct {
    uint64_t n;
    uint64_t nblocks;
    uint32_t block;            /* exponents per block */
    uint32_t slot_words;       /* 32-bit words per stream slot */
    uint64_t header_bytes;
    uint64_t sf_bytes;
    uint64_t slot_bytes;
    uint64_t marker_bytes;
    uint64_t blk_off_bytes;
    uint64_t fixed_bytes;      /* header + sf + slots + markers + blk_off */
    uint64_t worst_ovf_bytes;  /* n: every exponent spilled */
    uint64_t work_bytes;       /* d_work scratch */
    /* filled only when a tensor is passed (after a stream synchronise) */
    uint64_t ovf_used;         /* overflow bytes the last write needed */
    uint32_t status;           /* latched device status (lct_status) */
    int32_t delta;             /* the tensor's scale shift */
} lct_sizes;

/* Build a codebook from a distribution model ([EXP] "In bits"; the paper's
 * "precomputed codebooks", [ABS]).  Host only, deterministic.
 *   model  lct_model; scale > 0 (sigma, b or s); shape = alpha > 0 for the
 *          power-law model, ignored otherwise.
 * Exponent bucket e holds |x| in [2^(e-127), 2^(e-126)) (e = 0: zeros and
 * subnormals; e = 254 open above; e = 255 weight 0).  Bucket masses are
 * scaled by 2^40 and rounded to integers; for k = 1..min(255, nonzero
 * buckets) the k heaviest buckets (ties: smaller exponent first) get codes
 * alongside an escape of the remaining weight (at least 1), lengths from
 * package-merge capped at 8 bits; the k with the least expected bits wins
 * (smallest k on a tie).  Errors: LCT_ERR_INVALID_ARG for a NULL `out` or
 * bad parameters. */
lct_status lct_codebook_build(int model, double scale, double shape, lct_codebook *out);

/* The same with a point mass at zero: a fraction zero_frac (0 <= zero_frac <
 * 1) of the values are exactly zero, as in ReLU/GELU activations, and the
 * rest follow the model.  Bucket masses are (1 - zero_frac) * p(e), plus
 * zero_frac at e = 0; the rest of the construction is lct_codebook_build's.
 * The pages note that the user supplies the distribution and that one which
 * does not fit the tensor raises storage ([EXP] "Read the 3.5x longer context
 * claim carefully"); zeros are a common misfit, since any shift moves them to
 * an unused symbol and they escape at 16 bits each.  The resulting codebook
 * has zero_atom = 1: exponent 0 (zeros and subnormals) always codes as symbol
 * 0 whatever the tensor's shift, and a nonzero exponent that the shift maps
 * onto symbol 0 is escaped.  The pages have no such model; its encoding is
 * decoded by lct_decode like any other.  Returns LCT_ERR_INVALID_ARG for bad
 * parameters. */
lct_status lct_codebook_build_zero_atom(int model, double scale, double shape, double zero_frac,
                                        lct_codebook *out);

/* Region sizes for an n-value tensor at `level`, and, when `t` is not NULL,
 * the state of a written tensor: synchronises `stream`, then reads the
 * device header into out->ovf_used / status / delta.
 * Compression ratio = 2n / (fixed_bytes + ovf_used).  Errors:
 * LCT_ERR_INVALID_ARG (NULL out, bad level, n > 2^40, t->n or t->level not
 * matching), LCT_ERR_CUDA. */
lct_status lct_compressed_size(uint64_t n, int level, const lct_tensor *t, void *stream,
                               lct_sizes *out);

/* Compress n BF16 values d_x (device, 16-byte aligned) into `t`
 * ([EXP] "In bits" and "Compressing is easy").  Enqueues:
 *   1. the scale shift: at most 4096 values sampled at floor(k*n/m); the lower
 *      median of their normal exponents (1..254) minus cb->median_exp,
 *      clamped to [-127, 127], 0 if none; written to the header;
 *   2. one pass per block: sign-fraction bytes out, each exponent coded as
 *      its symbol's code or escape + 8-bit raw exponent, packed into its
 *      stream's slot until the first code that does not fit (the marker);
 *      the rest of the stream spills to d_ovf; blocks' overflow offsets come
 *      from a single-pass scan over d_work.
 * If the overflow exceeds t->ovf_cap, blocks that do not fit write no
 * overflow bytes and LCT_ERR_OVERFLOW_CAPACITY is latched; header.ovf_used
 * tells the size needed.  d_x is not modified. */
lct_status lct_encode(const uint16_t *d_x, const lct_codebook *cb, const lct_tensor *t,
                      void *stream);

/* lct_encode for callers that cannot allocate device memory.  (The paper has
 * no counterpart: this is a convenience of this library.)
 *
 * lct_encode needs `t->d_work`, a little device scratch (8 bytes per block)
 * for the scan that places each block's overflow bytes.  Some callers cannot
 * allocate it: a caching allocator or out-of-memory handler that compresses
 * tensors to free space would have to re-enter the allocator, or fail for
 * lack of memory, to get scratch; other code must avoid cudaMalloc/cudaFree
 * because they can synchronise the device.  This variant allocates nothing:
 * its scratch is a fixed array of LCT_STATIC_SCRATCH_BLOCKS 8-byte words
 * (128 KiB) compiled into the library, which every GPU that loads the library
 * holds until the process exits.  `t->d_work` is ignored and may be NULL;
 * everything else is exactly as for lct_encode (same checks, same output,
 * bit for bit).
 *   - Tensors needing more than LCT_STATIC_SCRATCH_BLOCKS blocks (n above
 *     2^30 values in CLEAN, 2^29 in MEDIUM and HIGH) are rejected with
 *     LCT_ERR_UNSUPPORTED before anything is enqueued.
 *   - Every call looks up the array's device address on the current device
 *     (nothing is cached, so the address stays right after cudaDeviceReset).
 *     The first call on a device may load the library's device code there;
 *     make that first call before any stream capture.
 *   - All calls share the one array.  Each call clears the words it uses
 *     before using them, but calls whose GPU work overlaps -- on different
 *     streams, or from different threads -- race on the array and may produce
 *     wrong overflow offsets.  Serialise them.
 * Errors: as lct_encode, plus LCT_ERR_UNSUPPORTED (too large) and
 * LCT_ERR_CUDA (the device address could not be obtained). */
#define LCT_STATIC_SCRATCH_BLOCKS 16384
lct_status lct_encode_static_scratch(const uint16_t *d_x, const lct_codebook *cb, const lct_tensor *t,
                                     void *stream);

/* Reconstruct the n BF16 values of `t` into d_y (device, 16-byte aligned),
 * bit for bit ([EXP] "In bits": every value decodes exactly).  `cb` must be
 * the codebook the tensor was written with (checked on the device by hash).
 * Latches LCT_ERR_CORRUPT (bad magic, n, level or hash, a marker beyond its
 * stream, a slot whose codes run past it, offsets that disagree with the
 * markers) or LCT_ERR_OVERFLOW_CAPACITY (overflow never written); d_y is then
 * unspecified.  d_y must not overlap the tensor. */
lct_status lct_decode(const lct_tensor *t, const lct_codebook *cb, uint16_t *d_y, void *stream);

/* Decode only blocks first_block .. first_block + nblocks - 1 of `t` into d_y
 * (device, 16-byte aligned): value i of block first_block goes to d_y[i], so
 * d_y holds min(nblocks * block, n - first_block * block) values.  This is
 * the piece for decoding a compressed matmul operand tile by tile into a
 * small dense buffer that a GEMM reads ([EXP] "Read the 3.5x longer context
 * claim carefully": decoding inside matmul kernels is named as future work;
 * decoding a tile at a time ahead of a library GEMM keeps only one tile
 * dense).  Blocks are independent given the stored shift and offsets.
 * nblocks = 0 enqueues nothing.  Errors as lct_decode (latched in t's
 * header), plus LCT_ERR_INVALID_ARG for a range past the last block. */
lct_status lct_decode_blocks(const lct_tensor *t, const lct_codebook *cb, uint64_t first_block, uint64_t nblocks,
                             uint16_t *d_y, void *stream);

/* One fused SGD step W <- W - eta*M on compressed W and M ([EXP] "Training
 * adds a second problem": read the compressed inputs, compute, write the new
 * bytes in one pass).  Per value, in float32: p = round(eta*m),
 * r = round(w - p) (two roundings, no fused multiply-add), then BF16 by
 * round-to-nearest-even (subnormals kept, NaN -> 0x7FC0).  The new W is coded
 * with cbW and W_in's stored shift (the codebook stays fixed).
 * W_in, M and W_out must have the same n and level.  W_out may share
 * d_header, d_sf, d_slots, d_markers and d_blk_off with W_in (in-place
 * update) but its d_ovf and d_work must not overlap W_in's or M's overflow,
 * and W_out must not overlap M.  M is read only. */
lct_status lct_sgd_step_fused(const lct_tensor *W_in, const lct_codebook *cbW, const lct_tensor *M,
                              const lct_codebook *cbM, float eta, const lct_tensor *W_out,
                              void *stream);

/* One fused SGD-with-momentum step on compressed W and M with a dense BF16
 * gradient d_g (n values, 16-byte aligned):
 *   M' = bf16(round(round(mu*m) + g)),   W' = bf16(round(w - round(eta*M')))
 * The pages name the momentum buffer of SGD with momentum as optimizer state
 * that LCT keeps compressed ([EXP] "Jargon", entry "Optimizer state"; [ABS])
 * and ask for a single-pass update of compressed tensors ([EXP] "Training
 * adds a second problem"); they print no update rule, so this is the
 * heavy-ball form without dampening or Nesterov term.  Every float32 product
 * and sum is rounded on its own (no fused multiply-add); the weight step uses
 * M' as stored (BF16); rounding to BF16 is round-to-nearest-even with
 * subnormals kept and NaN -> 0x7FC0.  W' is coded with cbW and W_in's stored
 * shift, M' with cbM and M_in's stored shift.
 * All four tensors must have the same n and level.  Each output may share
 * d_header, d_sf, d_slots, d_markers and d_blk_off with its own input (in
 * place) but not partly overlap them; its d_ovf and d_work must be apart from
 * every input region; W' and M' must not overlap each other, W' must not
 * overlap M_in, M' must not overlap W_in, and d_g must not overlap either
 * output.  Each output latches its own status (capacity, corrupt input,
 * timeout); a corrupt input or a timeout is latched in both. */
lct_status lct_sgd_momentum_step_fused(const lct_tensor *W_in, const lct_codebook *cbW, const lct_tensor *M_in,
                                       const lct_codebook *cbM, const uint16_t *d_g, float eta, float mu,
                                       const lct_tensor *W_out, const lct_tensor *M_out, void *stream);

/* Hyper-parameters of one AdamW step (step >= 1 counts the steps taken,
 * this one included). */
typedef struct {
    double lr;
    double beta1, beta2;   /* in [0, 1) */
    double eps;            /* > 0 */
    double weight_decay;   /* decoupled: W <- W - lr*weight_decay*W */
    uint64_t step;
} lct_adamw_params;

/* One fused AdamW step on compressed W, M (first moment) and V (second
 * moment) with a dense BF16 gradient d_g (n values, 16-byte aligned).  The
 * pages name optimizer state -- buffers the size of the weights that the
 * optimizer keeps -- among the tensors LCT stores compressed ([EXP] "Jargon",
 * entry "Optimizer state"; [ABS]) and ask for updates that read and write
 * compressed tensors in one pass ([EXP] "Training adds a second problem");
 * they print no optimizer, so this is AdamW with decoupled weight decay.
 * With float constants rounded once from the parameters in double,
 *   b1 = beta1, c1 = 1 - beta1, b2 = beta2, c2 = 1 - beta2,
 *   a = lr / (1 - beta1^step), r = 1 / sqrt(1 - beta2^step), e = eps,
 *   d = lr * weight_decay,
 * every value is updated with each float32 operation rounded on its own (no
 * fused multiply-add; sqrt and division correctly rounded):
 *   M' = bf16(b1*m + c1*g)
 *   V' = bf16(b2*v + c2*(g*g))
 *   W' = bf16((w - d*w) - (a*M') / (sqrt(V')*r + e))
 * where the weight update takes M' and V' as stored (BF16); rounding to BF16
 * is round-to-nearest-even with subnormals kept and NaN -> 0x7FC0.  Each
 * output is coded with its input's codebook and stored shift.  Two passes:
 * one kernel writes M' and V', a second one W' (reading M' and V').
 * All six tensors must have the same n and level.  Each output may share
 * d_header, d_sf, d_slots, d_markers and d_blk_off with its own input (in
 * place) but not partly overlap them; its d_ovf and d_work must be apart from
 * every input region; an output must not overlap another output or another
 * tensor's input, and d_g must not overlap any output.  Each output latches
 * its own status; LCT_ERR_INVALID_ARG for bad parameters. */
lct_status lct_adamw_step_fused(const lct_tensor *W_in, const lct_codebook *cbW, const lct_tensor *M_in,
                                const lct_codebook *cbM, const lct_tensor *V_in, const lct_codebook *cbV,
                                const uint16_t *d_g, const lct_adamw_params *p, const lct_tensor *W_out,
                                const lct_tensor *M_out, const lct_tensor *V_out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* LCT_H */
