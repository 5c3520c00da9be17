// Library-private declarations shared by the host entry points and the CUDA
// kernels of liblct.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/lct.h"

namespace lct {

constexpr int kStreams = LCT_STREAMS;
constexpr uint64_t kMaxN = 1ull << 40;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s bound on any device wait

struct Geometry {
    uint32_t block;       // exponents per block
    uint32_t slot_words;  // 32-bit words per stream slot
};

// [EXP] "Compressing is easy": 65,536-value blocks in CLEAN, 32,768 in MEDIUM
// and HIGH.  Slot sizes: 800 bits in CLEAN (the 1.4382x bound of [EXP] "Here
// is the idealized arithmetic"); 512 and 640 bits in MEDIUM and HIGH.
inline bool level_geometry(int level, Geometry *g)
{
    switch (level) {
    case LCT_LEVEL_CLEAN: *g = {65536u, 25u}; return true;
    case LCT_LEVEL_MEDIUM: *g = {32768u, 16u}; return true;
    case LCT_LEVEL_HIGH: *g = {32768u, 20u}; return true;
    default: return false;
    }
}

uint32_t codebook_hash(const lct_codebook &cb);
bool codebook_valid(const lct_codebook &cb);

// The codebook as kernels receive it (by value, in kernel parameters).
struct DevCodebook {
    uint8_t len[256];
    uint8_t code[256];
    uint16_t dec[256];
    uint8_t esc_len;
    uint8_t esc_code;
    uint8_t zero_atom;  // exponent 0 <-> symbol 0, unshifted
    uint8_t pad;
    uint32_t hash;
};

// Device view of one compressed tensor.
struct DevTensor {
    lct_header *hdr;
    uint8_t *sf;
    uint32_t *slots;
    uint16_t *markers;
    uint64_t *blk_off;
    uint8_t *ovf;
    unsigned long long *work;  // per-block scan status words
    uint64_t ovf_cap;
    uint64_t n;
    uint32_t nblocks;
    int32_t level;
};

// Every argument block carries two multipliers, 32 and 4, that the decoders
// use for address arithmetic: as launch arguments they are not compile-time
// constants, so the multiply-adds stay on the FMA pipe instead of becoming
// shifts on the integer ALU pipe.
struct EncodeArgs {
    const uint16_t *x;
    DevTensor t;
    DevCodebook cb;
    int32_t median_exp;
    uint32_t pad;
    uint64_t wait_ns;
    uint32_t mul_row, mul_ent, mul_sf, pad_mul;  // 32, 4 and 0x01010000 (set_multipliers)
    uint32_t deferred, pad_def;  // block offsets computed after the writer (set by its launcher)
};

struct DecodeArgs {
    DevTensor t;
    uint16_t *y;          // value i of block first_block is y[i]
    DevCodebook cb;
    uint64_t wait_ns;
    uint32_t first_block;  // the launch decodes blocks first_block .. + grid size
    uint32_t pad;
    uint32_t mul_row, mul_ent, mul_sf, pad_mul;  // 32, 4 and 0x01010000 (set_multipliers)
    uint32_t deferred, pad_def;  // block offsets computed after the writer (set by its launcher)
};

// Weight updates of the fused one-pass kernel.
enum : uint32_t { OP_SGD = 0, OP_ADAMW = 1 };

struct UpdateArgs {
    DevTensor in[3];      // W, M, and V for AdamW
    DevTensor w_out;
    DevCodebook cb[3];
    float k[8];           // the step's constants (SGD: k[0] = eta)
    uint32_t op;          // OP_SGD or OP_ADAMW
    uint32_t nin;         // inputs used: 2 or 3
    uint32_t in_place;    // W_out's sign-fraction bytes are W_in's
    uint32_t pad;
    uint64_t wait_ns;
    uint32_t mul_row, mul_ent, mul_sf, pad_mul;  // 32, 4 and 0x01010000 (set_multipliers)
    uint32_t deferred, pad_def;  // block offsets computed after the writer (set by its launcher)
};

// Updates of the fused two-state kernel (two compressed tensors and a dense
// gradient in, both tensors out).
enum : uint32_t { OP2_MOMENTUM = 0, OP2_ADAM_MOMENTS = 1 };

struct MomentumArgs {
    DevTensor w_in, m_in, w_out, m_out;  // the two states (W and M, or AdamW's M and V)
    const uint16_t *g;  // dense BF16 gradient, n values
    DevCodebook cbw, cbm;
    float k[8];         // the step's constants (momentum: k[0] = eta, k[1] = mu)
    uint32_t op;        // OP2_MOMENTUM or OP2_ADAM_MOMENTS
    uint32_t in_place;  // an output shares its input's sign-fraction bytes
    uint64_t wait_ns;
    uint32_t mul_row, mul_ent, mul_sf, pad_mul;  // 32, 4 and 0x01010000 (set_multipliers)
    uint32_t deferred, pad_def;  // block offsets computed after the writer (set by its launcher)
};

template <typename Args>
inline void set_multipliers(Args &a)
{
    a.mul_row = 32;
    a.mul_ent = 4;
    a.mul_sf = 0x01010000u;
    a.pad_mul = 0;
    a.deferred = 0;
    a.pad_def = 0;
}

cudaError_t launch_encode(const EncodeArgs &a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs &a, uint32_t nblocks, cudaStream_t s);
cudaError_t launch_update(const UpdateArgs &a, cudaStream_t s);
cudaError_t launch_momentum(const MomentumArgs &a, cudaStream_t s);
// Deferred placement (grids of at least four blocks per SM): a block with no
// overflow bytes publishes its count and leaves, blocks with bytes to place
// still wait for their exclusive prefix, and launch_block_offsets (after the
// writer) writes every block offset, ovf_used and the capacity check.
bool deferred_placement(uint32_t nblocks);
// Grids of at most two blocks per SM (the launch is latency-bound).
bool small_grid(uint32_t nblocks);
cudaError_t launch_block_offsets(const DevTensor &t, cudaStream_t s);
cudaError_t launch_block_offsets2(const DevTensor &t0, const DevTensor &t1, cudaStream_t s);  // same nblocks
cudaError_t launch_wait_probe(lct_header *hdr, unsigned long long *work, uint64_t wait_ns,
                              cudaStream_t s);

}  // namespace lct
