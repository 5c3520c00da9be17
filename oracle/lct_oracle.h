/*
 * lct_oracle.h -- plain, slow, single-threaded CPU oracle for the LCT BF16
 * exponent-Huffman codec and the fused compressed SGD step.
 *
 * TEST INFRASTRUCTURE ONLY.  This code exists to check the CUDA path.  Only
 * the test suite, the smoke check and the CPU-baseline leg of the benchmark
 * may load it.  It shares no source, header, table or constant with the CUDA
 * library; both are written independently from the same description.
 *
 * Sources (cited by page title and section):
 *   [ABS] "LCT: Losslessly Compressed Tensors with GPU friendly execution for
 *         Training" (Zhu, Sun, Lio, Yu), abstract page.
 *   [EXP] "LCT paper -- Lossless Huffman coding of BF16 training tensors --
 *         What does it mean?" (explainer page); paragraphs are named by their
 *         opening words: "In bits", "Compressing is easy", "Training adds a
 *         second problem", "Here is the idealized arithmetic".
 *
 * Where the pages leave a choice open, the oracle takes one reading and marks
 * it "(reading)".  The CUDA path must reproduce every such choice bit for bit.
 *
 * Parity status of each function (what pins it, besides itself):
 *   orc_model_pmf        closed-form entropies, scipy distributions, exact
 *                        2x scale-shift invariance                 (pinned)
 *   orc_package_merge    brute force on tiny alphabets, textbook Huffman
 *                        when the cap does not bind, all-8 special case (pinned)
 *   orc_codebook_*       Kraft equality, prefix freedom, E[len] in [H, H+0.2],
 *                        the pages' 2.5-3.2 bit figures            (pinned)
 *   ..._zero_atom        mass 1, the plain model's lengths at zero_frac 0,
 *                        one-bit zero code past p = 2/5, lossless for every
 *                        shift, 2^k scaling invariance of the markers (pinned)
 *   orc_shift            hand example, 2^k scaling law             (pinned)
 *   orc_encode/decode    bit-exact roundtrip on all 65,536 BF16 patterns,
 *                        hand-worked stream fixture, bit accounting (pinned;
 *                        the stream layout itself is a reading the pages do
 *                        not print, so only the hand fixture pins it)
 *   orc_sgd_step         torch CPU float32 ops + bf16 cast           (pinned)
 *   orc_sgd_momentum_step  torch CPU float32 ops + bf16 casts, one-FMA
 *                        sensitivity, the mu = 0 reduction           (pinned)
 *   orc_adamw_step       torch CPU float32 ops + bf16 casts, FMA sensitivity,
 *                        first step from zero moments = sign descent (pinned)
 */
#ifndef LCT_ORACLE_H
#define LCT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes (the oracle's own numbering). */
#define ORC_OK 0
#define ORC_BAD_ARG 1
#define ORC_CAPACITY 3
#define ORC_CORRUPT 4

/* Exponent models the user picks from ([EXP] "In bits"). */
#define ORC_GAUSSIAN 0
#define ORC_LAPLACE 1
#define ORC_POWERLAW 2

/* Escape pseudo-symbol id (one past the 256 exponent values). */
#define ORC_ESC 256

typedef struct {
    uint64_t weight[256]; /* integer model weight of exponent symbol s */
    uint8_t len[256];     /* code length of symbol s; 0 = sent under the escape */
    uint16_t code[256];   /* canonical code of symbol s, right-aligned in len bits */
    uint8_t esc_len;      /* length of the escape prefix */
    uint8_t pad0;
    uint16_t esc_code;    /* escape prefix, right-aligned */
    int32_t k;            /* number of symbols with their own code */
    int32_t median_exp;   /* model median of the biased exponent, in [1, 254] */
    uint16_t lut_sym[256];/* 8-bit window -> symbol, or ORC_ESC */
    uint8_t lut_len[256]; /* 8-bit window -> length of the code at its head */
    int32_t zero_atom;    /* 1: symbol 0 is the zero atom (exponent 0, never shifted) */
} orc_codebook;

/* One compressed tensor, as plain host arrays owned by the caller. */
typedef struct {
    uint64_t n;          /* number of BF16 values */
    uint32_t block;      /* exponents per block */
    uint32_t slot_words; /* 32-bit words in each stream's fixed slot */
    int32_t delta;       /* scale shift applied before the code lookup */
    uint32_t pad0;
    uint8_t *sf;         /* n sign-fraction bytes, element order */
    uint32_t *slots;     /* nblocks * slot_words * 256 words, [block][word][stream] */
    uint16_t *markers;   /* nblocks * 256: symbols held in each stream's slot */
    uint64_t *blk_off;   /* nblocks + 1: start of each block's overflow bytes */
    uint8_t *ovf;        /* overflow bytes (raw exponents) */
    uint64_t ovf_cap;    /* capacity of ovf in bytes */
    uint64_t ovf_used;   /* out: overflow bytes the tensor needs */
} orc_tensor;

int orc_level_geometry(int level, uint32_t *block, uint32_t *slot_words);

int orc_model_pmf(int model, double scale, double shape, double p[256]);
void orc_weights_from_pmf(const double p[256], uint64_t w[256]);

int orc_package_merge(int n, const uint64_t *w, const int32_t *id, int L, uint8_t *len_out);

int orc_codebook_from_weights(const uint64_t w[256], orc_codebook *cb);
int orc_codebook_build(int model, double scale, double shape, orc_codebook *cb);
int orc_codebook_build_zero_atom(int model, double scale, double shape, double zero_frac, orc_codebook *cb);
int orc_codebook_assign_codes(orc_codebook *cb);

int orc_shift(const uint16_t *x, uint64_t n, int median_exp);

int orc_encode(const uint16_t *x, const orc_codebook *cb, orc_tensor *t);
int orc_decode(const orc_tensor *t, const orc_codebook *cb, uint16_t *y);

uint16_t orc_bf16_rne(float f);
int orc_sgd_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                 const orc_codebook *cbM, float eta, orc_tensor *W_out);
int orc_sgd_momentum_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                          const orc_codebook *cbM, const uint16_t *g, float eta, float mu,
                          orc_tensor *W_out, orc_tensor *M_out, int rc[2]);
void orc_adamw_constants(double lr, double beta1, double beta2, double eps, double weight_decay,
                         uint32_t t, float k[8]);
int orc_adamw_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                   const orc_codebook *cbM, const orc_tensor *V, const orc_codebook *cbV,
                   const uint16_t *g, const float k[8], orc_tensor *W_out, orc_tensor *M_out,
                   orc_tensor *V_out, int rc[3]);

#ifdef __cplusplus
}
#endif
#endif
