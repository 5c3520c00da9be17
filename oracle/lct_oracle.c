/*
 * lct_oracle.c -- the CPU oracle (test infrastructure; see lct_oracle.h).
 *
 * Plain C99, single-threaded, built with floating-point contraction off.
 * Every step follows the explainer's description in its own order:
 *   1. split each BF16 value into a sign-fraction byte and an exponent byte
 *      ([EXP] "In bits");
 *   2. code the exponent with a precomputed Huffman codebook whose codes are
 *      at most 8 bits long, rare exponents going out as one escape prefix plus
 *      an 8-bit literal; the codebook comes from a chosen distribution model
 *      and is shifted to the tensor's scale from at most 4096 sampled values
 *      ([EXP] "In bits");
 *   3. deal the exponents of each block (65,536 in CLEAN, 32,768 in MEDIUM
 *      and HIGH) round-robin to 256 streams, each filling a slot of fixed
 *      length; what does not fit spills uncompressed to an overflow region and
 *      a marker records where the spill starts ([EXP] "Compressing is easy");
 *   4. the SGD update W - eta*M on compressed W and M ([EXP] "Training adds
 *      a second problem").
 */
#include "lct_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- geometry */

#define NSTREAMS 256
#define MAXLEN 8    /* code length cap ([EXP] "In bits") */
#define LITBITS 8   /* escape literal width ([EXP] "In bits") */

/* Block sizes are the pages' ([EXP] "Compressing is easy").  Slot sizes:
 * CLEAN 25 words = 800 bits per 256 exponents = 3.125 bits/exponent, the
 * value for which the payload ratio 2B/(B + 256*slot_bytes) is the 1.4382x
 * CLEAN bound of [EXP] "Here is the idealized arithmetic".  MEDIUM (16 words,
 * 4 bits/exponent) and HIGH (20 words, 5 bits/exponent) are not printed on
 * the pages (reading). */
int orc_level_geometry(int level, uint32_t *block, uint32_t *slot_words)
{
    switch (level) {
    case 0: *block = 65536; *slot_words = 25; return ORC_OK;
    case 1: *block = 32768; *slot_words = 16; return ORC_OK;
    case 2: *block = 32768; *slot_words = 20; return ORC_OK;
    default: return ORC_BAD_ARG;
    }
}

static uint64_t nblocks_of(uint64_t n, uint32_t block)
{
    return (n + block - 1) / block;
}

/* Values held by block b. */
static uint64_t block_count(uint64_t n, uint32_t block, uint64_t b)
{
    uint64_t start = b * (uint64_t)block;
    uint64_t left = n - start;
    return left < block ? left : block;
}

/* Symbols of stream j in a block of nb values: positions j, j+256, ... */
static uint32_t stream_count(uint64_t nb, uint32_t j)
{
    if (nb <= j) return 0;
    return (uint32_t)((nb - j + NSTREAMS - 1) / NSTREAMS);
}

/* ------------------------------------------------------------ byte split */

/* BF16 = 1 sign + 8 exponent + 7 fraction bits ([EXP] "In bits"). */
static uint8_t exponent_of(uint16_t h) { return (uint8_t)((h >> 7) & 0xFF); }

/* Sign in bit 7, fraction in bits 0..6 (reading). */
static uint8_t signfrac_of(uint16_t h)
{
    return (uint8_t)(((h >> 8) & 0x80) | (h & 0x7F));
}

static uint16_t join_bf16(uint8_t sf, uint8_t e)
{
    return (uint16_t)(((uint16_t)(sf & 0x80) << 8) | ((uint16_t)e << 7) | (sf & 0x7F));
}

/* ------------------------------------------------------------ model pmf */

/* Model cdf of |x|.  Gaussian: erf(t / (sigma sqrt 2)); Laplace: 1 - exp(-t/b);
 * power-law: the Lomax / Pareto-II form 1 - (1 + t/s)^-alpha (reading: the
 * pages only say "power-law"). */
static double model_cdf(int model, double scale, double shape, double t)
{
    if (isinf(t)) return 1.0;
    switch (model) {
    case ORC_GAUSSIAN: return erf(t / (scale * sqrt(2.0)));
    case ORC_LAPLACE: return 1.0 - exp(-t / scale);
    default: return 1.0 - pow(1.0 + t / scale, -shape);
    }
}

/* p(e) = mass of |x| in exponent bucket e: [2^(e-127), 2^(e-126)) for
 * 1 <= e <= 254, [0, 2^-126) for e = 0 (zeros and subnormals), the top bucket
 * open to +inf, and p(255) = 0 (reading: bucket edges ignore BF16 rounding). */
int orc_model_pmf(int model, double scale, double shape, double p[256])
{
    if (model < ORC_GAUSSIAN || model > ORC_POWERLAW) return ORC_BAD_ARG;
    if (!(scale > 0.0) || isinf(scale)) return ORC_BAD_ARG;
    if (model == ORC_POWERLAW && (!(shape > 0.0) || isinf(shape))) return ORC_BAD_ARG;
    for (int e = 0; e < 256; e++) {
        if (e == 255) { p[e] = 0.0; continue; }
        double lo = (e == 0) ? 0.0 : ldexp(1.0, e - 127);
        double hi = (e == 254) ? INFINITY : ldexp(1.0, e - 126);
        p[e] = model_cdf(model, scale, shape, hi) - model_cdf(model, scale, shape, lo);
    }
    return ORC_OK;
}

/* Integer weights w = round(p * 2^40) (reading: fixed-point so that the code
 * construction below is exact integer arithmetic). */
void orc_weights_from_pmf(const double p[256], uint64_t w[256])
{
    for (int e = 0; e < 256; e++) w[e] = (uint64_t)llround(ldexp(p[e], 40));
}

/* ------------------------------------------------ length-limited Huffman */

/* Package-merge (Larmore & Hirschberg) for code lengths capped at L.
 * Items are either leaves or packages of two items of the previous list. */
typedef struct {
    uint64_t w;
    int leaf;      /* leaf index, or -1 for a package */
    int a, b;      /* package: indices into the previous list */
} pm_item;

static void pm_count(pm_item **lists, int level, int idx, int *count)
{
    pm_item it = lists[level][idx];
    if (it.leaf >= 0) { count[it.leaf]++; return; }
    pm_count(lists, level - 1, it.a, count);
    pm_count(lists, level - 1, it.b, count);
}

/* Leaves are taken in order of (weight ascending, id ascending); when a leaf
 * and a package weigh the same, the leaf comes first.  Code length of a leaf
 * = number of times it occurs in the first 2n-2 items of the last list. */
int orc_package_merge(int n, const uint64_t *w, const int32_t *id, int L, uint8_t *len_out)
{
    if (n < 2 || L < 1 || L > 30 || (n > (1 << L))) return ORC_BAD_ARG;
    int *order = (int *)malloc(sizeof(int) * n);
    for (int i = 0; i < n; i++) order[i] = i;
    /* insertion sort: plain and obviously stable */
    for (int i = 1; i < n; i++) {
        int v = order[i], j = i - 1;
        while (j >= 0 && (w[order[j]] > w[v] || (w[order[j]] == w[v] && id[order[j]] > id[v]))) {
            order[j + 1] = order[j];
            j--;
        }
        order[j + 1] = v;
    }
    pm_item **lists = (pm_item **)malloc(sizeof(pm_item *) * L);
    int *sizes = (int *)malloc(sizeof(int) * L);
    lists[0] = (pm_item *)malloc(sizeof(pm_item) * n);
    for (int i = 0; i < n; i++) {
        lists[0][i].w = w[order[i]];
        lists[0][i].leaf = order[i];
        lists[0][i].a = lists[0][i].b = -1;
    }
    sizes[0] = n;
    for (int r = 1; r < L; r++) {
        int np = sizes[r - 1] / 2;
        lists[r] = (pm_item *)malloc(sizeof(pm_item) * (n + np));
        int li = 0, pi = 0, o = 0;
        while (li < n || pi < np) {
            int take_leaf;
            if (li >= n) take_leaf = 0;
            else if (pi >= np) take_leaf = 1;
            else {
                uint64_t pw = lists[r - 1][2 * pi].w + lists[r - 1][2 * pi + 1].w;
                take_leaf = (lists[0][li].w <= pw);
            }
            if (take_leaf) {
                lists[r][o++] = lists[0][li++];
            } else {
                pm_item it;
                it.w = lists[r - 1][2 * pi].w + lists[r - 1][2 * pi + 1].w;
                it.leaf = -1;
                it.a = 2 * pi;
                it.b = 2 * pi + 1;
                lists[r][o++] = it;
                pi++;
            }
        }
        sizes[r] = o;
    }
    int *count = (int *)calloc(n, sizeof(int));
    int take = 2 * n - 2;
    int rc = ORC_OK;
    if (sizes[L - 1] < take) rc = ORC_BAD_ARG;
    else
        for (int i = 0; i < take; i++) pm_count(lists, L - 1, i, count);
    for (int i = 0; i < n; i++) len_out[i] = (uint8_t)count[i];
    for (int r = 0; r < L; r++) free(lists[r]);
    free(lists); free(sizes); free(order); free(count);
    return rc;
}

/* ------------------------------------------------------------- codebook */

/* Canonical codes over the coded symbols plus the escape: order by
 * (length, id) with the escape's id 256, first code 0, then
 * code = (previous + 1) << (length - previous length).  Then the 8-bit
 * decode window table and nothing else (reading: canonical form). */
int orc_codebook_assign_codes(orc_codebook *cb)
{
    int ids[257], lens[257], m = 0;
    for (int s = 0; s < 256; s++)
        if (cb->len[s] > 0) { ids[m] = s; lens[m] = cb->len[s]; m++; }
    ids[m] = ORC_ESC; lens[m] = cb->esc_len; m++;
    for (int i = 0; i < m; i++)
        if (lens[i] < 1 || lens[i] > MAXLEN) return ORC_BAD_ARG;
    for (int i = 1; i < m; i++) {
        int vi = ids[i], vl = lens[i], j = i - 1;
        while (j >= 0 && (lens[j] > vl || (lens[j] == vl && ids[j] > vi))) {
            ids[j + 1] = ids[j]; lens[j + 1] = lens[j]; j--;
        }
        ids[j + 1] = vi; lens[j + 1] = vl;
    }
    uint32_t code = 0;
    for (int i = 0; i < m; i++) {
        if (i > 0) code = (code + 1) << (lens[i] - lens[i - 1]);
        if (code >= (1u << lens[i])) return ORC_BAD_ARG; /* Kraft sum above 1 */
        if (ids[i] == ORC_ESC) cb->esc_code = (uint16_t)code;
        else cb->code[ids[i]] = (uint16_t)code;
    }
    for (int v = 0; v < 256; v++) {
        cb->lut_sym[v] = 0xFFFF;
        cb->lut_len[v] = 0;
        for (int i = 0; i < m; i++) {
            int l = lens[i];
            uint32_t c = (ids[i] == ORC_ESC) ? cb->esc_code : cb->code[ids[i]];
            if ((uint32_t)(v >> (MAXLEN - l)) == c) {
                cb->lut_sym[v] = (uint16_t)ids[i];
                cb->lut_len[v] = (uint8_t)l;
            }
        }
    }
    cb->k = m - 1;
    return ORC_OK;
}

/* Code lengths with an escape ([EXP] "In bits": 8-bit cap, one escape prefix
 * for the rare exponents, each escaped exponent followed by an 8-bit literal).
 * Which exponents are "rare" is not printed (reading): symbols of nonzero
 * weight are ranked by (weight descending, exponent ascending); for every
 * k = 1 .. min(255, #nonzero) the top k get codes together with an escape leaf
 * of weight max(1, rest), and the k with the least expected cost
 * sum_K w*len + w_esc*(len_esc + 8) is kept, the smallest k on a tie. */
int orc_codebook_from_weights(const uint64_t w[256], orc_codebook *cb)
{
    memset(cb, 0, sizeof(*cb));
    memcpy(cb->weight, w, sizeof(uint64_t) * 256);
    int rank[256], nz = 0;
    for (int s = 0; s < 256; s++)
        if (w[s] > 0) rank[nz++] = s;
    if (nz == 0) return ORC_BAD_ARG;
    for (int i = 1; i < nz; i++) {
        int v = rank[i], j = i - 1;
        while (j >= 0 && (w[rank[j]] < w[v] || (w[rank[j]] == w[v] && rank[j] > v))) {
            rank[j + 1] = rank[j]; j--;
        }
        rank[j + 1] = v;
    }
    int kmax = nz < 255 ? nz : 255;
    uint64_t best_cost = 0;
    int best_k = 0;
    uint8_t best_len[257];
    for (int k = 1; k <= kmax; k++) {
        uint64_t wl[257];
        int32_t idl[257];
        uint8_t ll[257];
        uint64_t rest = 0;
        for (int i = 0; i < k; i++) { wl[i] = w[rank[i]]; idl[i] = rank[i]; }
        for (int i = k; i < nz; i++) rest += w[rank[i]];
        wl[k] = rest > 0 ? rest : 1;
        idl[k] = ORC_ESC;
        if (orc_package_merge(k + 1, wl, idl, MAXLEN, ll) != ORC_OK) return ORC_BAD_ARG;
        uint64_t cost = wl[k] * (uint64_t)(ll[k] + LITBITS);
        for (int i = 0; i < k; i++) cost += wl[i] * (uint64_t)ll[i];
        if (best_k == 0 || cost < best_cost) {
            best_cost = cost;
            best_k = k;
            memcpy(best_len, ll, k + 1);
        }
    }
    for (int i = 0; i < best_k; i++) cb->len[rank[i]] = best_len[i];
    cb->esc_len = best_len[best_k];
    int rc = orc_codebook_assign_codes(cb);
    if (rc != ORC_OK) return rc;
    /* Model median exponent over the normal range 1..254: the smallest e whose
     * cumulative weight reaches half of that range's total (reading). */
    uint64_t total = 0, cum = 0;
    for (int e = 1; e <= 254; e++) total += w[e];
    cb->median_exp = 127;
    if (total > 0) {
        for (int e = 1; e <= 254; e++) {
            cum += w[e];
            if (2 * cum >= total) { cb->median_exp = e; break; }
        }
    }
    return ORC_OK;
}

/* The codebook is precomputed from the model the user picks, never from the
 * data being coded ([EXP] "In bits"). */
int orc_codebook_build(int model, double scale, double shape, orc_codebook *cb)
{
    double p[256];
    uint64_t w[256];
    int rc = orc_model_pmf(model, scale, shape, p);
    if (rc != ORC_OK) return rc;
    orc_weights_from_pmf(p, w);
    return orc_codebook_from_weights(w, cb);
}

/* A model with a point mass at zero: a fraction zero_frac of the values are
 * exactly zero (ReLU/GELU activations), the rest follow the model.  Not in
 * the pages, which note that the user supplies the distribution and that one
 * which does not fit the tensor raises storage ([EXP] "Read the 3.5x longer
 * context claim carefully"); (reading) mixture pmf
 * p'(e) = (1 - z) p(e) + z [e = 0].  The
 * codebook is marked so that exponent 0 always codes as symbol 0, whatever
 * the shift, and a nonzero exponent that the shift would map onto symbol 0
 * is escaped instead (see symbol_code). */
int orc_codebook_build_zero_atom(int model, double scale, double shape, double zero_frac, orc_codebook *cb)
{
    if (!(zero_frac >= 0.0 && zero_frac < 1.0)) return ORC_BAD_ARG;
    double p[256];
    uint64_t w[256];
    int rc = orc_model_pmf(model, scale, shape, p);
    if (rc != ORC_OK) return rc;
    for (int e = 0; e < 256; e++) {
        double mixed = (1.0 - zero_frac) * p[e];
        if (e == 0) mixed = mixed + zero_frac;
        p[e] = mixed;
    }
    orc_weights_from_pmf(p, w);
    rc = orc_codebook_from_weights(w, cb);
    if (rc == ORC_OK) cb->zero_atom = 1;
    return rc;
}

/* ---------------------------------------------------------- scale shift */

/* The shift that makes the codebook follow the tensor's scale, from at most
 * 4096 sampled values ([EXP] "In bits").  Reading: m = min(n, 4096) samples at
 * positions floor(k*n/m); only normal exponents 1..254 count; the shift is the
 * lower median of their exponents minus the model's median exponent, clamped
 * to [-127, 127]; 0 when no sample counts. */
int orc_shift(const uint16_t *x, uint64_t n, int median_exp)
{
    uint64_t m = n < 4096 ? n : 4096;
    if (m == 0) return 0;
    uint8_t *kept = (uint8_t *)malloc(m);
    uint64_t c = 0;
    for (uint64_t k = 0; k < m; k++) {
        uint8_t e = exponent_of(x[(k * n) / m]);
        if (e >= 1 && e <= 254) kept[c++] = e;
    }
    int delta = 0;
    if (c > 0) {
        for (uint64_t i = 1; i < c; i++) {
            uint8_t v = kept[i];
            uint64_t j = i;
            while (j > 0 && kept[j - 1] > v) { kept[j] = kept[j - 1]; j--; }
            kept[j] = v;
        }
        delta = (int)kept[(c - 1) / 2] - median_exp;
        if (delta > 127) delta = 127;
        if (delta < -127) delta = -127;
    }
    free(kept);
    return delta;
}

/* --------------------------------------------------------------- encode */

/* Symbol of exponent e under shift delta: s = e - delta gets its own code
 * when 0 <= s <= 255 and len[s] > 0; otherwise the escape prefix is followed
 * by the raw exponent e as the 8-bit literal (reading: the literal is e, not
 * s).  Returns the bit count and the code value (right-aligned). */
static int symbol_code(const orc_codebook *cb, int delta, uint8_t e, uint32_t *code)
{
    int s = (int)e - delta;
    if (cb->zero_atom) {
        /* exponent 0 is the unshifted zero atom; symbol 0 belongs to it alone */
        if (e == 0) s = 0;
        else if (s == 0) s = -1;
    }
    if (s >= 0 && s <= 255 && cb->len[s] > 0) {
        *code = cb->code[s];
        return cb->len[s];
    }
    *code = ((uint32_t)cb->esc_code << LITBITS) | e;
    return cb->esc_len + LITBITS;
}

/* Write `bits` bits of `code`, most significant first, at bit position q of
 * stream j's slot in block b.  Word w of stream j sits at
 * slots[(b*W + w)*256 + j]; bit 0 of the stream is bit 31 of word 0
 * (reading: MSB-first, words interleaved across the 256 streams). */
static void put_bits(uint32_t *slots, uint64_t b, uint32_t W, uint32_t j, uint32_t q,
                     uint32_t code, int bits)
{
    for (int t = 0; t < bits; t++) {
        uint32_t bit = (code >> (bits - 1 - t)) & 1u;
        uint32_t pos = q + (uint32_t)t;
        uint64_t word = (b * W + pos / 32) * NSTREAMS + j;
        slots[word] |= bit << (31 - pos % 32);
    }
}

int orc_encode(const uint16_t *x, const orc_codebook *cb, orc_tensor *t)
{
    if (t->block == 0 || t->block % NSTREAMS != 0 || t->slot_words == 0) return ORC_BAD_ARG;
    const uint64_t n = t->n, B = t->block, W = t->slot_words;
    const uint64_t nb = nblocks_of(n, t->block);
    const uint32_t slot_bits = (uint32_t)(32 * W);

    /* step 1: byte split */
    for (uint64_t i = 0; i < n; i++) t->sf[i] = signfrac_of(x[i]);

    /* step 2+3: per block, per stream, greedy fill of the fixed slot */
    memset(t->slots, 0, sizeof(uint32_t) * nb * W * NSTREAMS);
    uint64_t *spill = (uint64_t *)calloc(nb + 1, sizeof(uint64_t));
    for (uint64_t b = 0; b < nb; b++) {
        uint64_t cnt = block_count(n, t->block, b);
        for (uint32_t j = 0; j < NSTREAMS; j++) {
            uint32_t nj = stream_count(cnt, j), used = 0, marker = nj;
            for (uint32_t k = 0; k < nj; k++) {
                uint8_t e = exponent_of(x[b * B + (uint64_t)k * NSTREAMS + j]);
                uint32_t code;
                int bits = symbol_code(cb, t->delta, e, &code);
                /* the first symbol whose whole code does not fit ends the slot */
                if (used + (uint32_t)bits > slot_bits) { marker = k; break; }
                put_bits(t->slots, b, (uint32_t)W, j, used, code, bits);
                used += (uint32_t)bits;
            }
            t->markers[b * NSTREAMS + j] = (uint16_t)marker;
            spill[b] += nj - marker;
        }
    }

    /* step 4: overflow offsets (exclusive prefix over blocks) and bytes in
     * (block, stream, symbol) order (reading) */
    t->blk_off[0] = 0;
    for (uint64_t b = 0; b < nb; b++) t->blk_off[b + 1] = t->blk_off[b] + spill[b];
    t->ovf_used = t->blk_off[nb];
    for (uint64_t b = 0; b < nb; b++) {
        if (t->blk_off[b + 1] > t->ovf_cap) continue; /* block does not fit: nothing written */
        uint64_t cnt = block_count(n, t->block, b), pos = t->blk_off[b];
        for (uint32_t j = 0; j < NSTREAMS; j++) {
            uint32_t nj = stream_count(cnt, j);
            for (uint32_t k = t->markers[b * NSTREAMS + j]; k < nj; k++)
                t->ovf[pos++] = exponent_of(x[b * B + (uint64_t)k * NSTREAMS + j]);
        }
    }
    free(spill);
    return t->ovf_used > t->ovf_cap ? ORC_CAPACITY : ORC_OK;
}

/* --------------------------------------------------------------- decode */

int orc_decode(const orc_tensor *t, const orc_codebook *cb, uint16_t *y)
{
    if (t->block == 0 || t->block % NSTREAMS != 0 || t->slot_words == 0) return ORC_BAD_ARG;
    const uint64_t n = t->n, B = t->block, W = t->slot_words;
    const uint64_t nb = nblocks_of(n, t->block);
    const uint32_t slot_bits = (uint32_t)(32 * W);

    /* code table by (length, value): the symbol, ORC_ESC, or -1 */
    int sym_at[MAXLEN + 1][256];
    for (int l = 0; l <= MAXLEN; l++)
        for (int c = 0; c < 256; c++) sym_at[l][c] = -1;
    for (int s = 0; s < 256; s++)
        if (cb->len[s] > 0) sym_at[cb->len[s]][cb->code[s]] = s;
    sym_at[cb->esc_len][cb->esc_code] = ORC_ESC;

    uint8_t *e = (uint8_t *)malloc(n > 0 ? n : 1);
    int rc = ORC_OK;
    for (uint64_t b = 0; b < nb && rc == ORC_OK; b++) {
        uint64_t cnt = block_count(n, t->block, b);
        uint64_t pos = t->blk_off[b];
        /* a block whose overflow did not fit the buffer cannot be decoded */
        if (t->blk_off[b + 1] > t->ovf_cap) { rc = ORC_CAPACITY; break; }
        for (uint32_t j = 0; j < NSTREAMS && rc == ORC_OK; j++) {
            uint32_t nj = stream_count(cnt, j), marker = t->markers[b * NSTREAMS + j];
            if (marker > nj) { rc = ORC_CORRUPT; break; }
            uint32_t q = 0; /* bit position in the slot */
            for (uint32_t k = 0; k < marker; k++) {
                int l = 0, sym = -1;
                uint32_t c = 0;
                while (sym < 0) {
                    if (l == MAXLEN || q >= slot_bits) { rc = ORC_CORRUPT; break; }
                    uint32_t word = t->slots[(b * W + q / 32) * NSTREAMS + j];
                    c = (c << 1) | ((word >> (31 - q % 32)) & 1u);
                    l++; q++;
                    sym = sym_at[l][c];
                }
                if (rc != ORC_OK) break;
                int ev;
                if (sym == ORC_ESC) {
                    uint32_t lit = 0;
                    for (int i = 0; i < LITBITS; i++) {
                        if (q >= slot_bits) { rc = ORC_CORRUPT; break; }
                        uint32_t word = t->slots[(b * W + q / 32) * NSTREAMS + j];
                        lit = (lit << 1) | ((word >> (31 - q % 32)) & 1u);
                        q++;
                    }
                    ev = (int)lit;
                } else if (cb->zero_atom && sym == 0) {
                    ev = 0;
                } else {
                    ev = sym + t->delta;
                    if (ev < 0 || ev > 255) rc = ORC_CORRUPT;
                }
                if (rc != ORC_OK) break;
                e[b * B + (uint64_t)k * NSTREAMS + j] = (uint8_t)ev;
            }
            for (uint32_t k = marker; k < nj && rc == ORC_OK; k++) {
                if (pos >= t->blk_off[b + 1] || pos >= t->ovf_cap) { rc = ORC_CORRUPT; break; }
                e[b * B + (uint64_t)k * NSTREAMS + j] = t->ovf[pos++];
            }
        }
        if (rc == ORC_OK && pos != t->blk_off[b + 1]) rc = ORC_CORRUPT;
    }
    if (rc == ORC_OK)
        for (uint64_t i = 0; i < n; i++) y[i] = join_bf16(t->sf[i], e[i]);
    free(e);
    return rc;
}

/* ------------------------------------------------------------------ SGD */

/* float32 -> BF16, round to nearest, ties to even, subnormals kept.  NaN
 * becomes the canonical quiet NaN 0x7FC0 (reading: keeps results independent
 * of the platform's NaN payload rules). */
uint16_t orc_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

static float bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* W <- W - eta*M on compressed W and M ([EXP] "Training adds a second
 * problem").  Arithmetic in float32: the product eta*m is rounded, then the
 * difference is rounded (two roundings, no fused multiply-add), then rounded
 * to BF16.  The new W is coded with W's codebook and W's stored shift (the
 * codebook stays fixed during training). */
int orc_sgd_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                 const orc_codebook *cbM, float eta, orc_tensor *W_out)
{
    if (W->n != M->n || W_out->n != W->n || W_out->block != W->block ||
        W_out->slot_words != W->slot_words)
        return ORC_BAD_ARG;
    uint64_t n = W->n;
    uint16_t *w = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    uint16_t *m = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    int rc = orc_decode(W, cbW, w);
    if (rc == ORC_OK) rc = orc_decode(M, cbM, m);
    if (rc == ORC_OK) {
        for (uint64_t i = 0; i < n; i++) {
            float wf = bf16_value(w[i]);
            float mf = bf16_value(m[i]);
            float prod = eta * mf;
            float r = wf - prod;
            w[i] = orc_bf16_rne(r);
        }
        W_out->delta = W->delta;
        rc = orc_encode(w, cbW, W_out);
    }
    free(w);
    free(m);
    return rc;
}

/* SGD with momentum on compressed W and M, with a dense BF16 gradient g
 * ([EXP] "Jargon", entry "Optimizer state": the momentum buffer of SGD with
 * momentum is the example of optimizer state; [ABS]: optimizer states are
 * kept compressed; [EXP] "Training adds a second problem": the update reads
 * and rewrites the compressed tensors).  The pages print no update rule;
 * (reading) the common heavy-ball form without dampening or Nesterov term:
 *   M' = bf16( fl32( fl32(mu*m) + g ) )
 *   W' = bf16( fl32( w - fl32(eta*M') ) )
 * Every float32 operation is rounded on its own (no fused multiply-add), and
 * the weight update uses the new momentum as stored (BF16).  Each output is
 * coded with its own input's codebook and stored shift.  rc[0] and rc[1] get
 * the status of W' and M'. */
int orc_sgd_momentum_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                          const orc_codebook *cbM, const uint16_t *g, float eta, float mu,
                          orc_tensor *W_out, orc_tensor *M_out, int rc[2])
{
    rc[0] = rc[1] = ORC_BAD_ARG;
    if (W->n != M->n || W_out->n != W->n || M_out->n != M->n || W_out->block != W->block ||
        W_out->slot_words != W->slot_words || M_out->block != M->block ||
        M_out->slot_words != M->slot_words)
        return ORC_BAD_ARG;
    uint64_t n = W->n;
    uint16_t *w = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    uint16_t *m = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    int st = orc_decode(W, cbW, w);
    if (st == ORC_OK) st = orc_decode(M, cbM, m);
    if (st == ORC_OK) {
        for (uint64_t i = 0; i < n; i++) {
            float scaled = mu * bf16_value(m[i]);
            float sum = scaled + bf16_value(g[i]);
            m[i] = orc_bf16_rne(sum);
            float step = eta * bf16_value(m[i]);
            float r = bf16_value(w[i]) - step;
            w[i] = orc_bf16_rne(r);
        }
        W_out->delta = W->delta;
        M_out->delta = M->delta;
        rc[0] = orc_encode(w, cbW, W_out);
        rc[1] = orc_encode(m, cbM, M_out);
        st = rc[0] != ORC_OK ? rc[0] : rc[1];
    } else {
        rc[0] = rc[1] = st;
    }
    free(w);
    free(m);
    return st;
}

/* Constants of one AdamW step, computed once in double from the
 * hyper-parameters and rounded to float (reading: the step size and the
 * second-moment correction fold the bias corrections of step t). */
void orc_adamw_constants(double lr, double beta1, double beta2, double eps, double weight_decay,
                         uint32_t t, float k[8])
{
    k[0] = (float)beta1;
    k[1] = (float)(1.0 - beta1);
    k[2] = (float)beta2;
    k[3] = (float)(1.0 - beta2);
    k[4] = (float)(lr / (1.0 - pow(beta1, (double)t)));           /* step size */
    k[5] = (float)(1.0 / sqrt(1.0 - pow(beta2, (double)t)));      /* 1/sqrt(1 - beta2^t) */
    k[6] = (float)eps;
    k[7] = (float)(lr * weight_decay);                            /* decoupled decay */
}

/* AdamW on compressed W, M (first moment) and V (second moment) with a
 * dense BF16 gradient g ([EXP] "Jargon", entry "Optimizer state": optimizer
 * states such as momentum buffers are the same size as the weights; [ABS]:
 * optimizer states are kept compressed).  The pages print no optimizer;
 * (reading) the AdamW update with decoupled weight decay, every float32
 * operation rounded on its own (no fused multiply-add), k from
 * orc_adamw_constants:
 *   M' = bf16( k0*m + k1*g )
 *   V' = bf16( k2*v + k3*(g*g) )
 *   W' = bf16( (w - k7*w) - (k4*M') / (sqrt(V')*k5 + k6) )
 * with the weight update taking M' and V' as stored (BF16); sqrt and the
 * division are the correctly rounded IEEE operations.  Each output is coded
 * with its input's codebook and stored shift.  rc[0..2] get the status of
 * W', M', V'. */
int orc_adamw_step(const orc_tensor *W, const orc_codebook *cbW, const orc_tensor *M,
                   const orc_codebook *cbM, const orc_tensor *V, const orc_codebook *cbV,
                   const uint16_t *g, const float k[8], orc_tensor *W_out, orc_tensor *M_out,
                   orc_tensor *V_out, int rc[3])
{
    rc[0] = rc[1] = rc[2] = ORC_BAD_ARG;
    const orc_tensor *in[3] = {W, M, V};
    orc_tensor *out[3] = {W_out, M_out, V_out};
    for (int i = 0; i < 3; i++)
        if (in[i]->n != W->n || out[i]->n != W->n || out[i]->block != in[i]->block ||
            out[i]->slot_words != in[i]->slot_words)
            return ORC_BAD_ARG;
    uint64_t n = W->n;
    uint16_t *w = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    uint16_t *m = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    uint16_t *v = (uint16_t *)malloc(2 * (n > 0 ? n : 1));
    int st = orc_decode(W, cbW, w);
    if (st == ORC_OK) st = orc_decode(M, cbM, m);
    if (st == ORC_OK) st = orc_decode(V, cbV, v);
    if (st == ORC_OK) {
        for (uint64_t i = 0; i < n; i++) {
            float gf = bf16_value(g[i]);
            float a1 = k[0] * bf16_value(m[i]);
            float a2 = k[1] * gf;
            float ms = a1 + a2;
            m[i] = orc_bf16_rne(ms);
            float b1 = k[2] * bf16_value(v[i]);
            float gg = gf * gf;
            float b2 = k[3] * gg;
            float vs = b1 + b2;
            v[i] = orc_bf16_rne(vs);
            float root = sqrtf(bf16_value(v[i]));
            float scaled = root * k[5];
            float den = scaled + k[6];
            float num = k[4] * bf16_value(m[i]);
            float upd = num / den;
            float wf = bf16_value(w[i]);
            float decay = k[7] * wf;
            float wd = wf - decay;
            float r = wd - upd;
            w[i] = orc_bf16_rne(r);
        }
        W_out->delta = W->delta;
        M_out->delta = M->delta;
        V_out->delta = V->delta;
        rc[0] = orc_encode(w, cbW, W_out);
        rc[1] = orc_encode(m, cbM, M_out);
        rc[2] = orc_encode(v, cbV, V_out);
        st = rc[0] != ORC_OK ? rc[0] : (rc[1] != ORC_OK ? rc[1] : rc[2]);
    } else {
        rc[0] = rc[1] = rc[2] = st;
    }
    free(w);
    free(m);
    free(v);
    return st;
}
