// Host-side codebook construction for liblct (lct_codebook_build).
//
// [EXP] "In bits": the exponent byte is Huffman-coded with codes capped at
// 8 bits; rare exponents share one escape prefix followed by an 8-bit
// literal; the codebook is precomputed from a distribution the user picks.
//
// Built with floating-point contraction off: the bucket masses below must be
// the same doubles on every host.
#include <algorithm>
#include <array>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/lct.h"
#include "internal.h"

namespace lct {
namespace {

// Model cdf of |x|: half-normal erf(t / (sigma sqrt 2)), exponential
// 1 - exp(-t/b), Lomax 1 - (1 + t/s)^-alpha.
double cdf_abs(int model, double scale, double shape, double t)
{
    if (std::isinf(t)) return 1.0;
    if (model == LCT_MODEL_GAUSSIAN) return std::erf(t / (scale * std::sqrt(2.0)));
    if (model == LCT_MODEL_LAPLACE) return 1.0 - std::exp(-t / scale);
    return 1.0 - std::pow(1.0 + t / scale, -shape);
}

// Integer weight of every biased-exponent bucket: mass * 2^40, rounded.
// With a point mass at zero the model's masses are scaled by (1 - zero) and
// the point mass is added to bucket 0.
std::array<uint64_t, 256> bucket_weights(int model, double scale, double shape, bool atom, double zero)
{
    std::array<uint64_t, 256> w{};
    for (int e = 0; e < 255; ++e) {
        const double lo = e == 0 ? 0.0 : std::ldexp(1.0, e - 127);
        const double hi = e == 254 ? HUGE_VAL : std::ldexp(1.0, e - 126);
        double p = cdf_abs(model, scale, shape, hi) - cdf_abs(model, scale, shape, lo);
        if (atom) {
            p = (1.0 - zero) * p;
            if (e == 0) p = p + zero;
        }
        w[e] = static_cast<uint64_t>(std::llround(std::ldexp(p, 40)));
    }
    w[255] = 0;
    return w;
}

struct Leaf {
    uint64_t weight;
    int id;  // exponent symbol, or 256 for the escape
};

// Length-limited code lengths by package-merge over `leaves` (already sorted
// by weight, then id), cap L.  A node is a leaf or a pair of nodes of the
// previous level; equal weights put the leaf first.  The first 2n-2 nodes of
// the last level are selected, and selection flows down level by level; a
// leaf's length is the number of levels where it is selected.
std::vector<int> package_merge(const std::vector<Leaf> &leaves, int L)
{
    const int n = static_cast<int>(leaves.size());
    struct Node {
        uint64_t weight;
        int leaf;   // index into leaves, or -1
        int child;  // first of the two children in the previous level
    };
    std::vector<std::vector<Node>> level(L);
    level[0].reserve(n);
    for (int i = 0; i < n; ++i) level[0].push_back({leaves[i].weight, i, -1});
    for (int r = 1; r < L; ++r) {
        const std::vector<Node> &prev = level[r - 1];
        const int pairs = static_cast<int>(prev.size()) / 2;
        std::vector<Node> &cur = level[r];
        cur.reserve(n + pairs);
        int i = 0, p = 0;
        while (i < n || p < pairs) {
            const uint64_t pw = p < pairs ? prev[2 * p].weight + prev[2 * p + 1].weight : 0;
            if (p >= pairs || (i < n && leaves[i].weight <= pw)) {
                cur.push_back({leaves[i].weight, i, -1});
                ++i;
            } else {
                cur.push_back({pw, -1, 2 * p});
                ++p;
            }
        }
    }
    std::vector<int> len(n, 0);
    std::vector<char> sel(level[L - 1].size(), 0);
    const size_t take = static_cast<size_t>(2 * n - 2);
    if (level[L - 1].size() < take) return {};
    std::fill(sel.begin(), sel.begin() + take, 1);
    for (int r = L - 1; r >= 0; --r) {
        std::vector<char> below(r > 0 ? level[r - 1].size() : 0, 0);
        for (size_t k = 0; k < level[r].size(); ++k) {
            if (!sel[k]) continue;
            const Node &nd = level[r][k];
            if (nd.leaf >= 0) {
                ++len[nd.leaf];
            } else {
                below[nd.child] = 1;
                below[nd.child + 1] = 1;
            }
        }
        sel.swap(below);
    }
    return len;
}

uint32_t fnv1a(const lct_codebook &cb)
{
    uint32_t h = 2166136261u;
    auto mix = [&h](uint8_t b) {
        h ^= b;
        h *= 16777619u;
    };
    for (int s = 0; s < 256; ++s) mix(cb.len[s]);
    for (int s = 0; s < 256; ++s) mix(cb.code[s]);
    mix(cb.esc_len);
    mix(cb.esc_code);
    mix(static_cast<uint8_t>(cb.zero_atom));
    return h;
}

}  // namespace

uint32_t codebook_hash(const lct_codebook &cb) { return fnv1a(cb); }

// A codebook is usable when every length is within the cap, the codes with
// the escape form a complete prefix code, and the window table agrees.
bool codebook_valid(const lct_codebook &cb)
{
    if (cb.esc_len < 1 || cb.esc_len > LCT_MAX_CODE_BITS || cb.zero_atom > 1) return false;
    uint32_t kraft = 1u << (LCT_MAX_CODE_BITS - cb.esc_len);
    for (int s = 0; s < 256; ++s) {
        if (cb.len[s] > LCT_MAX_CODE_BITS) return false;
        if (cb.len[s]) kraft += 1u << (LCT_MAX_CODE_BITS - cb.len[s]);
    }
    if (kraft != 256u) return false;
    for (int v = 0; v < 256; ++v) {
        const int sym = cb.dec[v] & 0x1FF, l = cb.dec[v] >> 12;
        if (l < 1 || l > 8 || sym > 256) return false;
        const int code = sym == 256 ? cb.esc_code : cb.code[sym];
        const int clen = sym == 256 ? cb.esc_len : cb.len[sym];
        if (clen != l || (v >> (8 - l)) != code) return false;
    }
    return cb.hash == fnv1a(cb);
}

}  // namespace lct

namespace lct {
namespace {

lct_status build(int model, double scale, double shape, bool atom, double zero, lct_codebook *out)
{
    if (!out) return LCT_ERR_INVALID_ARG;
    if (model < LCT_MODEL_GAUSSIAN || model > LCT_MODEL_POWERLAW) return LCT_ERR_INVALID_ARG;
    if (!(scale > 0.0) || std::isinf(scale)) return LCT_ERR_INVALID_ARG;
    if (model == LCT_MODEL_POWERLAW && (!(shape > 0.0) || std::isinf(shape)))
        return LCT_ERR_INVALID_ARG;
    if (atom && !(zero >= 0.0 && zero < 1.0)) return LCT_ERR_INVALID_ARG;

    const std::array<uint64_t, 256> w = bucket_weights(model, scale, shape, atom, zero);

    // Buckets of nonzero weight, heaviest first (smaller exponent on ties).
    std::vector<int> ranked;
    for (int e = 0; e < 256; ++e)
        if (w[e]) ranked.push_back(e);
    if (ranked.empty()) return LCT_ERR_INVALID_ARG;
    std::stable_sort(ranked.begin(), ranked.end(),
                     [&w](int a, int b) { return w[a] > w[b] || (w[a] == w[b] && a < b); });

    // Suffix sums give the escape weight of every split point.
    const int nz = static_cast<int>(ranked.size());
    std::vector<uint64_t> tail(nz + 1, 0);
    for (int i = nz - 1; i >= 0; --i) tail[i] = tail[i + 1] + w[ranked[i]];

    const int kmax = std::min(nz, 255);
    uint64_t best = UINT64_MAX;
    int best_k = 0;
    std::vector<int> best_len;
    for (int k = 1; k <= kmax; ++k) {
        std::vector<Leaf> leaves;
        leaves.reserve(k + 1);
        for (int i = 0; i < k; ++i) leaves.push_back({w[ranked[i]], ranked[i]});
        leaves.push_back({std::max<uint64_t>(tail[k], 1), 256});
        std::sort(leaves.begin(), leaves.end(), [](const Leaf &a, const Leaf &b) {
            return a.weight < b.weight || (a.weight == b.weight && a.id < b.id);
        });
        const std::vector<int> len = package_merge(leaves, LCT_MAX_CODE_BITS);
        if (len.empty()) return LCT_ERR_INVALID_ARG;
        uint64_t cost = 0;
        std::vector<int> by_id(257, 0);
        for (int i = 0; i <= k; ++i) {
            const int extra = leaves[i].id == 256 ? LCT_LITERAL_BITS : 0;
            cost += leaves[i].weight * static_cast<uint64_t>(len[i] + extra);
            by_id[leaves[i].id] = len[i];
        }
        if (cost < best) {
            best = cost;
            best_k = k;
            best_len = by_id;
        }
    }

    lct_codebook cb;
    std::memset(&cb, 0, sizeof(cb));
    for (int i = 0; i < best_k; ++i) cb.len[ranked[i]] = static_cast<uint8_t>(best_len[ranked[i]]);
    cb.esc_len = static_cast<uint8_t>(best_len[256]);
    cb.nsym = static_cast<uint16_t>(best_k);

    // Canonical codes: by (length, id), escape id 256.
    std::vector<std::pair<int, int>> order;  // (length, id)
    for (int s = 0; s < 256; ++s)
        if (cb.len[s]) order.emplace_back(cb.len[s], s);
    order.emplace_back(cb.esc_len, 256);
    std::sort(order.begin(), order.end());
    uint32_t next = 0;
    int prev_len = order.front().first;
    for (size_t i = 0; i < order.size(); ++i) {
        const int l = order[i].first, id = order[i].second;
        if (i) next = (next + 1) << (l - prev_len);
        prev_len = l;
        if (next >= (1u << l)) return LCT_ERR_INVALID_ARG;
        if (id == 256)
            cb.esc_code = static_cast<uint8_t>(next);
        else
            cb.code[id] = static_cast<uint8_t>(next);
        // every 8-bit window that starts with this code
        const uint32_t first = next << (8 - l), span = 1u << (8 - l);
        for (uint32_t v = first; v < first + span; ++v)
            cb.dec[v] = static_cast<uint16_t>(id | (l << 12));
    }

    // Median biased exponent of the model over the normal range.
    uint64_t total = 0;
    for (int e = 1; e <= 254; ++e) total += w[e];
    cb.median_exp = 127;
    if (total) {
        uint64_t run = 0;
        for (int e = 1; e <= 254; ++e) {
            run += w[e];
            if (run * 2 >= total) {
                cb.median_exp = e;
                break;
            }
        }
    }
    cb.model = model;
    cb.scale = scale;
    cb.shape = model == LCT_MODEL_POWERLAW ? shape : 0.0;
    cb.zero_frac = atom ? zero : 0.0;
    cb.zero_atom = atom ? 1u : 0u;
    cb.hash = fnv1a(cb);
    *out = cb;
    return LCT_OK;
}

}  // namespace
}  // namespace lct

extern "C" lct_status lct_codebook_build(int model, double scale, double shape, lct_codebook *out)
{
    return lct::build(model, scale, shape, false, 0.0, out);
}

extern "C" lct_status lct_codebook_build_zero_atom(int model, double scale, double shape, double zero_frac,
                                                   lct_codebook *out)
{
    return lct::build(model, scale, shape, true, zero_frac, out);
}
