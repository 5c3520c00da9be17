"""Pins for the CPU oracle: each test ties it to something other than itself --
numbers the LCT pages print, closed forms, library distributions, brute force
on tiny inputs, a hand-worked layout, invariants of the format.

Pages (by title): [ABS] "LCT: Losslessly Compressed Tensors with GPU friendly
execution for Training", abstract; [EXP] "LCT paper -- Lossless Huffman coding
of BF16 training tensors -- What does it mean?", paragraphs named by their
first words.
"""
import heapq
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from lossless_bf16_tensor_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
FIG = json.load(open(os.path.join(GOLD, "pages_figures.json")))["figures"]

MODELS = [(0, 0.02, 0.0), (0, 1.0, 0.0), (1, 0.01, 0.0), (1, 3e-5, 0.0), (2, 1e-3, 3.0), (2, 0.5, 1.5)]


# ------------------------------------------------------------- geometry

def test_geometry_matches_pages(orc):
    """Block sizes and the CLEAN slot against [EXP] 'Compressing is easy' and
    'Here is the idealized arithmetic'."""
    b0, w0 = orc.geometry(orc.CLEAN)
    b1, _ = orc.geometry(orc.MEDIUM)
    b2, _ = orc.geometry(orc.HIGH)
    assert b0 == FIG["block_clean"]["value"]
    assert b1 == b2 == FIG["block_medium_high"]["value"]
    slot_bytes = 4 * w0
    # allocated exponent bits in CLEAN within the pages' 3.0-3.2
    alloc = 8.0 * slot_bytes * FIG["streams_per_block"]["value"] / b0
    lo, hi = FIG["allocated_exponent_bits_clean"]["lo"], FIG["allocated_exponent_bits_clean"]["hi"]
    assert lo <= alloc <= hi
    # payload ratio of a CLEAN block = the pages' 1.4382x bound, ~11.1 bits/value
    ratio = 2.0 * b0 / (b0 + FIG["streams_per_block"]["value"] * slot_bytes)
    assert round(ratio, 4) == FIG["clean_ratio_bound"]["value"]
    assert round(8 + alloc, 1) == FIG["clean_ratio_bound"]["bits_per_value"]
    # the best-case figure is 16 bits over 8 + 3
    assert round(16 / FIG["best_ratio"]["bits_per_value"], 3) == FIG["best_ratio"]["value"]


# ---------------------------------------------------------------- model

def _bucket_edges():
    lo = np.array([0.0] + [2.0 ** (e - 127) for e in range(1, 255)])
    hi = np.array([2.0 ** (e - 126) for e in range(0, 254)] + [np.inf])
    return lo, hi


@pytest.mark.parametrize("model,scale,shape", MODELS)
def test_pmf_matches_scipy_distributions(orc, model, scale, shape):
    """Bucket masses of |x| from scipy's half-normal / exponential / Lomax."""
    from scipy import stats
    dist = {0: stats.halfnorm(scale=scale), 1: stats.expon(scale=scale),
            2: stats.lomax(c=shape if shape else 1.0, scale=scale)}[model]
    lo, hi = _bucket_edges()
    ref = dist.cdf(hi) - dist.cdf(lo)
    p = orc.model_pmf(model, scale, shape)
    assert p[255] == 0.0
    np.testing.assert_allclose(p[:255], ref, rtol=0, atol=2e-13)
    assert abs(p.sum() - 1.0) < 1e-12


@pytest.mark.parametrize("model,shape", [(0, 0.0), (1, 0.0), (2, 3.0)])
def test_pmf_scale_doubling_shifts_exponent(orc, model, shape):
    """Doubling the scale moves every interior bucket up by one, exactly."""
    p1 = orc.model_pmf(model, 0.01, shape)
    p2 = orc.model_pmf(model, 0.02, shape)
    assert np.array_equal(p2[2:254], p1[1:253])


def _entropy(p):
    q = p[p > 0]
    return float(-(q * np.log2(q)).sum())


def test_entropy_closed_forms(orc):
    """Differential entropy of log2|x| (scale-free): Gaussian
    [1/2 ln(pi e/2) + (gamma + ln 2)/2 - ln ln 2]/ln 2, Laplace
    [1 + gamma - ln ln 2]/ln 2; unit-width exponent buckets stay close."""
    g = 0.5772156649015329
    h_gauss = (0.5 * math.log(math.pi * math.e / 2) + (g + math.log(2)) / 2 - math.log(math.log(2))) / math.log(2)
    h_lap = (1 + g - math.log(math.log(2))) / math.log(2)
    assert abs(h_gauss - 2.4922) < 1e-3 and abs(h_lap - 2.8042) < 1e-3
    assert abs(_entropy(orc.model_pmf(0, 0.02, 0)) - h_gauss) < 0.06
    assert abs(_entropy(orc.model_pmf(1, 0.01, 0)) - h_lap) < 0.06


def test_ideal_cost_in_pages_range(orc):
    """[EXP] 'In bits': ideal exponent cost about 2.5-3.1 bits for the three models."""
    lo, hi = FIG["ideal_exponent_bits"]["lo"], FIG["ideal_exponent_bits"]["hi"]
    for model, scale, shape in [(0, 0.02, 0.0), (1, 0.01, 0.0), (2, 1e-3, 3.0)]:
        h = _entropy(orc.model_pmf(model, scale, shape))
        assert lo - 0.05 <= h <= hi + 0.05, (model, h)


def test_pmf_rejects_bad_parameters(orc):
    for args in [(0, 0.0, 0.0), (1, -1.0, 0.0), (2, 1.0, 0.0), (0, float("inf"), 0.0), (3, 1.0, 1.0)]:
        with pytest.raises(ValueError):
            orc.model_pmf(*args)


# ------------------------------------------------------ package-merge

def _brute_min_cost(w, L):
    n, best = len(w), None
    for ls in itertools.product(range(1, L + 1), repeat=n):
        if sum(2.0 ** -l for l in ls) <= 1.0 + 1e-12:
            c = sum(a * b for a, b in zip(w, ls))
            best = c if best is None else min(best, c)
    return best


def test_package_merge_equals_brute_force(orc):
    rng = np.random.default_rng(11)
    for trial in range(60):
        n = int(rng.integers(2, 8))
        L = int(rng.integers(max(1, math.ceil(math.log2(n))), 5))
        w = rng.integers(1, 50, size=n) if trial % 2 else rng.integers(1, 4, size=n) ** rng.integers(1, 6, size=n)
        lens = orc.package_merge(w, L)
        assert lens.max() <= L
        assert sum(2.0 ** -int(l) for l in lens) == 1.0
        assert int((w * lens).sum()) == _brute_min_cost(list(map(int, w)), L), (w, L, lens)


def _huffman_cost(w):
    h = [(int(x), i) for i, x in enumerate(w)]
    heapq.heapify(h)
    cost, k = 0, len(w)
    while len(h) > 1:
        a, b = heapq.heappop(h), heapq.heappop(h)
        cost += a[0] + b[0]
        heapq.heappush(h, (a[0] + b[0], k))
        k += 1
    return cost


def test_package_merge_without_binding_cap_is_huffman(orc):
    rng = np.random.default_rng(12)
    for _ in range(40):
        n = int(rng.integers(2, 12))
        w = rng.integers(1, 1000, size=n)
        lens = orc.package_merge(w, max(1, n - 1))
        assert int((w * lens).sum()) == _huffman_cost(w)


def test_without_escape_all_256_codes_are_8_bits(orc):
    """[EXP] 'In bits': covering all 256 exponents under an 8-bit cap forces
    every code to length 8."""
    w = np.random.default_rng(13).integers(1, 1 << 40, size=256)
    assert (orc.package_merge(w, 8) == 8).all()


# ------------------------------------------------------------ codebook

def _check_codebook(cb):
    lens = cb.lengths()
    codes = cb.codes()
    leaves = [(int(lens[s]), int(codes[s]), s) for s in range(256) if lens[s] > 0]
    leaves.append((int(cb.esc_len), int(cb.esc_code), 256))
    assert all(1 <= l <= 8 for l, _, _ in leaves)
    assert sum(1 << (8 - l) for l, _, _ in leaves) == 256  # Kraft equality
    # prefix-free, and the 8-bit window table agrees with it
    for (l1, c1, s1), (l2, c2, s2) in itertools.permutations(leaves, 2):
        if l1 <= l2:
            assert (c2 >> (l2 - l1)) != c1, (s1, s2)
    for v in range(256):
        hits = [(s, l) for l, c, s in leaves if (v >> (8 - l)) == c]
        assert hits == [(cb.lut_sym[v], cb.lut_len[v])]
    # canonical: ordered by (length, id), codes increase
    order = sorted(leaves, key=lambda t: (t[0], t[2]))
    vals = [c << (8 - l) for l, c, _ in order]
    assert vals == sorted(vals) and len(set(vals)) == len(vals)


@pytest.mark.parametrize("model,scale,shape", MODELS)
def test_codebook_is_complete_capped_prefix_code(orc, model, scale, shape):
    cb = orc.codebook_build(model, scale, shape)
    _check_codebook(cb)
    assert 1 <= cb.k <= 255


@pytest.mark.parametrize("model,scale,shape", MODELS)
def test_codebook_expected_length_near_entropy(orc, model, scale, shape):
    p = orc.model_pmf(model, scale, shape)
    cb = orc.codebook_build(model, scale, shape)
    lens = cb.lengths().astype(float)
    coded = lens > 0
    el = float((p[coded] * lens[coded]).sum() + p[~coded].sum() * (cb.esc_len + 8))
    h = _entropy(p)
    assert h <= el <= h + 0.2


@pytest.mark.parametrize("model,scale,shape", MODELS)
def test_median_exponent_is_model_median(orc, model, scale, shape):
    from scipy import stats
    dist = {0: stats.halfnorm(scale=scale), 1: stats.expon(scale=scale),
            2: stats.lomax(c=shape if shape else 1.0, scale=scale)}[model]
    q = dist.ppf(0.5)
    assert orc.codebook_build(model, scale, shape).median_exp == math.floor(math.log2(q)) + 127


def test_codebook_from_flat_weights(orc):
    """Flat weights over 4 symbols: the escape is never worth its literal, so
    the top symbols get codes; the result is still a complete code."""
    w = np.zeros(256, np.uint64)
    w[[10, 11, 12, 13]] = 1 << 30
    cb = orc.codebook_from_weights(w)
    _check_codebook(cb)
    assert cb.k == 4 and set(np.nonzero(cb.lengths())[0]) == {10, 11, 12, 13}


# ------------------------------------------------- escape-set choice

def _exact_capped_cost(weights, L=8):
    """Least sum(w * len) over prefix codes with every length <= L, by
    exhaustive search over how many leaves take each length 1..L (the
    heaviest leaves take the shortest lengths, which is optimal by
    rearrangement); no Huffman or package-merge step is used."""
    ws = sorted(weights, reverse=True)
    m = len(ws)
    pre = [0]
    for w in ws:
        pre.append(pre[-1] + w)
    best = [None]

    def rec(length, start, room, cost):  # room: Kraft budget in units of 2^-L
        if start == m:
            if best[0] is None or cost < best[0]:
                best[0] = cost
            return
        if length > L or (best[0] is not None and cost + length * (pre[m] - pre[start]) >= best[0]):
            return
        unit = 1 << (L - length)
        for c in range(min(m - start, room // unit), -1, -1):
            rec(length + 1, start + c, room - c * unit, cost + length * (pre[start + c] - pre[start]))

    rec(1, 0, 1 << L, 0)
    return best[0]


def _escape_cost(coded_weights, escaped_weights, L=8):
    """The code over the coded symbols plus one escape leaf whose weight is
    the escaped symbols' total (at least 1); every escape also pays the
    8-bit raw exponent ([EXP] 'In bits')."""
    w_esc = max(1, sum(escaped_weights))
    return _exact_capped_cost(list(coded_weights) + [w_esc], L) + 8 * w_esc


def _oracle_cost(cb, w):
    lens = cb.lengths()
    coded = lens > 0
    w_esc = max(1, int(w[~coded].sum()))
    return int((w[coded].astype(object) * lens[coded].astype(object)).sum()) + w_esc * (int(cb.esc_len) + 8)


def _skewed_weights(rng, nsym):
    """nsym nonzero exponents with a fast-decaying tail, so that the 8-bit
    cap binds and escaping the rarest exponents can pay."""
    w = np.zeros(256, np.uint64)
    exps = rng.choice(np.arange(1, 255), size=nsym, replace=False)
    ratio = rng.uniform(1.6, 3.5)
    vals = [max(1, int(rng.integers(1, 1 << 20) * ratio ** -i * (1 << 20))) for i in range(nsym)]
    rng.shuffle(vals)
    w[exps] = vals
    return w


def test_escape_set_is_optimal_over_every_subset(orc):
    """[EXP] 'In bits': rare exponents share one escape prefix.  Over every
    subset of 9-11 exponents that could be escaped and every length vector,
    no codebook is cheaper than the oracle's, and the oracle's cost is
    reached: this pins the escape weight, its 8-bit literal and the choice
    of how many exponents get codes."""
    rng = np.random.default_rng(31)
    escaped_somewhere = 0
    for trial in range(12):
        nsym = int(rng.integers(9, 12))
        w = _skewed_weights(rng, nsym)
        cb = orc.codebook_from_weights(w)
        nz = [int(v) for v in w[w > 0]]
        best = None
        for r in range(1, nsym + 1):
            for coded in itertools.combinations(range(nsym), r):
                rest = [nz[i] for i in range(nsym) if i not in coded]
                c = _escape_cost([nz[i] for i in coded], rest)
                best = c if best is None else min(best, c)
        assert _oracle_cost(cb, w) == best, (trial, nz)
        escaped_somewhere += int(cb.k < nsym)
    assert escaped_somewhere >= 3  # the cases do exercise the escape


def test_escape_set_is_the_smallest_optimal_prefix_of_the_ranking(orc):
    """The coded exponents are the k heaviest (weight descending, exponent
    ascending), and k is the smallest count reaching the least cost (the
    reading on ties), over alphabets of up to 16 exponents."""
    rng = np.random.default_rng(32)
    for trial in range(20):
        nsym = int(rng.integers(9, 17))
        w = _skewed_weights(rng, nsym)
        if trial % 4 == 0:  # equal weights in the tail: ties between prefixes
            tail = np.argsort(w)[-nsym:][: nsym // 2]
            w[tail] = w[tail].min()
        cb = orc.codebook_from_weights(w)
        order = sorted(np.nonzero(w)[0], key=lambda e: (-int(w[e]), int(e)))
        costs = [_escape_cost([int(w[e]) for e in order[:k]], [int(w[e]) for e in order[k:]])
                 for k in range(1, nsym + 1)]
        k_best = 1 + costs.index(min(costs))
        assert cb.k == k_best, (trial, costs)
        assert set(np.nonzero(cb.lengths())[0]) == set(order[:k_best])
        assert _oracle_cost(cb, w) == min(costs)


# Exponent weights for which coding k or k+1 (or k+2) exponents costs exactly
# the same (found by a search over power-of-two-like weights; the tied counts
# are recomputed by the reference below, not taken from the oracle).
TIED_WEIGHTS = [
    [131072, 65536, 8192, 4096, 512, 256, 32, 8, 4, 1],
    [16777216, 4194304, 524288, 131072, 32768, 8192, 2048, 512, 256, 64, 8, 2, 1],
    [1024, 1024, 512, 128, 128, 32, 16, 16, 8, 2, 1, 1],
    [2048, 2048, 1024, 512, 128, 64, 32, 32, 16, 4, 4, 2, 1],
    [1024, 512, 512, 256, 128, 32, 16, 16, 8, 4, 2, 1],
]


@pytest.mark.parametrize("vals", TIED_WEIGHTS)
def test_escape_set_ties_go_to_the_fewest_codes(orc, vals):
    """When several counts of coded exponents reach the least cost, the
    oracle codes the fewest of them (the reading on ties)."""
    w = np.zeros(256, np.uint64)
    exps = np.arange(40, 40 + len(vals))
    w[exps] = vals
    order = sorted(np.nonzero(w)[0], key=lambda e: (-int(w[e]), int(e)))
    costs = [_escape_cost([int(w[e]) for e in order[:k]], [int(w[e]) for e in order[k:]])
             for k in range(1, len(vals) + 1)]
    tied = [k + 1 for k, c in enumerate(costs) if c == min(costs)]
    assert len(tied) >= 2
    cb = orc.codebook_from_weights(w)
    assert cb.k == tied[0] and _oracle_cost(cb, w) == min(costs)


# ---------------------------------------------------------------- shift

def _with_exponents(exps, sf=0):
    e = np.asarray(exps, dtype=np.uint16)
    return ((sf & 0x80) << 8) | (e << 7) | (sf & 0x7F)


def test_shift_hand_examples(orc):
    """Lower median of the normal-range sampled exponents minus the model median."""
    assert orc.shift(_with_exponents([120, 0, 125, 118, 255]), 118) == 2   # kept 118,120,125
    assert orc.shift(_with_exponents([118, 120, 122, 125]), 120) == 0      # lower median 120
    assert orc.shift(_with_exponents([0, 0, 255]), 100) == 0               # nothing kept
    assert orc.shift(_with_exponents([254, 254]), 1) == 127                # clamped
    assert orc.shift(_with_exponents([1, 1, 1]), 254) == -127
    assert orc.shift(np.zeros(0, np.uint16), 120) == 0
    # 8192 values: samples at even positions only
    e = np.where(np.arange(8192) % 2 == 0, 100, 200)
    assert orc.shift(_with_exponents(e), 90) == 10
    # 10000 values: sample k sits at floor(k*10000/4096)
    pos = (np.arange(4096) * 10000) // 4096
    e = np.full(10000, 200)
    e[pos] = 50
    assert orc.shift(_with_exponents(e), 40) == 10


def test_shift_matched_scale_is_zero(orc):
    x = synth.generate("gauss_block")
    cb = orc.codebook_build(0, 0.02)
    assert orc.shift(x, cb.median_exp) == 0


def test_shift_follows_power_of_two_scaling(orc):
    """x * 2^k moves the shift by k and leaves every marker unchanged (zeros
    always escape)."""
    x0 = synth.gelu_sparse(1 << 17, seed=5)
    cb = orc.codebook_build(0, 1.0)
    ref = None
    for k in range(-4, 5):
        xk = synth.scale_pow2(x0, k)
        c = orc.encode(xk, cb, orc.HIGH)
        if ref is None:
            ref, d0 = c, c.delta - k
        assert c.delta == d0 + k
        assert np.array_equal(c.markers, ref.markers)
        assert c.ovf_used == ref.ovf_used


# ------------------------------------------------------- encode / decode

def _x_hand(g):
    n = g["geometry"]["n"]
    e = np.full(n, g["input"]["default_exponent"], np.uint16)
    for k, v in g["input"]["exponents"].items():
        e[int(k)] = v
    x = _with_exponents(e, g["input"]["default_signfrac"]).astype(np.uint16)
    for k, v in g["input"]["raw_bf16"].items():
        x[int(k)] = int(v, 16)
    return x


def test_hand_worked_stream_layout(orc):
    g = json.load(open(os.path.join(GOLD, "hand_stream.json")))
    geo = g["geometry"]
    lengths = np.zeros(256, np.uint8)
    for s, l in g["codebook"]["lengths"].items():
        lengths[int(s)] = l
    cb = orc.codebook_from_lengths(lengths, g["codebook"]["esc_len"])
    for s, c in g["codebook"]["canonical_codes"].items():
        l, v = (cb.esc_len, cb.esc_code) if s == "esc" else (cb.len[int(s)], cb.code[int(s)])
        assert format(v, "0%db" % l) == c
    x = _x_hand(g)
    n, B, W = geo["n"], geo["block"], geo["slot_words"]
    nb = (n + B - 1) // B
    for case in g["cases"]:
        c = orc.encode(x, cb, block=B, slot_words=W, delta=case["delta"])
        assert c.status == orc.OK
        for i, v in g["expect_signfrac"].items():
            assert c.sf[int(i)] == int(v, 16)
        slots = c.slots.reshape(nb, W, 256)
        for b in range(nb):
            cnt = min(B, n - b * B)
            for j in range(256):
                nj = max(0, -(-(cnt - j) // 256))
                want = case["words"].get("%d:%d" % (b, j), case["default_words"].get("%d:%d" % (b, nj)))
                assert slots[b, 0, j] == int(want, 16), (case["delta"], b, j, hex(slots[b, 0, j]))
                assert c.markers[b * 256 + j] == case["markers"].get("%d:%d" % (b, j), nj)
        assert list(c.overflow_bytes()) == case["overflow"]
        assert list(c.blk_off) == case["blk_off"]
        rc, y = orc.decode(c, cb)
        assert rc == orc.OK and np.array_equal(y, x)


def _cost(cb, delta, e):
    s = int(e) - delta
    if 0 <= s <= 255 and cb.len[s] > 0:
        return cb.len[s]
    return cb.esc_len + 8


def _check_accounting(orc, x, cb, c):
    """Greedy fill: kept codes fit the slot, the next one would not, unused
    slot bits are zero, spill count = sum of (n_j - marker_j)."""
    B, W = c.block, c.slot_words
    nb = c.nblocks
    slots = c.slots.reshape(nb, W, 256)
    total_spill = 0
    for b in range(nb):
        cnt = min(B, c.n - b * B)
        for j in range(256):
            nj = max(0, -(-(cnt - j) // 256))
            m = int(c.markers[b * 256 + j])
            es = x[b * B + j: b * B + cnt: 256] >> 7 & 0xFF
            costs = [_cost(cb, c.delta, e) for e in es]
            used = sum(costs[:m])
            assert used <= 32 * W
            if m < nj:
                assert used + costs[m] > 32 * W
            bits = "".join(format(int(v), "032b") for v in slots[b, :, j])
            assert set(bits[used:]) <= {"0"}
            total_spill += nj - m
        assert c.blk_off[b + 1] - c.blk_off[b] == sum(
            max(0, -(-(cnt - j) // 256)) - int(c.markers[b * 256 + j]) for j in range(256))
    assert total_spill == c.ovf_used


def test_bit_accounting_with_spill(orc):
    x = synth.heavy_tail(3 * 32768 + 777, seed=2)
    cb = orc.codebook_build(2, 1e-3, 3.0)
    c = orc.encode(x, cb, orc.MEDIUM)
    _check_accounting(orc, x, cb, c)
    # a tighter slot (13 words = 3.25 bits/exponent) makes the escapes spill
    c = orc.encode(x, cb, block=32768, slot_words=13)
    assert c.ovf_used > 0
    _check_accounting(orc, x, cb, c)
    rc, y = orc.decode(c, cb)
    assert rc == orc.OK and np.array_equal(y, x)
    x5 = synth.gelu_sparse(2 * 32768 + 300, seed=5)
    cb5 = orc.codebook_build(0, 1.0)
    c5 = orc.encode(x5, cb5, orc.HIGH)
    assert c5.ovf_used > 0
    _check_accounting(orc, x5, cb5, c5)


@pytest.mark.parametrize("level", [0, 1, 2])
def test_roundtrip_every_bf16_pattern(orc, level):
    """Losslessness ([EXP] TL;DR and 'In bits'): every bit pattern -- zeros,
    subnormals, infinities, NaN payloads -- comes back unchanged."""
    x = synth.all_bf16_patterns()
    for model, scale, shape in [(0, 0.02, 0.0), (2, 1e-3, 3.0)]:
        cb = orc.codebook_build(model, scale, shape)
        for delta in [None, -127, -3, 0, 5, 127]:
            c = orc.encode(x, cb, level, delta=delta)
            assert c.status == orc.OK
            rc, y = orc.decode(c, cb)
            assert rc == orc.OK and np.array_equal(y, x)


@pytest.mark.parametrize("name,n", [("laplace_16m", 3 * 65536 + 4321), ("heavy_64m", 5 * 32768 + 17),
                                    ("gelu_act", 4 * 32768 - 5), ("gauss_block", 1)])
def test_roundtrip_workloads_ragged(orc, name, n):
    w = synth.WORKLOADS[name]
    x = synth.generate(name, n)
    model = {"gaussian": 0, "laplace": 1, "powerlaw": 2}[w["model"]]
    cb = orc.codebook_build(model, w["scale"], w["shape"])
    c = orc.encode(x, cb, {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}[w["level"]])
    rc, y = orc.decode(c, cb)
    assert c.status == orc.OK and rc == orc.OK and np.array_equal(y, x)


def test_allocated_and_used_bits_for_matched_models(orc):
    """Used bits per exponent on matched data land near the pages' ideal
    2.5-3.1 range, and under the CLEAN slot's 3.125 allocated bits."""
    for name, model in [("gauss_block", 0), ("laplace_16m", 1)]:
        w = synth.WORKLOADS[name]
        x = synth.generate(name, 4 * 65536)
        cb = orc.codebook_build(model, w["scale"], w["shape"])
        c = orc.encode(x, cb, orc.CLEAN)
        used = sum(_cost(cb, c.delta, e) for e in (x >> 7 & 0xFF)[:65536]) / 65536
        assert 2.5 <= used <= 3.125, (name, used)


def test_empty_tensor(orc):
    cb = orc.codebook_build(0, 0.02)
    c = orc.encode(np.zeros(0, np.uint16), cb, orc.CLEAN)
    assert c.status == orc.OK and c.ovf_used == 0 and c.nblocks == 0
    rc, y = orc.decode(c, cb)
    assert rc == orc.OK and y.size == 0


def test_overflow_capacity_is_reported(orc):
    x = synth.gelu_sparse(3 * 32768, seed=5)
    cb = orc.codebook_build(0, 1.0)
    full = orc.encode(x, cb, orc.HIGH)
    cap = int(full.blk_off[1]) + 3   # block 0 fits, block 1 does not
    assert full.blk_off[2] > cap
    c = orc.encode(x, cb, orc.HIGH, ovf_cap=cap)
    assert c.status == orc.CAPACITY and c.ovf_used == full.ovf_used
    assert np.array_equal(c.ovf[: full.blk_off[1]], full.ovf[: full.blk_off[1]])
    assert not c.ovf[full.blk_off[1]:].any()
    assert np.array_equal(c.slots, full.slots) and np.array_equal(c.markers, full.markers)
    rc, _ = orc.decode(c, cb)
    assert rc == orc.CAPACITY


def test_corrupt_marker_is_detected(orc):
    x = synth.generate("gauss_block")
    cb = orc.codebook_build(0, 0.02)
    c = orc.encode(x, cb, orc.CLEAN)
    c.markers[7] = 257
    rc, _ = orc.decode(c, cb)
    assert rc == orc.CORRUPT


# ------------------------------------------------------------------ SGD

def _bf16_tensor(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)


def test_bf16_rounding_matches_torch(orc):
    rng = np.random.default_rng(21)
    u = rng.integers(0, 1 << 32, size=4000, dtype=np.uint64).astype(np.uint32)
    u[:8] = [0x3F808000, 0x3F818000, 0x3F80FFFF, 0x00008000, 0x80018000, 0x7F7FFFFF, 0x7F800000, 0xFF800000]
    f = u.view(np.float32)
    f = f[~np.isnan(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.bf16_rne(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, ref)
    assert orc.bf16_rne(float("nan")) == 0x7FC0


def test_sgd_matches_torch_two_roundings(orc):
    """W - eta*M in float32 with the product and the difference rounded
    separately ([EXP] 'Training adds a second problem'); torch CPU does the
    same two ops.  A fused multiply-add gives different bits somewhere."""
    n = 3 * 65536 + 999
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    w[:4] = [0x0001, 0x8001, 0x0000, 0x7F80]   # subnormals, zero, +inf
    m[:4] = [0x0003, 0x0001, 0x8000, 0x3F80]
    eta = np.float32(1e-3)
    # cancellation: w ~ eta*m, where the rounding of the product decides the
    # result, so that a fused multiply-add shows up in the bits
    sl = slice(1000, 3000)
    w[sl] = (torch.tensor(float(eta)) * _bf16_tensor(m[sl]).float()).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)
    cbw, cbm = orc.codebook_build(0, 0.02), orc.codebook_build(0, 1e-3)
    W, M = orc.encode(w, cbw, orc.CLEAN), orc.encode(m, cbm, orc.CLEAN)
    out = orc.sgd_step(W, cbw, M, cbm, float(eta))
    assert out.status == orc.OK and out.delta == W.delta
    rc, got = orc.decode(out, cbw)
    assert rc == orc.OK
    wt, mt = _bf16_tensor(w).float(), _bf16_tensor(m).float()
    prod = torch.tensor(float(eta), dtype=torch.float32) * mt
    ref = (wt - prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
    fma = (wt.double() - float(eta) * mt.double()).float().to(torch.bfloat16)
    assert (fma.view(torch.int16).numpy().view(np.uint16) != ref).any()
    # encoding of the new W uses W's stored shift, not a re-estimate
    again = orc.encode(got, cbw, orc.CLEAN, delta=W.delta)
    assert np.array_equal(again.slots, out.slots) and np.array_equal(again.sf, out.sf)


def test_sgd_nan_is_canonical(orc):
    w = np.array([0x7FC1, 0xFF80, 0x3F80], np.uint16)   # NaN payload, -inf, 1.0
    m = np.array([0x3F80, 0xFF80, 0x7FA0], np.uint16)   # 1.0, -inf, NaN
    cb = orc.codebook_build(0, 1.0)
    W, M = orc.encode(w, cb, orc.CLEAN), orc.encode(m, cb, orc.CLEAN)
    out = orc.sgd_step(W, cb, M, cb, 1.0)
    rc, got = orc.decode(out, cb)
    assert rc == orc.OK and list(got) == [0x7FC0, 0x7FC0, 0x7FC0]


# ------------------------------------------------------ momentum step

def _bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_momentum_step_matches_torch_separate_roundings(orc):
    """Heavy-ball momentum on compressed optimizer state ([EXP] 'Jargon',
    'Optimizer state'; [ABS]): M' = bf16(mu*m + g), W' = bf16(w - eta*M'),
    every float32 op rounded on its own, the weight step taking the stored
    BF16 M'.  torch CPU runs the same separate ops.  Cancellation slices make
    a fused multiply-add in either update show up in the bits."""
    n = 2 * 65536 + 4321
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-3, 4)
    g = synth.normal(n, 1e-4, 6)
    w[:5] = [0x0001, 0x8001, 0x0000, 0x7F80, 0x3F80]   # subnormals, zero, +inf, 1
    m[:5] = [0x0003, 0x0001, 0x8000, 0x3F80, 0x0000]
    g[:5] = [0x8000, 0x0002, 0x8000, 0x0000, 0x8000]
    eta, mu = np.float32(1e-3), np.float32(0.9)
    eta_t, mu_t = torch.tensor(float(eta)), torch.tensor(float(mu))
    # g ~ -mu*m: the rounding of the product decides the new momentum
    sl = slice(1000, 3000)
    g[sl] = _bits(-(mu_t * _bf16_tensor(m[sl]).float()))
    mt, gt = _bf16_tensor(m).float(), _bf16_tensor(g).float()
    m_new = _bits((mu_t * mt) + gt)
    # w ~ eta*M': the rounding of the weight step's product decides
    sl2 = slice(5000, 7000)
    w[sl2] = _bits(eta_t * _bf16_tensor(m_new[sl2]).float())
    wt = _bf16_tensor(w).float()
    w_new = _bits(wt - eta_t * _bf16_tensor(m_new).float())

    cbw, cbm = orc.codebook_build(0, 0.02), orc.codebook_build(0, 1e-3)
    W, M = orc.encode(w, cbw, orc.CLEAN), orc.encode(m, cbm, orc.CLEAN)
    W2, M2 = orc.sgd_momentum_step(W, cbw, M, cbm, g, float(eta), float(mu))
    assert W2.status == orc.OK and M2.status == orc.OK
    assert W2.delta == W.delta and M2.delta == M.delta
    rc_w, got_w = orc.decode(W2, cbw)
    rc_m, got_m = orc.decode(M2, cbm)
    assert rc_w == orc.OK and rc_m == orc.OK
    assert np.array_equal(got_m, m_new)
    assert np.array_equal(got_w, w_new)
    # the checks above would catch a fused multiply-add in either update
    fma_m = _bits((mu_t.double() * mt.double() + gt.double()).float())
    assert (fma_m != m_new).any()
    fma_w = _bits((wt.double() - eta_t.double() * _bf16_tensor(m_new).float().double()).float())
    assert (fma_w != w_new).any()
    # ... and the weight step taking the old momentum, or the unrounded new one
    old_m = _bits(wt - eta_t * mt)
    assert (old_m != w_new).any()
    unrounded = _bits(wt - eta_t * ((mu_t * mt) + gt))
    assert (unrounded != w_new).any()
    # each output is coded with its input's stored shift
    again = orc.encode(got_m, cbm, orc.CLEAN, delta=M.delta)
    assert np.array_equal(again.slots, M2.slots) and np.array_equal(again.markers, M2.markers)


def test_momentum_step_with_zero_mu_is_plain_sgd_on_the_gradient(orc):
    """With mu = 0 and finite m the new momentum is the gradient itself
    (0*m + g = g exactly, except that -0 + +0 gives +0), so the weight step
    reduces to the plain fused SGD step with M = g."""
    n = 65536 + 777
    w = synth.normal(n, 0.02, 7)
    m = synth.normal(n, 1e-3, 8)
    g = synth.normal(n, 1e-4, 9)
    g[g == 0x8000] = 0x0000
    cbw, cbm = orc.codebook_build(0, 0.02), orc.codebook_build(0, 1e-3)
    W, M = orc.encode(w, cbw, orc.CLEAN), orc.encode(m, cbm, orc.CLEAN)
    W2, M2 = orc.sgd_momentum_step(W, cbw, M, cbm, g, 1e-3, 0.0)
    _, got_m = orc.decode(M2, cbm)
    assert np.array_equal(got_m, g)
    G = orc.encode(g, cbm, orc.CLEAN)
    plain = orc.sgd_step(W, cbw, G, cbm, 1e-3)
    assert np.array_equal(W2.slots, plain.slots) and np.array_equal(W2.sf, plain.sf)
    assert np.array_equal(W2.markers, plain.markers)


def test_momentum_step_spills_and_status_per_output(orc):
    """Each output has its own overflow region: a too-small capacity for the
    new momentum latches capacity on M' only."""
    n = 65536
    w = synth.normal(n, 0.02, 10)
    m = synth.gelu_sparse(n, 11)   # far off the momentum codebook: heavy spill
    g = synth.normal(n, 1e-2, 12)
    cbw, cbm = orc.codebook_build(0, 0.02), orc.codebook_build(0, 1e-3)
    W, M = orc.encode(w, cbw, orc.CLEAN), orc.encode(m, cbm, orc.CLEAN)
    W2, M2 = orc.sgd_momentum_step(W, cbw, M, cbm, g, 1e-3, 0.9, ovf_cap_m=16)
    assert W2.status == orc.OK
    assert M2.status == orc.CAPACITY and M2.ovf_used > 16
    W3, M3 = orc.sgd_momentum_step(W, cbw, M, cbm, g, 1e-3, 0.9)
    assert M3.status == orc.OK and M3.ovf_used == M2.ovf_used
    rc, got = orc.decode(M3, cbm)
    assert rc == orc.OK


# ------------------------------------------------------ zero-atom model

def test_zero_atom_reduces_to_the_plain_model(orc):
    """With no point mass the mixture is the plain model: same lengths and
    codes; with one, every other bucket's weight is scaled by 1 - z."""
    for model, scale, shape in [(0, 1.0, 0.0), (1, 0.01, 0.0), (2, 1e-3, 3.0)]:
        plain = orc.codebook_build(model, scale, shape)
        z0 = orc.codebook_build_zero_atom(model, scale, shape, 0.0)
        assert z0.zero_atom == 1
        assert np.array_equal(z0.lengths(), plain.lengths()) and np.array_equal(z0.codes(), plain.codes())
        assert z0.esc_len == plain.esc_len and z0.median_exp == plain.median_exp
        z = orc.codebook_build_zero_atom(model, scale, shape, 0.3)
        wp = np.array(plain.weight[:], dtype=np.float64)
        wz = np.array(z.weight[:], dtype=np.float64)
        big = wp[1:] > 1e8                                 # integer rounding below 1e-8 relative
        assert np.allclose(wz[1:][big] / wp[1:][big], 0.7, rtol=1e-8)
        assert abs(wz.sum() - 2.0 ** 40) < 256          # total mass 1, up to rounding
        assert z.median_exp == plain.median_exp          # the atom sits outside 1..254
        _check_codebook(z)


def test_zero_atom_above_two_fifths_gets_a_one_bit_code(orc):
    """A symbol of probability above 2/5 has a one-bit codeword in every
    optimal prefix code (a textbook property of Huffman codes)."""
    for zf in (0.41, 0.5, 0.9):
        cb = orc.codebook_build_zero_atom(0, 1.0, 0.0, zf)
        assert cb.len[0] == 1
    assert orc.codebook_build_zero_atom(0, 1.0, 0.0, 0.3).len[0] >= 2


def test_zero_atom_lossless_for_every_pattern_and_shift(orc):
    """All 65,536 BF16 patterns round-trip for shifts that put the zero
    symbol's collision (a nonzero exponent equal to the shift) anywhere."""
    x = synth.all_bf16_patterns()
    cb = orc.codebook_build_zero_atom(0, 1.0, 0.0, 0.3)
    for level in (orc.CLEAN, orc.HIGH):
        for delta in (-127, -3, 0, 5, 126, 127):
            c = orc.encode(x, cb, level, delta=delta)
            rc, y = orc.decode(c, cb)
            assert rc == orc.OK and np.array_equal(y, x), (level, delta)


def test_zero_atom_codes_zeros_unshifted_and_escapes_the_collision(orc):
    """Zeros cost len[0] bits whatever the shift; a nonzero value whose
    exponent equals the shift (symbol 0 after the shift) is escaped with its
    raw exponent.  Checked on the bits of one stream (MSB first)."""
    cb = orc.codebook_build_zero_atom(0, 1.0, 0.0, 0.3)
    l0, c0 = int(cb.len[0]), int(cb.code[0])
    delta = 40
    x = np.zeros(65536, np.uint16)                   # +0.0 everywhere
    x[256] = 0x8000                                  # -0.0, stream 0 symbol 1
    x[512] = delta << 7                              # exponent == shift, stream 0 symbol 2
    c = orc.encode(x, cb, orc.CLEAN, delta=delta)
    bits = "".join(format(int(w), "032b") for w in c.slots.reshape(25, 256)[:, 0])
    code0 = format(c0, "0%db" % l0)
    esc = format(int(cb.esc_code), "0%db" % int(cb.esc_len)) + format(delta, "08b")
    assert bits.startswith(code0 + code0 + esc + code0)
    # a stream of zeros only holds floor(800 / len0) of them in its slot
    assert c.markers[1] == min(256, 800 // l0)
    rc, y = orc.decode(c, cb)
    assert rc == orc.OK and np.array_equal(y, x)


def test_zero_atom_keeps_markers_under_power_of_two_scaling(orc):
    """x * 2^k moves the shift by k; zeros stay symbol 0 and every other
    exponent keeps its symbol, so the markers and the spill do not change,
    and the spill is far below the plain model's (whose zeros escape)."""
    x0 = synth.gelu_sparse(1 << 17, seed=5)
    cb = orc.codebook_build_zero_atom(0, 1.0, 0.0, 0.3)
    plain = orc.encode(x0, orc.codebook_build(0, 1.0), orc.HIGH)
    ref = None
    for k in range(-4, 5):
        c = orc.encode(synth.scale_pow2(x0, k), cb, orc.HIGH)
        if ref is None:
            ref, d0 = c, c.delta - k
        assert c.delta == d0 + k
        assert np.array_equal(c.markers, ref.markers) and c.ovf_used == ref.ovf_used
    assert ref.ovf_used < plain.ovf_used / 4


# ------------------------------------------------------------ AdamW step

def _adamw_torch(w, m, v, g, k):
    """The AdamW step as separate torch CPU float32 ops (each rounded)."""
    kt = [torch.tensor(float(x), dtype=torch.float32) for x in k]
    wt, mt, vt, gt = (_bf16_tensor(a).float() for a in (w, m, v, g))
    m_new = _bits((kt[0] * mt) + (kt[1] * gt))
    v_new = _bits((kt[2] * vt) + (kt[3] * (gt * gt)))
    mf, vf = _bf16_tensor(m_new).float(), _bf16_tensor(v_new).float()
    den = (torch.sqrt(vf) * kt[5]) + kt[6]
    upd = (kt[4] * mf) / den
    w_new = _bits((wt - (kt[7] * wt)) - upd)
    return w_new, m_new, v_new, (wt, mf, den, upd)


def test_adamw_matches_torch_separate_roundings(orc):
    """AdamW on compressed weights and moments (optimizer state, [EXP]
    'Jargon'; [ABS]): M' = bf16(b1*m + (1-b1)*g), V' = bf16(b2*v + (1-b2)*g*g),
    W' = bf16((w - lr*wd*w) - step*M' / (sqrt(V')*rs + eps)), every float32
    operation rounded on its own; torch CPU runs the same ops.  A fused
    multiply-add in the update changes the bits somewhere."""
    n = 2 * 65536 + 3333
    w = synth.normal(n, 0.02, 3)
    m = synth.normal(n, 1e-4, 4)
    v = synth.bf16_bits(np.abs(synth.bits_to_f32(synth.normal(n, 1e-8, 5))))   # a second moment is >= 0
    g = synth.normal(n, 1e-4, 6)
    w[:4] = [0x0000, 0x8000, 0x7F80, 0x0001]
    m[:4] = [0x0000, 0x3F80, 0x0000, 0x8001]
    v[:4] = [0x0000, 0x0000, 0x3F80, 0x0001]
    g[:4] = [0x0000, 0x8000, 0x3F80, 0x0002]
    k = orc.adamw_constants(1e-3, 0.9, 0.999, 1e-8, 0.01, 7)
    cbw, cbm, cbv = orc.codebook_build(0, 0.02), orc.codebook_build(0, 1e-4), orc.codebook_build(1, 1e-8)
    W, M, V = (orc.encode(x, cb, orc.CLEAN) for x, cb in ((w, cbw), (m, cbm), (v, cbv)))
    W2, M2, V2 = orc.adamw_step(W, cbw, M, cbm, V, cbv, g, k)
    assert W2.status == M2.status == V2.status == orc.OK
    assert (W2.delta, M2.delta, V2.delta) == (W.delta, M.delta, V.delta)
    got = [orc.decode(t, cb)[1] for t, cb in ((W2, cbw), (M2, cbm), (V2, cbv))]
    w_new, m_new, v_new, (wt, mf, den, upd) = _adamw_torch(w, m, v, g, k)
    assert np.array_equal(got[1], m_new)
    assert np.array_equal(got[2], v_new)
    # NaN results (inf - inf at the +inf weight) are this library's 0x7FC0;
    # torch keeps the sign of the NaN it computed
    nan = ((w_new & 0x7F80) == 0x7F80) & ((w_new & 0x7F) != 0)
    assert nan.sum() == 1 and (got[0][nan] == 0x7FC0).all()
    assert np.array_equal(got[0][~nan], w_new[~nan])
    # the check above would catch a fused multiply-add in the moment update
    kt = [float(x) for x in k]
    fma_m = _bits((kt[0] * _bf16_tensor(m).double() + torch.tensor(kt[1], dtype=torch.float32).double()
                   * _bf16_tensor(g).double()).float())
    assert (fma_m != m_new).any()
    # ... or the weight step without the decoupled decay
    no_decay = _bits(wt - upd)
    assert (no_decay != w_new).any()


def test_adamw_first_step_from_zero_moments_is_sign_descent(orc):
    """From zero moments, step 1 of Adam moves every weight by lr * sign(g)
    (the bias corrections undo (1 - b1) and (1 - b2) exactly), up to the BF16
    rounding of the stored moments."""
    n = 65536 + 100
    lr = 1e-3
    w = synth.normal(n, 1e-4, 7)             # |w| small: its BF16 spacing is far below lr
    g = synth.normal(n, 1e-2, 8)
    g[g == 0x8000] = 0x0000
    z = np.zeros(n, np.uint16)
    k = orc.adamw_constants(lr, 0.9, 0.999, 1e-12, 0.0, 1)
    cbw, cbm, cbv = orc.codebook_build(0, 1e-4), orc.codebook_build(0, 1e-3), orc.codebook_build(0, 1e-5)
    W, M, V = orc.encode(w, cbw, orc.CLEAN), orc.encode(z, cbm, orc.CLEAN), orc.encode(z, cbv, orc.CLEAN)
    W2, _, _ = orc.adamw_step(W, cbw, M, cbm, V, cbv, g, k)
    _, got = orc.decode(W2, cbw)
    step = synth.bits_to_f32(got).astype(np.float64) - synth.bits_to_f32(w).astype(np.float64)
    sign = np.sign(synth.bits_to_f32(g).astype(np.float64))
    nz = sign != 0
    assert np.allclose(step[nz], -lr * sign[nz], rtol=2e-2, atol=0)
    assert np.array_equal(got[~nz], w[~nz])   # zero gradient, zero moments: no move
