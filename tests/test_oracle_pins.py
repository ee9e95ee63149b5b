"""Pins for the CPU oracle: checks against what the Unweight blog post and
plain mathematics fix, never against the oracle's own formulas retyped.

Each test names what pins it: the BF16 number format, a hand-worked example
(tests/golden), brute force over tiny alphabets, the textbook Huffman
construction, the Kraft inequality, the entropy bound, or an independent
numpy computation.
"""
import heapq
import itertools
import json
import math
import os

import numpy as np
import pytest

import workloads as wl

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- BF16 fields
def test_field_split_hand_values(oracle):
    # BF16 = 1 sign bit, 8 exponent bits, 7 mantissa bits (Unweight blog, BF16 layout paragraph).
    cases = {
        0x3F80: (127, 0x00),   # +1.0
        0xBF80: (127, 0x80),   # -1.0
        0x3FC0: (127, 0x40),   # +1.5  (mantissa 1000000b)
        0x4049: (128, 0x49),   # +3.140625
        0x0001: (0, 0x01),     # smallest positive subnormal
        0x8000: (0, 0x80),     # -0.0
        0x7F80: (255, 0x00),   # +inf
        0xFFC1: (255, 0xC1),   # negative NaN with payload 1000001b
    }
    w = np.array(list(cases), np.uint16)
    e, sm = oracle.split(w)
    for i, (ee, ss) in enumerate(cases.values()):
        assert (e[i], sm[i]) == (ee, ss)


def test_field_split_matches_float_value(oracle):
    # For every normal BF16 pattern, the value is (-1)^s * 2^(e-127) * (1 + m/128):
    # recover s, e, m from the float value with frexp and compare.
    pats = wl.all_bf16_patterns().ravel()
    e, sm = oracle.split(pats)
    with np.errstate(invalid="ignore"):
        vals = wl.bf16_to_f32(pats).astype(np.float64)
    normal = np.isfinite(vals) & (np.abs(vals) >= 2.0 ** -126)
    frac, ex = np.frexp(np.abs(vals[normal]))          # |v| = frac * 2^ex, frac in [0.5, 1)
    assert np.array_equal(e[normal].astype(np.int64), ex - 1 + 127)
    mant = np.round((frac * 2 - 1) * 128).astype(np.int64)
    assert np.array_equal((sm[normal] & 0x7F).astype(np.int64), mant)
    assert np.array_equal(sm[normal] >> 7, np.signbit(vals[normal]).astype(np.uint8))


def test_join_inverts_split_for_every_pattern(oracle):
    pats = wl.all_bf16_patterns().ravel()
    e, sm = oracle.split(pats)
    back = np.array([oracle.join(a, b) for a, b in zip(e[::97], sm[::97])], np.uint16)
    assert np.array_equal(back, pats[::97])


# ---------------------------------------------------------------- histogram / palette
def test_histogram_matches_frexp_exponents(oracle):
    w = wl.normal_weights(64, 512, 0.02, seed=3)
    v = wl.bf16_to_f32(w).astype(np.float64).ravel()
    _, ex = np.frexp(np.abs(v))
    biased = np.where(v == 0, 0, ex - 1 + 127)      # no subnormals at this scale
    assert np.array_equal(oracle.histogram(w), np.bincount(biased, minlength=256).astype(np.uint64))


def test_palette_order_ties_and_limit(oracle):
    c = np.zeros(256, np.uint64)
    # 20 distinct exponents; counts chosen so that ties decide the order.
    for v, n in [(100, 7), (120, 5), (121, 5), (90, 5), (3, 1), (200, 0)]:
        c[v] = n
    for v in range(130, 145):
        c[v] = 2
    pal = oracle.palette(c)
    assert pal[:4] == [100, 90, 120, 121]          # count desc, then exponent asc
    assert pal[4:] == list(range(130, 142))         # 12 of the 15 twos, smallest first
    assert len(pal) == 16 and 3 not in pal and 200 not in pal


def test_palette_skips_zero_counts(oracle):
    c = np.zeros(256, np.uint64)
    c[[5, 9]] = [3, 1]
    assert oracle.palette(c) == [5, 9]


# ---------------------------------------------------------------- escapes
def test_escape_flags_one_decision_per_row_of_64(oracle):
    # A group of 64 is escaped iff it holds an exponent outside the palette
    # (Unweight blog, paragraph on rows of 64 with rare exponents).
    w = np.full((2, 128), 0x3C00, np.uint16)     # exponent 120 everywhere
    w[0, 70] = 0x3800                             # exponent 112 in group (0, 1)
    pal = [120]
    assert list(oracle.escape_flags(w, pal)) == [0, 1, 0, 0]
    assert list(oracle.escape_flags(w, [120, 112])) == [0, 0, 0, 0]


# ---------------------------------------------------------------- code lengths
def _brute_force_min_cost(freq, lmax):
    """Enumerate every per-symbol length vector (not count vectors)."""
    idx = [i for i, f in enumerate(freq) if f > 0]
    best = None
    for lens in itertools.product(range(1, lmax + 1), repeat=len(idx)):
        if sum(2.0 ** -l for l in lens) <= 1.0 + 1e-12:
            cost = sum(freq[i] * l for i, l in zip(idx, lens))
            best = cost if best is None else min(best, cost)
    return best


def _huffman_cost(freq):
    h = [f for f in freq if f > 0]
    if len(h) == 1:
        return h[0]
    heapq.heapify(h)
    cost = 0
    while len(h) > 1:
        a, b = heapq.heappop(h), heapq.heappop(h)
        cost += a + b
        heapq.heappush(h, a + b)
    return cost


def _cost(freq, lens):
    return sum(f * l for f, l in zip(freq, lens))


def _package_merge_lengths(freq, lmax):
    """Optimal length-limited code lengths by package-merge (Larmore and
    Hirschberg, 1990), written here independently of the oracle's exhaustive
    search: the coin collector's problem over lmax denominations.  Each of
    the n used symbols is a coin of every width 2^-1 .. 2^-lmax with its
    frequency as numismatic value; repeatedly pair up the cheapest coins of
    the narrowest width (packages) and merge them with the next width's
    coins; the 2n - 2 cheapest items of the widest list pay for total width
    n - 1, and a symbol's code length is the number of chosen items that
    contain it."""
    used = [i for i, f in enumerate(freq) if f > 0]
    lens = [0] * len(freq)
    if len(used) == 1:
        lens[used[0]] = 1
        return lens
    if not used:
        return lens
    leaves = sorted(((int(freq[i]), (i,)) for i in used), key=lambda t: t[0])
    items = list(leaves)
    for _ in range(lmax - 1):
        packages = [(items[j][0] + items[j + 1][0], items[j][1] + items[j + 1][1])
                    for j in range(0, len(items) - 1, 2)]
        items = sorted(leaves + packages, key=lambda t: t[0])
    for _, members in items[: 2 * len(used) - 2]:
        for i in members:
            lens[i] += 1
    return lens


def _skewed_histogram(rng):
    """Counts of 16 palette symbols shaped like trained-layer exponents: a
    geometric-ish decay with a random rate, random noise, and now and then a
    few near-ties or a very rare symbol."""
    rate = rng.uniform(0.45, 0.9)
    base = rng.uniform(1e3, 1e6) * rate ** np.arange(16) * rng.uniform(0.7, 1.3, 16)
    if rng.random() < 0.3:
        base[rng.integers(0, 16)] = rng.integers(1, 5)
    if rng.random() < 0.3:
        j = int(rng.integers(0, 15))
        base[j + 1] = base[j]
    return [max(1, int(v)) for v in base]


def _kraft(lens):
    return sum(2.0 ** -l for l in lens if l > 0)


@pytest.mark.parametrize("seed", range(40))
def test_code_lengths_brute_force_tiny_alphabets(oracle, seed):
    rng = np.random.default_rng(seed)
    m = int(rng.integers(1, 7))
    lmax = int(rng.integers(max(1, math.ceil(math.log2(m)) if m > 1 else 1), 7))
    freq = [int(v) for v in rng.integers(0, 50, m)]
    if seed % 5 == 0:
        freq = [int(v) for v in rng.integers(1, 4, m)]      # many ties
    lens = oracle.code_lengths(freq, lmax)
    if sum(freq) == 0:
        assert all(l == 0 for l in lens)
        return
    assert all((l == 0) == (f == 0) for l, f in zip(lens, freq))
    assert max(lens) <= lmax and _kraft(lens) <= 1.0
    assert _cost(freq, lens) == _brute_force_min_cost(freq, lmax)


def test_code_lengths_tie_rule(oracle):
    # freq (2,2,1,1): optimal cost 12 is reached by (2,2,2,2) and by
    # (1,2,3,3).  The rule prefers more symbols on shorter levels
    # (lexicographically larger (n_1, n_2, ...)): (1,2,3,3).
    assert oracle.code_lengths([2, 2, 1, 1], 6) == [1, 2, 3, 3]
    # equal frequencies: lower palette index gets the shorter code
    assert oracle.code_lengths([1, 1, 1], 6) == [1, 2, 2]


def test_code_lengths_hand_examples(oracle):
    assert oracle.code_lengths([1, 1, 1, 1], 6) == [2, 2, 2, 2]
    assert oracle.code_lengths([8, 4, 2, 1, 1], 6) == [1, 2, 3, 4, 4]      # textbook Huffman
    assert oracle.code_lengths([8, 4, 2, 1, 1], 3) == [1, 3, 3, 3, 3]      # worked: cost 32 < 34
    assert oracle.code_lengths([0, 7, 0], 6) == [0, 1, 0]                  # one symbol -> 1 bit
    assert oracle.code_lengths([40, 16, 8], 6) == [1, 2, 2]
    with pytest.raises(ValueError):
        oracle.code_lengths([1] * 5, 2)                                    # 5 symbols > 2^2


@pytest.mark.parametrize("seed", range(20))
def test_code_lengths_equal_textbook_huffman_when_limit_is_loose(oracle, seed):
    rng = np.random.default_rng(100 + seed)
    m = int(rng.integers(2, 12))
    freq = [int(v) for v in rng.integers(1, 1000, m)]
    lens = oracle.code_lengths(freq, 15)
    assert _cost(freq, lens) == _huffman_cost(freq)
    assert abs(_kraft(lens) - 1.0) < 1e-12          # an optimal code is complete


@pytest.mark.parametrize("seed", range(36))
@pytest.mark.parametrize("lmax", [5, 6])
def test_code_lengths_equal_package_merge_cost_16_symbols(oracle, seed, lmax):
    # The shipped configuration: a full 16-symbol palette under a binding
    # length limit (5 is the format's; 6 too).  The optimal total cost is
    # unique even where the lengths are not, so the oracle's cost must equal
    # package-merge's, and its lengths must form a valid prefix code.
    rng = np.random.default_rng(7000 + seed)
    freq = _skewed_histogram(rng)
    lens = oracle.code_lengths(freq, lmax)
    ref = _package_merge_lengths(freq, lmax)
    assert max(ref) <= lmax and _kraft(ref) <= 1.0
    assert max(lens) <= lmax and _kraft(lens) <= 1.0 and min(lens) >= 1
    assert _cost(freq, lens) == _cost(freq, ref)


def test_package_merge_agrees_with_brute_force():
    # the test-side package-merge itself, against enumeration on tiny alphabets
    for seed in range(30):
        rng = np.random.default_rng(9000 + seed)
        m = int(rng.integers(2, 7))
        lmax = int(rng.integers(max(1, math.ceil(math.log2(m))), 6))
        freq = [int(v) for v in rng.integers(1, 60, m)]
        assert _cost(freq, _package_merge_lengths(freq, lmax)) == _brute_force_min_cost(freq, lmax)


def test_mean_length_within_one_bit_of_entropy(oracle):
    # Textbook bound H <= L < H + 1 on the symbol distribution of the coded
    # groups of a N(0, 0.02) matrix (the blog: ~2.6 bits of entropy), at the
    # code-length limit the format ships (oracle.LMAX).  The limit binds here
    # (an unlimited code would be shorter), and the bound still holds.
    assert oracle.LMAX == 5
    w = wl.normal_weights(512, 1024, 0.02, seed=0)
    pal = oracle.palette(oracle.histogram(w))
    flags = oracle.escape_flags(w, pal).astype(bool)
    e = ((w.astype(np.uint32) >> 7) & 0xFF).reshape(-1, 64)[~flags]
    freq = np.array([(e == v).sum() for v in pal], np.float64)
    lens = oracle.code_lengths(freq.astype(np.uint64), oracle.LMAX)
    p = freq / freq.sum()
    H = -(p[p > 0] * np.log2(p[p > 0])).sum()
    L = (p * np.array(lens)).sum()
    assert H <= L < H + 1
    assert 2.4 < H < 2.8
    assert _cost(freq.astype(np.int64), lens) == _cost(freq.astype(np.int64),
                                                       _package_merge_lengths(freq.astype(np.int64), oracle.LMAX))
    assert _cost(freq.astype(np.int64), lens) > _huffman_cost([int(v) for v in freq])   # the limit binds


# ---------------------------------------------------------------- canonical codes
def test_canonical_codes_hand_example(oracle):
    # lengths by symbol: s0:3 s1:2 s2:3 s3:2 -> order (2,s1) (2,s3) (3,s0) (3,s2)
    assert oracle.canonical_codes([3, 2, 3, 2]) == [0b100, 0b00, 0b101, 0b01]
    assert oracle.canonical_codes([1, 2, 2]) == [0b0, 0b10, 0b11]
    assert oracle.canonical_codes([0, 1, 0]) == [0, 0, 0]


@pytest.mark.parametrize("seed", range(20))
def test_canonical_codes_are_prefix_free(oracle, seed):
    rng = np.random.default_rng(seed)
    freq = rng.integers(0, 10_000, 16).astype(np.uint64)
    lens = oracle.code_lengths(freq, 6)
    codes = oracle.canonical_codes(lens)
    words = [format(c, "0%db" % l) for c, l in zip(codes, lens) if l > 0]
    for a, b in itertools.permutations(words, 2):
        assert not b.startswith(a)


# ---------------------------------------------------------------- hand-worked blobs
def _golden(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _worked_matrix():
    g = _golden("worked_example_1x64.json")
    i = np.arange(64)
    e = np.array(g["exponent_period"])[i % 8]
    w = ((i % 2) << 15) | (e << 7) | i
    return w.astype(np.uint16).reshape(1, 64), g


def test_worked_example_blob(oracle):
    w, g = _worked_matrix()
    blob, info = oracle.compress(w)
    b = np.frombuffer(blob, np.uint8)
    assert info["palette"] == g["palette"]
    assert info["code_len"][:3] == g["code_len"] and info["code_bits"] == g["code_bits"]
    assert len(blob) == g["blob_bytes"]
    for k, v in g["sections"].items():
        assert info[k] == v
    assert b[:4].tobytes() == b"UWB1"
    assert b[g["sections"]["off_glen"]] == g["glen"]
    code = b[g["sections"]["off_code"]: g["sections"]["off_code"] + 16].tobytes().hex()
    assert code == g["code_region_hex"]
    sm = b[256:320]
    assert list(sm) == [((k % 2) << 7) | k for k in range(64)]
    tc = np.frombuffer(blob[768:776], np.uint32)
    te = np.frombuffer(blob[1024:1032], np.uint32)
    assert list(tc) == g["tcode"] and list(te) == g["tesc"]
    assert np.array_equal(oracle.decompress(blob), w)


def test_worked_ragged_row_example(oracle):
    # A row of 70 weights: extended to 128 with the filler, true width kept.
    with open(os.path.join(GOLD, "worked_example_ragged_1x70.json")) as f:
        g = json.load(f)
    i = np.arange(g["cols"])
    w = (((120 + (i % 2)) << 7) | i).astype(np.uint16)[None, :]
    blob, info = oracle.compress(w)
    b = np.frombuffer(blob, np.uint8)
    assert info["cols"] == 70 and info["rows"] == 1
    assert info["palette"] == g["palette"] and info["code_len"][:2] == g["code_len"]
    assert info["code_bits"] == g["code_bits"] and info["n_groups"] == g["n_groups"]
    assert info["n_tiles"] == g["n_tiles"] and len(blob) == g["blob_bytes"]
    for k, v in g["sections"].items():
        assert info[k] == v
    assert oracle.filler(info["palette"]) == g["filler"]
    assert list(b[512:514]) == g["glen"]
    assert list(np.frombuffer(blob[768:780], np.uint32)) == g["tcode"]
    assert list(np.frombuffer(blob[1024:1036], np.uint32)) == g["tesc"]
    assert b[1280:1312].tobytes().hex() == g["code_region_hex"]
    assert list(b[256:384]) == list(range(70)) + [0] * 58          # sign+mantissa, then the filler's
    assert np.array_equal(oracle.decompress(blob), w)


@pytest.mark.parametrize("shape", [(1, 1), (3, 100), (33, 130), (77, 4097), (40, 14335)])
def test_ragged_round_trip(oracle, shape):
    w = wl.normal_weights(*shape, 0.02, seed=shape[1])
    blob, info = oracle.compress(w)
    assert info["cols"] == shape[1]
    assert np.array_equal(oracle.decompress(blob), w)
    # the blob is the extended matrix's blob apart from the recorded width
    wp = oracle.pad(w, info["palette"])
    assert wp.shape[1] % 64 == 0 and np.array_equal(wp[:, : shape[1]], w)
    assert np.all(wp[:, shape[1]:] == oracle.filler(info["palette"]))
    blob_p, info_p = oracle.compress(wp)
    a, bb = np.frombuffer(blob, np.uint8), np.frombuffer(blob_p, np.uint8)
    assert a.size == bb.size and np.array_equal(a[:16], bb[:16]) and np.array_equal(a[24:], bb[24:])


def test_filler_rule(oracle):
    assert oracle.filler([121, 120]) == 121 << 7
    assert oracle.filler([255, 3]) == 3 << 7          # never an Inf/NaN exponent
    assert oracle.filler([255]) == 0
    assert oracle.stored_cols(1) == 64 and oracle.stored_cols(64) == 64 and oracle.stored_cols(65) == 128


def test_worked_escape_example(oracle):
    g = _golden("worked_example_escape_1x128.json")
    k = np.arange(128)
    e = np.where(k < 64, 100 + (k % 16), 100)
    e[127] = 99
    w = ((e << 7) | (k % 128)).astype(np.uint16).reshape(1, 128)
    blob, info = oracle.compress(w)
    b = np.frombuffer(blob, np.uint8)
    assert info["palette"] == g["palette"] and info["code_len"] == g["code_len"]
    assert info["n_escaped"] == g["n_escaped"]
    assert list(b[info["off_glen"]: info["off_glen"] + 2]) == g["glen"]
    assert b[info["off_code"]: info["off_code"] + 32].tobytes().hex() == g["code_region_hex"]
    assert list(np.frombuffer(b[info["off_tcode"]: info["off_tcode"] + 12].tobytes(), np.uint32)) == g["tcode"]
    assert list(np.frombuffer(b[info["off_tesc"]: info["off_tesc"] + 12].tobytes(), np.uint32)) == g["tesc"]
    assert list(b[info["off_esc"]: info["off_esc"] + 64]) == [100] * 63 + [99]
    assert np.array_equal(oracle.decompress(blob), w)


# ---------------------------------------------------------------- palette-4 form

def test_palette4_worked_example(oracle):
    # The 1 x 64 worked matrix: exponents 120,120,120,121,120,121,120,119
    # repeating, palette (120, 121, 119), so indices 0,0,0,1,0,1,0,2
    # repeating.  Byte i of a chunk packs weights 2i (low nibble) and 2i+1:
    # 0x00, 0x10, 0x10, 0x20 repeating; one row, so chunk 1 follows chunk 0.
    w, g = _worked_matrix()
    assert oracle.palette4(w, g["palette"]).tobytes().hex() == "00101020" * 8


def test_palette4_escaped_group_is_zero(oracle):
    # The escape example: group 0 has exponent 100 + (k mod 16) = palette
    # index k mod 16, so byte i of either chunk is (2i mod 16) | (2i+1 mod 16) << 4;
    # group 1 is escaped and holds zeros.  One row: group kg at bytes 32kg..32kg+31.
    g = _golden("worked_example_escape_1x128.json")
    k = np.arange(128)
    e = np.where(k < 64, 100 + (k % 16), 100)
    e[127] = 99
    w = ((e << 7) | (k % 128)).astype(np.uint16).reshape(1, 128)
    p4 = oracle.palette4(w, g["palette"])
    chunk = [(2 * i) % 16 | (((2 * i + 1) % 16) << 4) for i in range(16)]
    assert list(p4[:32]) == chunk + chunk
    assert not p4[32:].any()


def _palette4_numpy(w, pal, esc):
    """The palette-4 layout built with whole-array reshapes (a second reading
    of the layout, written independently of the oracle's per-weight loop)."""
    rows, cols = w.shape
    gpr = cols // 64
    lut = np.zeros(256, np.int64)
    lut[np.array(pal, np.int64)] = np.arange(len(pal))
    idx = lut[(w.astype(np.int64) >> 7) & 0xFF]
    idx[np.repeat(esc.reshape(rows, gpr).astype(bool), 64, axis=1)] = 0
    out = np.zeros(rows * cols // 2, np.uint8)
    for rb in range((rows + 31) // 32):
        R = min(32, rows - 32 * rb)
        blk = idx[32 * rb: 32 * rb + R].reshape(R, gpr, 2, 16, 2)     # row, group, chunk, byte, nibble
        packed = (blk[..., 0] | (blk[..., 1] << 4)).astype(np.uint8)   # [R, gpr, 2, 16]
        base = 32 * 32 * rb * gpr
        out[base: base + 32 * R * gpr] = packed.transpose(1, 2, 0, 3).ravel()
    return out


@pytest.mark.parametrize("shape", [(1, 64), (33, 128), (70, 192), (64, 64)])
def test_palette4_layout_and_round_trip(oracle, shape):
    rows, cols = shape
    w = wl.heavy_tailed_weights(rows, cols, seed=rows + cols)
    pal = oracle.palette(oracle.histogram(w))
    esc = oracle.escape_flags(w, pal)
    p4 = oracle.palette4(w, pal)
    assert np.array_equal(p4, _palette4_numpy(w, pal, esc))
    # every weight of a group that is not escaped comes back from its index
    e, sm = oracle.split(w)
    ok = ~np.repeat(esc.reshape(rows, cols // 64).astype(bool), 64, axis=1).ravel()
    lut = np.zeros(256, np.int64)
    lut[np.array(pal, np.int64)] = np.arange(len(pal))
    assert np.array_equal(np.array(pal, np.int64)[lut[e[ok]]], e[ok].astype(np.int64))
    # the index of every position is used exactly once: nibble histogram
    nib = np.concatenate([p4 & 15, p4 >> 4])
    want = np.bincount(np.where(ok, lut[e], 0), minlength=16)
    assert np.array_equal(np.bincount(nib, minlength=16), want)


# ---------------------------------------------------------------- exponent form

def test_exponent_form_worked_example(oracle):
    # One row: the exponents in weight order (chunk c = weights 16c..16c+15).
    w, g = _worked_matrix()
    assert list(oracle.exponents(w)) == [g["exponent_period"][k % 8] for k in range(64)]


@pytest.mark.parametrize("shape", [(1, 64), (33, 128), (70, 192)])
def test_exponent_form_is_the_sm_layout_of_exponents(oracle, shape):
    # The blob's sign+mantissa section has the same layout: rebuilding every
    # weight from (exponent form, sm section) at the same byte gives W back.
    rows, cols = shape
    w = wl.heavy_tailed_weights(rows, cols, seed=rows * 7 + cols)
    blob, info = oracle.compress(w)
    sm = np.frombuffer(blob, np.uint8)[info["off_sm"]: info["off_sm"] + rows * cols].astype(np.uint16)
    ex = oracle.exponents(w).astype(np.uint16)
    bits = ((sm & 0x80) << 8) | (ex << 7) | (sm & 0x7F)
    # and the layout itself, read with whole-array reshapes
    out = np.zeros(rows * cols, np.uint8)
    e = ((w.astype(np.int64) >> 7) & 0xFF).astype(np.uint8)
    gpr = cols // 64
    for rb in range((rows + 31) // 32):
        R = min(32, rows - 32 * rb)
        blk = e[32 * rb: 32 * rb + R].reshape(R, gpr, 4, 16).transpose(1, 2, 0, 3)
        out[64 * 32 * rb * gpr: 64 * 32 * rb * gpr + 64 * R * gpr] = blk.ravel()
    assert np.array_equal(oracle.exponents(w), out)
    want = np.zeros(rows * cols, np.uint16)
    for rb in range((rows + 31) // 32):
        R = min(32, rows - 32 * rb)
        want[64 * 32 * rb * gpr: 64 * 32 * rb * gpr + 64 * R * gpr] = \
            w[32 * rb: 32 * rb + R].reshape(R, gpr, 4, 16).transpose(1, 2, 0, 3).ravel()
    assert np.array_equal(bits, want)


# ---------------------------------------------------------------- round trips
def test_round_trip_every_bf16_pattern(oracle):
    w = wl.all_bf16_patterns()
    blob, info = oracle.compress(w)
    assert info["n_escaped"] == 1024 - 64          # 16 exponents per sign coded
    assert np.array_equal(oracle.decompress(blob), w)


@pytest.mark.parametrize("shape", [(1, 64), (3, 128), (33, 192), (65, 1024), (256, 1024)])
def test_round_trip_normal_and_ragged(oracle, shape):
    w = wl.normal_weights(*shape, sigma=0.02, seed=shape[0])
    blob, info = oracle.compress(w)
    assert np.array_equal(oracle.decompress(blob), w)
    assert info["n_tiles"] == -(-shape[0] // 32) * (shape[1] // 64)


def test_round_trip_heavy_tailed_has_escapes(oracle):
    w = wl.heavy_tailed_weights(512, 512, seed=0)
    blob, info = oracle.compress(w)
    assert 0.02 < info["n_escaped"] / info["n_groups"] < 0.2
    assert np.array_equal(oracle.decompress(blob), w)


def test_round_trip_single_symbol_and_all_escaped(oracle):
    z = np.zeros((5, 128), np.uint16)
    blob, info = oracle.compress(z)
    assert info["code_len"][0] == 1 and info["code_bits"] == 64 * 10
    assert np.array_equal(oracle.decompress(blob), z)
    # every group holds 32 distinct exponents: at most 16 fit the palette
    k = np.arange(64)
    row = (((100 + k % 32) << 7) | k).astype(np.uint16)
    a = np.tile(row, (4, 3))
    blob, info = oracle.compress(a)
    assert info["n_escaped"] == info["n_groups"] == 12
    assert np.array_equal(oracle.decompress(blob), a)


def test_sign_and_mantissa_stored_untouched(oracle):
    # The blob's sign+mantissa section is a permutation of the raw bytes.
    w = wl.normal_weights(40, 256, 0.02, seed=9)
    blob, info = oracle.compress(w)
    sm_blob = np.frombuffer(blob, np.uint8)[info["off_sm"]: info["off_sm"] + w.size]
    raw = ((w >> 8) & 0x80) | (w & 0x7F)
    assert np.array_equal(np.sort(sm_blob), np.sort(raw.ravel().astype(np.uint8)))


def test_decoder_rejects_corruption(oracle):
    w, _ = _worked_matrix()
    blob = bytearray(oracle.compress(w)[0])
    bad = bytearray(blob)
    bad[0] ^= 1
    assert oracle.decompress_status(bytes(bad)) == -1
    bad = bytearray(blob)
    bad[512] = 12                                  # glen says 12 bytes, code has 11
    assert oracle.decompress_status(bytes(bad)) == -3


# ---------------------------------------------------------------- statistics
def test_exponent_statistics_match_the_blog(oracle):
    # Top-16 exponents cover >99% and the entropy is ~2.6 bits (blog, exponent skew).
    w = wl.normal_weights(1024, 1024, 0.02, seed=0)
    c = oracle.histogram(w).astype(np.float64)
    pal = oracle.palette(c.astype(np.uint64))
    assert c[pal].sum() / c.sum() > 0.99
    p = c[c > 0] / c.sum()
    assert 2.4 < -(p * np.log2(p)).sum() < 2.8
    blob, info = oracle.compress(w)
    ratio = len(blob) / (2 * w.size)
    assert 0.66 < ratio < 0.71                     # blog: ~30% fewer MLP bytes


# ---------------------------------------------------------------- fp64 matmul
def test_matmul_one_hot_picks_columns(oracle):
    w = wl.normal_weights(8, 128, 0.02, seed=1)
    x = np.zeros((1, 128), np.uint16)
    x[0, 37] = 0x3F80                                 # 1.0
    y, a = oracle.matmul_f64(x, w)
    assert np.array_equal(y[0], wl.bf16_to_f32(w[:, 37]).astype(np.float64))
    assert np.array_equal(a[0], np.abs(y[0]))


def test_matmul_exact_small_integers(oracle):
    rng = np.random.default_rng(5)
    xi = rng.integers(-8, 9, (3, 64)).astype(np.float32)
    wi = rng.integers(-8, 9, (5, 64)).astype(np.float32)
    y, _ = oracle.matmul_f64(wl.bf16_bits(xi), wl.bf16_bits(wi))
    assert np.array_equal(y, xi.astype(np.int64) @ wi.astype(np.int64).T)


def test_matmul_agrees_with_numpy_and_row_window(oracle):
    w = wl.normal_weights(40, 256, 0.02, seed=2)
    x = wl.activations(2, 256, seed=2)
    ref = wl.bf16_to_f32(x).astype(np.float64) @ wl.bf16_to_f32(w).astype(np.float64).T
    y, a = oracle.matmul_f64(x, w)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-15)
    y2, _ = oracle.matmul_f64(x, w, n0=7, nr=9)
    assert np.array_equal(y2, y[:, 7:16])
    assert np.all(a >= np.abs(y))


def test_swiglu_closed_form(oracle):
    g = wl.bf16_bits(np.array([0.0, 1.0, -2.0, 3.5], np.float32))
    u = wl.bf16_bits(np.array([5.0, 2.0, 1.0, -1.0], np.float32))
    h = oracle.swiglu_f64(g, u)
    z = np.array([0.0, 1.0, -2.0, 3.5])
    assert np.allclose(h, z * (1 / (1 + np.exp(-z))) * np.array([5.0, 2.0, 1.0, -1.0]), rtol=1e-15)
    assert h[0] == 0.0
