"""Library host side against the oracle (no GPU needed): the blob the
library writes must be byte-identical to the oracle's, its header checks
must reject corrupted blobs, and the shared library must export every
entry point include/uw.h declares."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib(uw):
    return uw


def _declared_functions():
    with open(os.path.join(ROOT, "include", "uw.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(uw_\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 14
    so = ctypes.CDLL(lib.LIB_PATH)
    bound = {n for n, _, _ in lib.SIGNATURES}
    for n in names:
        assert hasattr(so, n), n
        assert n in bound, n


CASES = {
    "small": lambda: wl.normal_weights(256, 1024, 0.02, seed=0),
    "ragged_rows": lambda: wl.normal_weights(77, 192, 0.02, seed=4),
    "one_row": lambda: wl.normal_weights(1, 64, 0.02, seed=5),
    "heavy": lambda: wl.heavy_tailed_weights(512, 512, seed=0),
    "all_patterns": wl.all_bf16_patterns,
    "zeros": lambda: np.zeros((40, 128), np.uint16),
    "wide_sigma": lambda: wl.normal_weights(64, 4096, 0.04, seed=7),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_blob_identical_to_oracle(lib, oracle, name):
    w = CASES[name]()
    ob, oinfo = oracle.compress(w)
    lb = lib.compress(w)
    d = lib.blob_info(lb)
    assert list(d.palette)[: d.n_palette] == oinfo["palette"]
    assert list(d.code_len) == oinfo["code_len"]
    assert d.code_bits == oinfo["code_bits"] and d.n_escaped == oinfo["n_escaped"]
    assert lb.tobytes() == ob
    assert np.array_equal(oracle.decompress(lb.tobytes()), w)


def _random_matrix(rng):
    rows = int(rng.integers(1, 100))
    cols = 64 * int(rng.integers(1, 9))
    kind = int(rng.integers(4))
    if kind == 0:  # normal at a random scale
        sigma = float(10.0 ** rng.uniform(-4, 1))
        return wl.normal_weights(rows, cols, sigma, seed=int(rng.integers(1 << 30)))
    if kind == 1:  # raw random bit patterns: every exponent, most groups escaped
        return rng.integers(0, 1 << 16, (rows, cols)).astype(np.uint16)
    sm = rng.integers(0, 1 << 16, (rows, cols)).astype(np.uint16) & np.uint16(0x807F)
    if kind == 2:  # a few exponents with random weights, a sprinkle of rare ones
        m = int(rng.integers(1, 21))
        vals = rng.choice(256, size=m, replace=False)
        e = vals[rng.choice(m, size=(rows, cols), p=rng.dirichlet(np.ones(m)))]
        rare = rng.random((rows, cols)) < 0.002
        e = np.where(rare, rng.integers(0, 256, (rows, cols)), e)
    else:  # the extremes: zero / subnormal and Inf / NaN exponents mixed with ordinary ones
        e = rng.choice(np.array([0, 0, 255, 120, 121, 122]), size=(rows, cols))
    return (sm | (e.astype(np.uint16) << 7)).astype(np.uint16)


@pytest.mark.parametrize("seed", range(30))
def test_blob_identical_to_oracle_random_matrices(lib, oracle, seed):
    w = _random_matrix(np.random.default_rng(1000 + seed))
    ob, oinfo = oracle.compress(w)
    lb = lib.compress(w)
    assert lb.tobytes() == ob
    assert lib.blob_info_status(lb) == 0
    assert np.array_equal(oracle.decompress(ob), w)


@pytest.mark.parametrize("j", [0, 2])
def test_blob_identical_to_oracle_on_the_extreme_sigma_layers(lib, oracle, j):
    # The 32-layer model's smallest and largest sigma (layers argmin and
    # argmax of the draw), on a slice of rows of the gate and down matrices.
    sig = wl.model_sigmas()
    for layer in (int(np.argmin(sig)), int(np.argmax(sig))):
        w = np.ascontiguousarray(wl.model_matrix(layer, j)[:96])
        ob, _ = oracle.compress(w)
        assert lib.compress(w).tobytes() == ob
        assert np.array_equal(oracle.decompress(ob), w)


def test_blob_identical_to_oracle_gate_proj_shape(lib, oracle):
    w = wl.normal_weights(1024, 4096, 0.02, seed=11)
    assert lib.compress(w).tobytes() == oracle.compress(w)[0]


RAGGED = [(1, 1), (3, 70), (33, 100), (40, 200), (2, 4097), (31, 127), (65, 14335)]


@pytest.mark.parametrize("rows,cols", RAGGED)
def test_blob_identical_to_oracle_ragged_rows(lib, oracle, rows, cols):
    # rows of any length: filler to the next multiple of 64, true cols in the
    # header, the true columns back from the oracle's decompression
    for w in (wl.normal_weights(rows, cols, 0.02, seed=cols), wl.heavy_tailed_weights(rows, cols, seed=rows)):
        ob, _ = oracle.compress(w)
        assert lib.compress(w).tobytes() == ob
        assert np.array_equal(oracle.decompress(ob), w)


def test_blob_identical_to_oracle_ragged_with_escapes(lib, oracle):
    # a rare exponent in the last, partial group of a row escapes that group
    w = wl.normal_weights(40, 1000, 0.02, seed=5)
    w[7, 999] = np.uint16(0x7F80)  # +inf: exponent 255
    w[8, 970] = np.uint16(0x4000)  # 2.0: exponent 128
    ob, info = oracle.compress(w)
    assert info["n_palette"] == 16 and 255 not in info["palette"] and 128 not in info["palette"]
    assert info["n_escaped"] >= 2
    assert lib.compress(w).tobytes() == ob
    assert np.array_equal(oracle.decompress(ob), w)


@pytest.mark.parametrize("seed", range(12))
def test_code_lengths_equal_oracle_on_skewed_histograms(lib, oracle, seed):
    # Random exponent histograms (through real matrices) exercise the code
    # length choice and its tie rule against the oracle's exhaustive search.
    rng = np.random.default_rng(seed)
    m = int(rng.integers(2, 17))
    probs = rng.dirichlet(np.full(m, 0.3 if seed % 2 else 3.0))
    exps = 100 + rng.choice(m, size=(64, 256), p=probs)
    w = ((exps.astype(np.uint16) << 7) | rng.integers(0, 256, (64, 256)).astype(np.uint16) & 0x807F)
    d = lib.blob_info(lib.compress(w))
    _, oinfo = oracle.compress(w)
    assert list(d.code_len) == oinfo["code_len"]


def test_compress_rejects_bad_shapes(lib):
    L = lib.load()
    n = ctypes.c_size_t(0)
    w = np.zeros((4, 64), np.uint16)
    assert L.uw_compress(w.ctypes.data, 0, 64, None, ctypes.byref(n)) == 2
    assert L.uw_compress(w.ctypes.data, 4, 0, None, ctypes.byref(n)) == 2
    assert L.uw_compress(None, 4, 64, None, ctypes.byref(n)) == 1
    assert L.uw_compress(w.ctypes.data, 4, 64, None, ctypes.byref(n)) == 3 and n.value > 0
    assert L.uw_compress(w.ctypes.data, 4, 63, None, ctypes.byref(n)) == 3 and n.value > 0  # ragged rows
    # beyond 2^31 rows or columns (checked before the data is read)
    assert L.uw_compress(w.ctypes.data, 1, (1 << 31) + 64, None, ctypes.byref(n)) == 7
    assert L.uw_compress(w.ctypes.data, (1 << 31) + 1, 64, None, ctypes.byref(n)) == 7


def _corrupt(blob, pos, value):
    b = bytearray(blob.tobytes())
    b[pos] = value
    return bytes(b)


def test_blob_info_rejects_corruption(lib):
    w = wl.normal_weights(64, 256, 0.02, seed=1)
    blob = lib.compress(w)
    d = lib.blob_info(blob)
    assert lib.blob_info_status(blob) == 0
    assert lib.blob_info_status(_corrupt(blob, 0, 0)) == 4                 # magic
    assert lib.blob_info_status(_corrupt(blob, 4, 9)) == 4                 # version
    assert lib.blob_info_status(_corrupt(blob, 24, 32)) == 4               # group size
    assert lib.blob_info_status(_corrupt(blob, 56, 9)) == 4                # code length > 5
    assert lib.blob_info_status(blob[: len(blob) - 256]) == 4              # truncated
    assert lib.blob_info_status(_corrupt(blob, d.off_glen, 0)) == 4        # glen vs tile table
    assert lib.blob_info_status(_corrupt(blob, d.off_glen + 3, 49)) == 4   # glen > 48
    assert lib.blob_info_status(_corrupt(blob, d.off_tcode + 4, 200)) == 4 # tile offsets
    assert lib.blob_info_status(blob.tobytes()[:200]) == 4                  # shorter than header


@pytest.mark.parametrize("name", ["heavy", "normal"])
def test_blob_info_and_oracle_under_random_corruption(lib, oracle, name):
    # Seeded random byte changes in the header, glen and tile tables (the
    # sections a decoder trusts for addresses).  Neither decoder may crash;
    # whatever the library's host check accepts must be structurally sound
    # for the oracle's independent reader too: at most a bad code or a group
    # length that disagrees with its codes, which only decoding can reveal
    # (the GPU reports those through its status word).
    w = (wl.heavy_tailed_weights(96, 512, seed=3) if name == "heavy"
         else wl.normal_weights(70, 256, 0.02, seed=5))
    blob = lib.compress(w).tobytes()
    d = lib.blob_info(blob)
    regions = [(0, 256), (d.off_glen, d.off_tcode), (d.off_tcode, d.off_tesc), (d.off_tesc, d.off_code)]
    rng = np.random.default_rng(11)
    accepted = 0
    for _ in range(1500):
        lo, hi = regions[int(rng.integers(len(regions)))]
        pos = int(rng.integers(lo, hi))
        mb = bytearray(blob)
        new = int(rng.integers(256))
        if new == mb[pos]:
            continue
        mb[pos] = new
        mb = bytes(mb)
        sl = lib.blob_info_status(mb)
        so = oracle.decompress_status(mb)
        assert sl in (0, 4), (pos, new, sl)
        assert so in (0, -1, -2, -3, -4), (pos, new, so)
        if sl == 0:
            accepted += 1
            assert so in (0, -2, -3), (pos, new, so)
    assert accepted > 0
    for cut in rng.integers(0, len(blob), 50):
        assert lib.blob_info_status(blob[:int(cut)]) == 4
        assert oracle.decompress_status(blob[:int(cut)]) == -1


def test_compression_ratio_and_statistics(lib):
    # ~30% fewer bytes for N(0, 0.02) weights (blog: ~30% on MLP weights).
    w = wl.normal_weights(1024, 4096, 0.02, seed=0)
    blob = lib.compress(w)
    d = lib.blob_info(blob)
    ratio = d.blob_bytes / (2 * w.size)
    assert 0.68 < ratio < 0.71, ratio
    # codes limited to 5 bits: about 0.4 bit above the ~2.6-bit entropy
    mean_len = d.code_bits / (64 * (d.n_groups - d.n_escaped))
    assert 2.8 < mean_len < 3.1
    assert d.n_escaped / d.n_groups < 0.01


def test_palette4_host_side(lib):
    w = wl.normal_weights(96, 256, 0.02, seed=2)
    d = lib.blob_info(lib.compress(w))
    assert lib.palette4_bytes(d) == 96 * 256 // 2
    L = lib.load()
    # argument checks happen before any device work
    assert L.uw_transcode_palette4(ctypes.byref(d), None, None, None, 0, None) == 1
    assert L.uw_matmul_palette4(ctypes.byref(d), None, None, None, 1, None, -1, None, 0, None) == 1
    assert lib.variant_count(lib.STRATEGY_PALETTE4) == lib.variant_count(lib.STRATEGY_FUSED)
    assert lib.exponent_bytes(d) == 96 * 256
    assert L.uw_decode_exponents(ctypes.byref(d), None, None, None, 0, None) == 1
    assert L.uw_matmul_exponents(ctypes.byref(d), None, None, None, 1, None, -1, None, 0, None) == 1
    assert lib.variant_count(lib.STRATEGY_EXPONENT) == lib.variant_count(lib.STRATEGY_FUSED)

