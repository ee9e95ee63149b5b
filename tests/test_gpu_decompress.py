"""GPU decompression (uw_decompress) must restore every weight bit-exactly:
the method is lossless (Unweight blog, results paragraph: 100% bit-exact)."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


SHAPES = [
    ("one_group", lambda: wl.normal_weights(1, 64, 0.02, seed=1)),
    ("ragged", lambda: wl.normal_weights(77, 192, 0.02, seed=2)),
    ("tile_edges", lambda: wl.normal_weights(33, 2112, 0.02, seed=3)),
    ("small", lambda: wl.workload_weights("small")),
    ("all_patterns", wl.all_bf16_patterns),
    ("zeros", lambda: np.zeros((40, 128), np.uint16)),
    ("heavy", lambda: wl.workload_weights("heavy")),
    ("sigma_0.04", lambda: wl.normal_weights(512, 1024, 0.04, seed=9)),
]


@pytest.mark.parametrize("name", [s[0] for s in SHAPES])
def test_decompress_bit_exact(g, name):
    w = dict(SHAPES)[name]()
    c = g.Compressed(w)
    assert np.array_equal(c.decompress(), w)


def test_decompress_gate_proj_full_size(g):
    w = wl.workload_weights("gate")
    c = g.Compressed(w)
    assert c.desc.rows == 14336 and c.desc.cols == 4096
    assert np.array_equal(c.decompress(), w)


def test_decompress_down_proj_full_size(g):
    w = wl.normal_weights(*wl.DOWN_SHAPE, 0.02, seed=2)
    c = g.Compressed(w)
    assert np.array_equal(c.decompress(), w)


def test_gpu_decodes_oracle_blobs(g, oracle):
    # The oracle's own encoder output goes through the library's GPU decoder.
    for w in (wl.normal_weights(70, 256, 0.02, seed=5), wl.heavy_tailed_weights(128, 512, seed=1),
              wl.all_bf16_patterns()):
        blob, _ = oracle.compress(w)
        c = g.Compressed(w, blob=np.frombuffer(blob, np.uint8).copy())
        assert np.array_equal(c.decompress(), w)


def test_all_escaped_matrix(g):
    k = np.arange(64)
    row = (((100 + k % 32) << 7) | k).astype(np.uint16)
    w = np.tile(row, (70, 5))
    c = g.Compressed(w)
    assert c.desc.n_escaped == c.desc.n_groups
    assert np.array_equal(c.decompress(), w)


def test_device_detects_corruption_after_header_check(g, uw):
    # The header (host copy) is valid; the device copy is then damaged.  The
    # kernel must flag it in the workspace instead of faulting.
    w = wl.normal_weights(64, 512, 0.02, seed=7)
    c = g.Compressed(w)
    d = c.desc
    out = g.empty_bits(d.rows, d.cols)
    # (1) one group claims one more code byte than its codes use
    blob = c.blob.copy()
    blob[d.off_glen + 5] += 1
    bad = torch.from_numpy(blob).cuda()
    ws = c.ws()
    uw.decompress(d, bad, out, ws)
    assert uw.check_status(ws) == 4
    # (2) a tile offset points far past the code section
    blob = c.blob.copy()
    blob[d.off_tcode + 4 * 3: d.off_tcode + 4 * 4] = np.frombuffer(np.uint32(1 << 30).tobytes(), np.uint8)
    bad = torch.from_numpy(blob).cuda()
    uw.decompress(d, bad, out, ws)
    assert uw.check_status(ws) == 4
    # the workspace is usable again afterwards
    uw.decompress(d, c.blob_dev, out, ws)
    assert uw.check_status(ws) == 0
    assert np.array_equal(g.host_bits(out), w)
