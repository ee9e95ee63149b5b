"""Host-side logic of the MLP chain (no GPU): workspace sizing by plan and
schedule, and argument checks that return before any device work."""
import numpy as np
import pytest

import workloads as wl

D, F = 256, 512


@pytest.fixture(scope="module")
def layer(uw):
    out = []
    for (rows, cols), seed in zip([(F, D), (F, D), (D, F)], (1, 2, 3)):
        w = wl.normal_weights(rows, cols, 0.02, seed)
        blob = uw.compress(w)
        out.append((uw.blob_info(blob), blob))
    return out


def mats(uw, layer, strategies, forms=(None, None, None), n_layers=1):
    fake = np.zeros(64, np.uint8)  # never dereferenced by the host-side checks
    entries = []
    for _ in range(n_layers):
        for (d, blob), st, form in zip(layer, strategies, forms):
            entries.append((d, blob, form, uw.Plan(st, -1, 0, 0.0)))
    return uw.mlp_matrices(entries), fake


def test_workspace_grows_with_the_preprocess_slots(uw, layer):
    batch = 32
    fused, _ = mats(uw, layer, [uw.STRATEGY_FUSED] * 3)
    expo, _ = mats(uw, layer, [uw.STRATEGY_EXPONENT] * 3)
    pal, _ = mats(uw, layer, [uw.STRATEGY_PALETTE4] * 3)
    dec, _ = mats(uw, layer, [uw.STRATEGY_DECOMPRESS_GEMM] * 3)
    two, one = uw.Schedule(2, 0), uw.Schedule(1, 0)
    n = D * F
    base = uw.mlp_workspace_size(fused, batch, two)
    # activations alone: x ping-pong [batch, D] and g, u, h [batch, F]
    assert base >= 2 * 2 * batch * D + 3 * 2 * batch * F
    assert uw.mlp_workspace_size(fused, batch, one) == base  # no hard matrix: no slot
    for m, form in ((pal, n // 2), (expo, n), (dec, 2 * n)):
        w2, w1 = uw.mlp_workspace_size(m, batch, two), uw.mlp_workspace_size(m, batch, one)
        assert w2 - w1 == form  # one slot holds the largest form (sizes here are 256-byte multiples)
        assert w1 >= base + form - 4096
    # an easy matrix (palette-4 form made at load) needs no slot
    easy, _ = mats(uw, layer, [uw.STRATEGY_PALETTE4] * 3, forms=[np.zeros(16, np.uint8)] * 3)
    assert uw.mlp_workspace_size(easy, batch, two) == uw.mlp_workspace_size(easy, batch, one)
    # NULL schedule = two slots
    assert uw.mlp_workspace_size(expo, batch, None) == uw.mlp_workspace_size(expo, batch, two)


def test_autotune_workspace_covers_every_candidate(uw, layer):
    for batch in (1, 32):
        fused, _ = mats(uw, layer, [uw.STRATEGY_FUSED] * 3)
        dec, _ = mats(uw, layer, [uw.STRATEGY_DECOMPRESS_GEMM] * 3)
        assert uw.mlp_autotune_workspace_size(fused, batch) >= uw.mlp_workspace_size(dec, batch, None)


def test_chain_argument_checks(uw, layer):
    m, fake = mats(uw, layer, [uw.STRATEGY_EXPONENT] * 3)
    L = uw.load()

    def fwd(mm, n_layers, sched=None, ws_bytes=1 << 30, x=fake):
        return L.uw_mlp_forward(mm, n_layers, x.ctypes.data, 4, fake.ctypes.data,
                                None if sched is None else __import__("ctypes").byref(sched),
                                fake.ctypes.data, ws_bytes, None, None)
    assert fwd(m, 1, ws_bytes=1024) == 3                 # UW_ERR_BUFFER_TOO_SMALL
    assert fwd(m, 1, uw.Schedule(3, 0)) == 1             # more than two slots
    assert fwd(m, 1, uw.Schedule(2, -1)) == 1            # negative split
    assert fwd(m, 0) == 1                                # no layer
    assert fwd(m, 1, x=fake[1:]) == 1                    # x not 16-byte aligned
    # shapes: the down projection must map F back to D
    (dg, bg), (du, bu), (dd, bd) = layer
    bad = uw.mlp_matrices([(dg, bg, None, None), (du, bu, None, None), (dg, bg, None, None)])
    assert fwd(bad, 1) == 2                              # UW_ERR_SHAPE
    # a load-time form must be 16-byte aligned
    mis, _ = mats(uw, layer, [uw.STRATEGY_PALETTE4] * 3, forms=[fake[1:]] * 3)
    assert fwd(mis, 1) == 1


def test_chain_refuses_ragged_rows(uw):
    # consistent shapes, but D = 100 is not a multiple of 64: the chain keeps
    # whole groups (the single matmuls take ragged rows)
    fake = np.zeros(64, np.uint8)
    entries = []
    for (rows, cols), seed in zip([(128, 100), (128, 100), (100, 128)], (1, 2, 3)):
        blob = uw.compress(wl.normal_weights(rows, cols, 0.02, seed))
        entries.append((uw.blob_info(blob), blob, None, None))
    m = uw.mlp_matrices(entries)
    L = uw.load()
    assert L.uw_mlp_forward(m, 1, fake.ctypes.data, 4, fake.ctypes.data, None, fake.ctypes.data, 1 << 30,
                            None, None) == 2         # UW_ERR_SHAPE
