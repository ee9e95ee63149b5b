"""The measured workloads end to end on the GPU, at the sizes they are
measured at: the Llama-3.1-8B-shaped SwiGLU MLP layer at batches 1, 8 and 32,
the heavy-tailed 4096 x 4096 matrix (rare exponents, escaped groups) at
batches 1, 16, 64 and 256, and a slice of the 32-layer model with the
autotuner choosing the plan per matrix and batch.

Checks: every fused output equals the same kernel fed uncompressed BF16
weights bit for bit; every MLP output at batch <= 8, and sampled outputs
elsewhere, lie within 4 * 2^-8 * sum_k |x_k w_k| of
the fp64 oracle; the SwiGLU output lies within one BF16 ulp of silu(g) * u
computed in fp64 from the GPU's own g and u; the down projection is checked
against the oracle fed the GPU's h, so that stage-to-stage rounding does not
compound."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def _sample_rows(n, k, seed):
    return np.random.default_rng(seed).choice(n, k, replace=False)


def _check_rows(g, oracle, x, w, y, rows):
    for n in rows:
        y_ref, absum = oracle.matmul_f64(x, w, n0=int(n), nr=1)
        g.assert_within_bound(y[:, n:n + 1], y_ref, absum)


def _check_all_or_rows(g, oracle, x, w, y, rows):
    if rows is None:
        y_ref, absum = oracle.matmul_f64(x, w)
        g.assert_within_bound(y, y_ref, absum)
    else:
        _check_rows(g, oracle, x, w, y, rows)


@pytest.fixture(scope="module")
def mlp(g):
    mats = []
    for shape, seed in zip(wl.WORKLOADS["mlp"]["shapes"], wl.WORKLOADS["mlp"]["seeds"]):
        w = wl.normal_weights(*shape, wl.WORKLOADS["mlp"]["sigma"], seed)
        mats.append((w, g.Compressed(w), g.dev_bits(w)))
    return mats


@pytest.mark.parametrize("batch", wl.WORKLOADS["mlp"]["batches"])
def test_mlp_layer(g, uw, oracle, mlp, batch):
    (wg, cg, wgd), (wu, cu, wud), (wd, cd, wdd) = mlp
    x = wl.activations(batch, wl.GATE_SHAPE[1], seed=batch)
    xd = g.dev_bits(x)
    gate = cg.matmul(xd)
    up = cu.matmul(xd)
    assert np.array_equal(gate, g.matmul_bf16(wgd, xd))
    assert np.array_equal(up, g.matmul_bf16(wud, xd))
    # every output at batch <= 8, a seeded sample of rows above that
    full = batch <= 8
    rows = None if full else _sample_rows(wl.GATE_SHAPE[0], 16, batch)
    _check_all_or_rows(g, oracle, x, wg, gate, rows)
    _check_all_or_rows(g, oracle, x, wu, up, rows)

    h_dev = g.empty_bits(batch, wl.GATE_SHAPE[0])
    uw.swiglu(g.dev_bits(gate), g.dev_bits(up), h_dev)
    torch.cuda.synchronize()
    h = g.host_bits(h_dev)
    h_ref = oracle.swiglu_f64(gate, up).reshape(h.shape)
    hv = wl.bf16_to_f32(h).astype(np.float64)
    ulp = np.spacing(np.abs(wl.bf16_to_f32(wl.bf16_bits(h_ref))).astype(np.float32)).astype(np.float64) * 65536
    assert np.all(np.abs(hv - h_ref) <= ulp)

    y = cd.matmul(h_dev)
    assert np.array_equal(y, g.matmul_bf16(wdd, h_dev))
    _check_all_or_rows(g, oracle, h, wd, y, None if full else _sample_rows(wl.DOWN_SHAPE[0], 16, batch + 1))


@pytest.fixture(scope="module")
def heavy(g):
    w = wl.workload_weights("heavy")
    return w, g.Compressed(w), g.dev_bits(w)


def test_heavy_tailed_blob(g, heavy):
    w, c, _ = heavy
    frac = c.desc.n_escaped / c.desc.n_groups
    assert 0.05 < frac < 0.10                      # about 7.5% of groups escaped
    assert np.array_equal(c.decompress(), w)


@pytest.mark.parametrize("batch", wl.WORKLOADS["heavy"]["batches"])
def test_heavy_tailed_batches(g, uw, oracle, heavy, batch):
    w, c, wd = heavy
    x = wl.activations(batch, w.shape[1], seed=batch)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert np.array_equal(y, g.matmul_bf16(wd, xd))
    _check_rows(g, oracle, x, w, y, _sample_rows(w.shape[0], 16, batch))


def test_model_slice_autotuned(g, uw, oracle):
    # The first and the last layer of the 32-layer model, every matrix
    # autotuned over a spread of batches (the layers with the smallest and
    # largest sigma are compared with the oracle on the CPU).
    batches = [1, 16, 256]
    for layer in (0, 31):
        for j in range(3):
            w = wl.model_matrix(layer, j)
            c = g.Compressed(w)
            assert np.array_equal(c.decompress(), w)
            ws = g.workspace(uw.autotune_workspace_size(c.desc, batches))
            plans = uw.autotune(c.desc, c.blob_dev, batches, ws)
            wdev = g.dev_bits(w)
            for plan in plans:
                x = wl.activations(plan.batch, w.shape[1], seed=layer * 3 + j)
                xd = g.dev_bits(x)
                y = c.matmul(xd, plan)
                assert np.array_equal(y, g.matmul_bf16(wdev, xd, plan.variant))
                _check_rows(g, oracle, x, w, y, _sample_rows(w.shape[0], 4, plan.batch))


@pytest.mark.parametrize("shape", [(4096, 4096), (1024, 4096)])
@pytest.mark.parametrize("batch", [1, 16])
def test_attention_projection_shapes(g, uw, oracle, shape, batch):
    # Matrices outside the MLP: the Llama-3.1-8B-shaped attention projections
    # (q and o 4096 x 4096; k and v 1024 x 4096 with grouped-query heads).
    w = wl.normal_weights(*shape, 0.02, seed=shape[0] + batch)
    c = g.Compressed(w)
    assert np.array_equal(c.decompress(), w)
    x = wl.activations(batch, shape[1], seed=batch)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert np.array_equal(y, g.matmul_bf16(g.dev_bits(w), xd))   # both take the default variant
    _check_rows(g, oracle, x, w, y, _sample_rows(shape[0], 16, batch))

