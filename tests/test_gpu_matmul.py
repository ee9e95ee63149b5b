"""GPU matmul parity: the fused compressed kernel must equal the same kernel
fed uncompressed BF16 weights bit for bit, and both must lie within
4 * 2^-8 * sum_k |x_k w_k| of the fp64 oracle for every output."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def _case(rows, cols, batch, seed=0, heavy=False):
    w = wl.heavy_tailed_weights(rows, cols, seed=seed) if heavy else wl.normal_weights(rows, cols, 0.02, seed)
    x = wl.activations(batch, cols, seed=seed)
    return w, x


@pytest.mark.parametrize("rows,cols,batch", [
    (1, 64, 1), (32, 64, 1), (77, 192, 1), (100, 2112, 3), (1024, 1024, 1), (256, 4096, 2),
    (64, 512, 4), (96, 1024, 8), (50, 640, 9), (40, 256, 17),
])
def test_fused_equals_uncompressed_and_oracle(g, uw, oracle, rows, cols, batch):
    w, x = _case(rows, cols, batch, seed=rows + cols)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    y_twin = g.matmul_bf16(g.dev_bits(w), xd)
    assert np.array_equal(y, y_twin)
    y_ref, absum = oracle.matmul_f64(x, w)
    g.assert_within_bound(y, y_ref, absum)


@pytest.mark.parametrize("variant", range(27))
def test_every_variant_bit_identical(g, uw, oracle, variant):
    w, x = _case(96, 2048, 1, seed=variant)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    wd = g.dev_bits(w)
    plan = uw.Plan(uw.STRATEGY_FUSED, variant, 1, 0.0)
    y = c.matmul(xd, plan)
    assert np.array_equal(y, g.matmul_bf16(wd, xd, variant))
    plan_d = uw.Plan(uw.STRATEGY_DECOMPRESS_GEMM, variant, 1, 0.0)
    assert np.array_equal(c.matmul(xd, plan_d), y)
    y_ref, absum = oracle.matmul_f64(x, w)
    g.assert_within_bound(y, y_ref, absum)


def test_gate_proj_batch1_full_size(g, uw, oracle):
    # The benchmark's workload: 14336 x 4096, batch 1, every output checked.
    w = wl.workload_weights("gate")
    x = wl.activations(1, 4096, seed=0)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert np.array_equal(y, g.matmul_bf16(g.dev_bits(w), xd))
    y_ref, absum = oracle.matmul_f64(x, w)
    g.assert_within_bound(y, y_ref, absum)


def test_down_proj_shape_split_k(g, uw, oracle):
    w = wl.normal_weights(*wl.DOWN_SHAPE, 0.02, seed=2)
    x = wl.activations(1, wl.DOWN_SHAPE[1], seed=2)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert np.array_equal(y, g.matmul_bf16(g.dev_bits(w), xd))
    y_ref, absum = oracle.matmul_f64(x, w)
    g.assert_within_bound(y, y_ref, absum)


@pytest.mark.parametrize("batch", [1, 16])
def test_heavy_tailed_escapes(g, uw, oracle, batch):
    w, x = _case(4096, 4096, batch, heavy=True)
    c = g.Compressed(w)
    assert c.desc.n_escaped / c.desc.n_groups > 0.03
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert np.array_equal(y, g.matmul_bf16(g.dev_bits(w), xd))
    rows = np.random.default_rng(0).choice(4096, 256, replace=False)
    for n in rows[:64]:
        y_ref, absum = oracle.matmul_f64(x, w, n0=int(n), nr=1)
        g.assert_within_bound(y[:, n:n + 1], y_ref, absum)


def test_repeated_calls_reuse_workspace(g, uw):
    w, x = _case(200, 1024, 1, seed=3)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    plan = uw.Plan(uw.STRATEGY_FUSED, 7, 1, 0.0)     # 8 warps, 4 splits: uses counters
    ws = c.ws(1, plan)
    first = c.matmul(xd, plan, ws)
    for _ in range(5):
        assert np.array_equal(c.matmul(xd, plan, ws), first)


def test_swiglu_within_one_ulp(g, uw, oracle):
    n = 14336 * 3 + 5
    gb = wl.activations(1, n, seed=1)[0]
    ub = wl.activations(1, n, seed=2)[0]
    h = g.empty_bits(n)
    uw.swiglu(g.dev_bits(gb), g.dev_bits(ub), h)
    torch.cuda.synchronize()
    hv = wl.bf16_to_f32(g.host_bits(h)).astype(np.float64)
    ref = oracle.swiglu_f64(gb, ub)
    ulp = np.spacing(np.abs(wl.bf16_to_f32(wl.bf16_bits(ref))).astype(np.float32)).astype(np.float64) * 65536
    assert np.all(np.abs(hv - ref) <= ulp)


def test_autotune_picks_a_runnable_plan(g, uw):
    w, x = _case(2048, 1024, 1, seed=4)
    c = g.Compressed(w)
    nb = uw.autotune_workspace_size(c.desc, [1, 4])
    ws = g.workspace(nb)
    plans = uw.autotune(c.desc, c.blob_dev, [1, 4], ws)
    assert [p.batch for p in plans] == [1, 4]
    for p in plans:
        assert p.us > 0 and p.strategy in (uw.STRATEGY_DECOMPRESS_GEMM, uw.STRATEGY_FUSED, uw.STRATEGY_PALETTE4, uw.STRATEGY_EXPONENT) and 0 <= p.variant < uw.variant_count(p.strategy)
    xd = g.dev_bits(x)
    assert np.array_equal(c.matmul(xd, plans[0]), c.matmul(xd))
