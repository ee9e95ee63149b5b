"""Tensor-core path (tcgen05 with the accumulator in tensor memory) for
batches of 16 and up, stream-K over every SM.  The fused kernel decodes each
32 x 64 tile into a tensor-memory A stage; its twin writes the uncompressed
rows there, over the same cut of the units, so the two must agree bit for
bit, and both must lie within 4 * 2^-8 * sum_k |x_k w_k| of the fp64
oracle."""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu

TC_FIRST = 27                      # variants 27..29: tc_g2, tc_g3, tc_g4 (producer groups)
TC_VARIANTS = list(range(TC_FIRST, TC_FIRST + 3))
UNSUPPORTED = 7


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def _check(g, uw, oracle, w, x, variant=-1, sample_rows=None):
    c = g.Compressed(w)
    xd, wd = g.dev_bits(x), g.dev_bits(w)
    plan = uw.Plan(uw.STRATEGY_FUSED, variant, x.shape[0], 0.0)
    if variant >= 0:
        # a variant whose stages do not fit this batch must say so, not run
        probe = g.empty_bits(x.shape[0], w.shape[0])
        st = uw.matmul_status(c.desc, c.blob_dev, xd, probe, c.ws(x.shape[0], plan), plan)
        if st == UNSUPPORTED:
            pytest.skip("variant %s does not fit batch %d" % (uw.variant_name(1, variant), x.shape[0]))
        assert st == 0
    y = c.matmul(xd, plan)
    assert np.array_equal(y, g.matmul_bf16(wd, xd, variant)), "fused != uncompressed twin"
    plan_d = uw.Plan(uw.STRATEGY_DECOMPRESS_GEMM, variant, x.shape[0], 0.0)
    assert np.array_equal(c.matmul(xd, plan_d), y), "decompress-then-GEMM != fused"
    if sample_rows is None:
        y_ref, absum = oracle.matmul_f64(x, w)
        g.assert_within_bound(y, y_ref, absum)
    else:
        for n in sample_rows:
            y_ref, absum = oracle.matmul_f64(x, w, n0=int(n), nr=1)
            g.assert_within_bound(y[:, n:n + 1], y_ref, absum)
    return y


def test_variant_names(uw):
    names = [uw.variant_name(uw.STRATEGY_FUSED, v) for v in TC_VARIANTS]
    assert names == ["tc_g2", "tc_g3", "tc_g4"]


@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_every_tc_variant(g, uw, oracle, variant):
    # 300 rows: three CTAs of 128, the last one ragged (44 rows, two row
    # blocks of it past the matrix); 1024 columns = 16 pipeline stages.
    w = wl.normal_weights(300, 1024, 0.02, seed=variant)
    x = wl.activations(40, 1024, seed=variant)
    _check(g, uw, oracle, w, x, variant)


@pytest.mark.parametrize("rows,cols,batch", [
    (128, 64, 16),        # one CTA, one stage
    (32, 128, 16),        # a single row block
    (1000, 1024, 33),     # padded batch 48
    (256, 2048, 64),
    (512, 1024, 256),     # the widest MMA (N = 256)
    (200, 512, 300),      # two launches: 256 + 44
    (96, 192, 1),         # batch 1 through the tensor cores (padded to 16)
])
def test_shapes_and_batches(g, uw, oracle, rows, cols, batch):
    w = wl.normal_weights(rows, cols, 0.02, seed=rows + batch)
    x = wl.activations(batch, cols, seed=rows + batch)
    for variant in (-1, TC_FIRST, TC_FIRST + 2):  # default, tc_g2, tc_g4
        _check(g, uw, oracle, w, x, variant)


def test_default_plan_matches_a_tc_variant(g, uw):
    # From batch 16 the default plan runs one of the tensor-core variants.
    w = wl.normal_weights(640, 2048, 0.02, seed=11)
    x = wl.activations(16, 2048, seed=11)
    c = g.Compressed(w)
    xd = g.dev_bits(x)
    y = c.matmul(xd)
    assert any(np.array_equal(y, c.matmul(xd, uw.Plan(uw.STRATEGY_FUSED, v, 16, 0.0))) for v in TC_VARIANTS)


def test_heavy_tailed_escapes_through_tensor_cores(g, uw, oracle):
    w = wl.heavy_tailed_weights(4096, 4096, seed=5)
    x = wl.activations(64, 4096, seed=5)
    rows = np.random.default_rng(5).choice(4096, 48, replace=False)
    c = g.Compressed(w)
    assert c.desc.n_escaped / c.desc.n_groups > 0.03
    _check(g, uw, oracle, w, x, -1, sample_rows=rows)


@pytest.mark.parametrize("batch", [16, 64, 256])
def test_gate_proj_full_size(g, uw, oracle, batch):
    w = wl.workload_weights("gate")
    x = wl.activations(batch, 4096, seed=batch)
    rows = np.random.default_rng(batch).choice(14336, 24, replace=False)
    _check(g, uw, oracle, w, x, -1, sample_rows=rows)


def test_down_proj_full_size(g, uw, oracle):
    w = wl.normal_weights(*wl.DOWN_SHAPE, 0.02, seed=7)
    x = wl.activations(32, wl.DOWN_SHAPE[1], seed=7)
    rows = np.random.default_rng(7).choice(wl.DOWN_SHAPE[0], 24, replace=False)
    _check(g, uw, oracle, w, x, TC_FIRST + 1, sample_rows=rows)   # tc_g3
