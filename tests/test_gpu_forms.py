"""Palette and exponent-only pipelines (the Unweight blog's palette transcode
at run time / direct palette at model load, and exponent-only decode): the
Huffman codes turned into 4-bit palette indices, or into exponent bytes, on
the GPU, and matmuls that rebuild BF16 from those forms.

Checks: each form equals the oracle's byte for byte (escaped groups
included, ragged row blocks included); every matmul output from a form
equals the same kernel fed uncompressed BF16 weights bit for bit, and lies
within 4 * 2^-8 * sum_k |x_k w_k| of the fp64 oracle; the PALETTE4 and
EXPONENT strategies of uw_matmul give the same bits as the fused Huffman
path with the same variant."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

COL_VARIANTS = list(range(15, 27))   # col_w{4,8,16}x{1..4}
TC_VARIANTS = list(range(27, 30))    # tc_g2, tc_g3, tc_g4
UNSUPPORTED = 7


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


FORMS = ["palette4", "exponent"]


def _form(g, uw, c, form):
    n = uw.palette4_bytes(c.desc) if form == "palette4" else uw.exponent_bytes(c.desc)
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    ws = c.ws()
    (uw.transcode_palette4 if form == "palette4" else uw.decode_exponents)(c.desc, c.blob_dev, out, ws)
    assert uw.check_status(ws) == 0
    return out


def _oracle_form(oracle, c, form):
    if form == "palette4":
        return oracle.palette4(c.w, list(c.desc.palette)[: c.desc.n_palette])
    return oracle.exponents(c.w)


def _check_matmul(g, uw, oracle, c, fdev, x, variant, form, sample_rows=None):
    xd, wd = g.dev_bits(x), g.dev_bits(c.w)
    plan = uw.Plan(uw.STRATEGY_FUSED, variant, x.shape[0], 0.0)
    ws = c.ws(x.shape[0], plan)
    y = g.empty_bits(x.shape[0], c.desc.rows)
    call = uw.matmul_palette4_status if form == "palette4" else uw.matmul_exponents_status
    st = call(c.desc, c.blob_dev, fdev, xd, y, ws, variant)
    if st == UNSUPPORTED:
        pytest.skip("variant %s does not fit batch %d" % (uw.variant_name(1, variant), x.shape[0]))
    assert st == 0
    assert uw.check_status(ws) == 0
    yh = g.host_bits(y)
    assert np.array_equal(yh, g.matmul_bf16(wd, xd, variant)), form + " != uncompressed twin"
    rows = range(c.desc.rows) if sample_rows is None else sample_rows
    if sample_rows is None:
        y_ref, absum = oracle.matmul_f64(x, c.w)
        g.assert_within_bound(yh, y_ref, absum)
    else:
        for n in rows:
            y_ref, absum = oracle.matmul_f64(x, c.w, n0=int(n), nr=1)
            g.assert_within_bound(yh[:, n:n + 1], y_ref, absum)
    return yh


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("shape,kind", [
    ((1, 64), "normal"), ((33, 128), "normal"), ((300, 1024), "normal"),
    ((70, 192), "heavy"), ((4096, 4096), "heavy"), ((14336, 4096), "gate"),
])
def test_form_matches_oracle(g, uw, oracle, shape, kind, form):
    if kind == "gate":
        w = wl.workload_weights("gate")
    elif kind == "heavy":
        w = wl.heavy_tailed_weights(*shape, seed=shape[0])
    else:
        w = wl.normal_weights(*shape, 0.02, seed=shape[0])
    c = g.Compressed(w)
    assert np.array_equal(_form(g, uw, c, form).cpu().numpy(), _oracle_form(oracle, c, form))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("variant", COL_VARIANTS)
def test_every_column_variant(g, uw, oracle, variant, form):
    # 300 rows: ten row blocks, the last ragged (12 rows); heavy tails for escapes
    w = wl.heavy_tailed_weights(300, 1024, seed=variant)
    c = g.Compressed(w)
    assert c.desc.n_escaped > 0
    x = wl.activations(1, 1024, seed=variant)
    _check_matmul(g, uw, oracle, c, _form(g, uw, c, form), x, variant, form)


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("variant", TC_VARIANTS)
def test_every_tc_variant(g, uw, oracle, variant, form):
    w = wl.heavy_tailed_weights(300, 1024, seed=100 + variant)
    c = g.Compressed(w)
    x = wl.activations(40, 1024, seed=variant)
    _check_matmul(g, uw, oracle, c, _form(g, uw, c, form), x, variant, form)


@pytest.fixture(scope="module")
def gate(g):
    return g.Compressed(wl.workload_weights("gate"))


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("batch", [1, 16, 64, 256])
def test_gate_proj_full_size(g, uw, oracle, gate, batch, form):
    x = wl.activations(batch, 4096, seed=batch)
    rows = np.random.default_rng(batch).choice(14336, 24, replace=False)
    _check_matmul(g, uw, oracle, gate, _form(g, uw, gate, form), x, -1, form, sample_rows=rows)


def test_strategy_palette4_equals_fused(g, uw):
    w = wl.heavy_tailed_weights(640, 2048, seed=3)
    c = g.Compressed(w)
    for batch, variant in ((1, 17), (16, 28), (48, 27)):
        xd = g.dev_bits(wl.activations(batch, 2048, seed=batch))
        fused = c.matmul(xd, uw.Plan(uw.STRATEGY_FUSED, variant, batch, 0.0))
        for strategy in (uw.STRATEGY_PALETTE4, uw.STRATEGY_EXPONENT):
            assert np.array_equal(fused, c.matmul(xd, uw.Plan(strategy, variant, batch, 0.0)))
    # batch 4 has no palette-4 row kernel: the strategy's default is a tensor-core variant
    x = wl.activations(4, 2048, seed=4)
    xd, wd = g.dev_bits(x), g.dev_bits(w)
    pal = c.matmul(xd, uw.Plan(uw.STRATEGY_PALETTE4, -1, 4, 0.0))
    assert any(np.array_equal(pal, g.matmul_bf16(wd, xd, v)) for v in TC_VARIANTS)


def test_row_variant_is_unsupported(g, uw):
    c = g.Compressed(wl.normal_weights(64, 256, 0.02, seed=1))
    xd = g.dev_bits(wl.activations(4, 256, seed=1))
    y = g.empty_bits(4, 64)
    ws = c.ws(4)
    assert uw.matmul_palette4_status(c.desc, c.blob_dev, _form(g, uw, c, "palette4"), xd, y, ws, 0) == UNSUPPORTED
    assert uw.matmul_exponents_status(c.desc, c.blob_dev, _form(g, uw, c, "exponent"), xd, y, ws, 0) == UNSUPPORTED


def _all_escaped():
    k = np.arange(64)
    row = (((100 + k % 32) << 7) | k).astype(np.uint16)   # 32 distinct exponents in every group
    return np.tile(row, (70, 5))


DEGENERATE = [
    ("one_group", lambda: wl.normal_weights(1, 64, 0.02, seed=1)),
    ("tile_edges", lambda: wl.normal_weights(33, 2112, 0.02, seed=3)),
    ("all_patterns", wl.all_bf16_patterns),                # NaN, Inf, subnormals, zeros
    ("zeros", lambda: np.zeros((40, 128), np.uint16)),
    ("all_escaped", _all_escaped),
    ("one_exponent", lambda: (((np.arange(96 * 256) % 2) << 15) | (118 << 7) | (np.arange(96 * 256) % 128))
     .astype(np.uint16).reshape(96, 256)),
]


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("name", [d[0] for d in DEGENERATE])
def test_degenerate_matrices(g, uw, oracle, name, form):
    # The form byte for byte, and the matmul from it bit-identical to the
    # uncompressed twin (non-finite weights included) for a column and a
    # tensor-core variant.
    w = dict(DEGENERATE)[name]()
    c = g.Compressed(w)
    fdev = _form(g, uw, c, form)
    assert np.array_equal(fdev.cpu().numpy(), _oracle_form(oracle, c, form))
    wd = g.dev_bits(w)
    call = uw.matmul_palette4_status if form == "palette4" else uw.matmul_exponents_status
    for batch, variant in ((1, 17), (16, 28)):
        x = wl.activations(batch, w.shape[1], seed=batch)
        xd = g.dev_bits(x)
        ws = c.ws(batch, uw.Plan(uw.STRATEGY_FUSED, variant, batch, 0.0))
        y = g.empty_bits(batch, w.shape[0])
        assert call(c.desc, c.blob_dev, fdev, xd, y, ws, variant) == 0
        assert uw.check_status(ws) == 0
        assert np.array_equal(g.host_bits(y), g.matmul_bf16(wd, xd, variant))

