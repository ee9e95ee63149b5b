"""Rows whose length is not a multiple of 64.  The blob stores each row
extended to the next multiple with filler weights and keeps the true column
count; decompression must give back exactly the original matrix (nothing
written past its true columns), and every matmul path must stay bit-identical
to the uncompressed kernel of the same variant (fed the true-width weights)
and within 4 * 2^-8 * sum_k |x_k w_k| of the fp64 oracle.

cols 100, 127 and 14335 have a row pitch that is not a multiple of 16 bytes
(element-wise stores in the decompression); cols 200 and 4104 do (the
tensor-map store path, which drops the filler columns)."""
import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu

SHAPES = [(96, 100), (64, 4097), (33, 14335), (40, 200), (1, 1), (31, 127), (300, 4104)]
COL_W16X1, TC = 17, (27, 28, 29)   # col_w16x1, tc_g2 / tc_g3 / tc_g4
ROW = (1, 4, 7, 10, 13)            # w8s1 .. w8s16: K split 1 to 16 ways (long rows need the splits)
UNSUPPORTED = 7                    # UW_ERR_UNSUPPORTED: the variant does not fit this shape


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def _weights(rows, cols, heavy):
    return wl.heavy_tailed_weights(rows, cols, seed=rows + cols) if heavy else \
        wl.normal_weights(rows, cols, 0.02, seed=rows + cols)


@pytest.mark.parametrize("heavy", [False, True])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_decompress_gives_back_the_true_columns(g, uw, oracle, rows, cols, heavy):
    w = _weights(rows, cols, heavy)
    c = g.Compressed(w)
    assert c.blob.tobytes() == oracle.compress(w)[0]
    guard = 4096
    out = torch.full((rows * cols + guard,), 0x5A5A, dtype=torch.int16, device="cuda")
    ws = c.ws()
    uw.decompress(c.desc, c.blob_dev, out, ws)
    assert uw.check_status(ws) == 0
    got = g.host_bits(out)
    assert np.array_equal(got[: rows * cols].reshape(rows, cols), oracle.decompress(c.blob.tobytes()))
    assert np.array_equal(got[: rows * cols].reshape(rows, cols), w)
    assert np.all(got[rows * cols:] == 0x5A5A), "decompression wrote past the matrix"


def _check(g, uw, oracle, c, x, strategy, variant, may_not_fit=False):
    xd, wd = g.dev_bits(x), g.dev_bits(c.w)
    plan = uw.Plan(strategy, variant, x.shape[0], 0.0)
    y = g.empty_bits(x.shape[0], c.desc.rows)
    ws = c.ws(x.shape[0], plan)
    st = uw.matmul_status(c.desc, c.blob_dev, xd, y, ws, plan)
    if may_not_fit and st == UNSUPPORTED:
        return None
    assert st == 0, uw.status_string(st)
    assert uw.check_status(ws) == 0
    yh = g.host_bits(y)
    assert np.array_equal(yh, g.matmul_bf16(wd, xd, variant)), "not the uncompressed kernel's result"
    y_ref, absum = oracle.matmul_f64(x, c.w)
    g.assert_within_bound(yh, y_ref, absum)
    return yh


STRATEGIES = ["FUSED", "DECOMPRESS_GEMM", "PALETTE4", "EXPONENT"]


@pytest.mark.parametrize("strategy", STRATEGIES)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_batch1_column_kernel(g, uw, oracle, rows, cols, strategy):
    c = g.Compressed(_weights(rows, cols, True))
    x = wl.activations(1, cols, seed=cols)
    _check(g, uw, oracle, c, x, getattr(uw, "STRATEGY_" + strategy), COL_W16X1)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_row_kernel(g, uw, oracle, rows, cols):
    c = g.Compressed(_weights(rows, cols, False))
    x = wl.activations(3, cols, seed=cols)
    ran = 0
    for v in ROW:  # the variants whose shared memory holds this row length
        y = _check(g, uw, oracle, c, x, uw.STRATEGY_FUSED, v, may_not_fit=True)
        if y is not None:
            ran += 1
            assert np.array_equal(y, _check(g, uw, oracle, c, x, uw.STRATEGY_DECOMPRESS_GEMM, v))
    assert ran > 0


@pytest.mark.parametrize("strategy", STRATEGIES)
@pytest.mark.parametrize("batch", [16, 64])
@pytest.mark.parametrize("rows,cols", [(96, 100), (300, 4097), (130, 14335), (40, 200)])
def test_tensor_core_kernels(g, uw, oracle, rows, cols, batch, strategy):
    c = g.Compressed(_weights(rows, cols, True))
    x = wl.activations(batch, cols, seed=batch + cols)
    for v in TC:
        _check(g, uw, oracle, c, x, getattr(uw, "STRATEGY_" + strategy), v)


@pytest.mark.parametrize("rows,cols", [(96, 100), (33, 14335)])
def test_default_plans(g, uw, oracle, rows, cols):
    c = g.Compressed(_weights(rows, cols, True))
    for batch in (1, 5, 32):
        x = wl.activations(batch, cols, seed=batch)
        y_ref, absum = oracle.matmul_f64(x, c.w)
        g.assert_within_bound(c.matmul(g.dev_bits(x)), y_ref, absum)


@pytest.mark.parametrize("form", ["palette4", "exponent"])
@pytest.mark.parametrize("rows,cols", [(96, 100), (33, 4097)])
def test_forms_have_the_stored_width(g, uw, oracle, rows, cols, form):
    w = _weights(rows, cols, True)
    c = g.Compressed(w)
    pal = list(c.desc.palette)[: c.desc.n_palette]
    wp = oracle.pad(w, pal)
    ws = c.ws()
    if form == "palette4":
        out = torch.empty(uw.palette4_bytes(c.desc), dtype=torch.uint8, device="cuda")
        uw.transcode_palette4(c.desc, c.blob_dev, out, ws)
        want = oracle.palette4(wp, pal)
    else:
        out = torch.empty(uw.exponent_bytes(c.desc), dtype=torch.uint8, device="cuda")
        uw.decode_exponents(c.desc, c.blob_dev, out, ws)
        want = oracle.exponents(wp)
    assert uw.check_status(ws) == 0
    assert np.array_equal(out.cpu().numpy(), want)

