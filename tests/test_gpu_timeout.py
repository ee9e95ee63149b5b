"""Failure detection without a GPU fault: a kernel whose bounded wait runs
out (a barrier that nothing arrives on) must set the timeout flag and
return; uw_check_status reports UW_ERR_TIMEOUT, clears the word, and the
context keeps working (a matmul afterwards is still right)."""
import numpy as np
import pytest

import workloads as wl

pytestmark = pytest.mark.gpu

UW_ERR_TIMEOUT = 6


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


@pytest.mark.parametrize("tries", [1, 64, 4096])
def test_withheld_arrival_reports_timeout(g, uw, tries):
    ws = g.workspace(256)
    uw.selftest_bounded_wait(ws, tries)
    assert uw.check_status(ws) == UW_ERR_TIMEOUT
    assert uw.check_status(ws) == 0          # read once, then cleared


def test_context_usable_after_timeout(g, uw, oracle):
    ws = g.workspace(256)
    uw.selftest_bounded_wait(ws, 1000)
    assert uw.check_status(ws) == UW_ERR_TIMEOUT
    w = wl.normal_weights(256, 1024, 0.02, seed=3)
    x = wl.activations(1, 1024, seed=3)
    c = g.Compressed(w)
    y = c.matmul(g.dev_bits(x))
    y_ref, absum = oracle.matmul_f64(x, w)
    g.assert_within_bound(y, y_ref, absum)


def test_tries_outside_the_limit_are_refused(g, uw):
    ws = g.workspace(256)
    L = uw.load()
    assert L.uw_selftest_bounded_wait(ws.data_ptr(), 256, 0, None) == 1
    assert L.uw_selftest_bounded_wait(ws.data_ptr(), 256, (1 << 22) + 1, None) == 1
