"""uw_matmul_noalloc: the fused matmul for callers that cannot allocate device
memory (code where cudaMalloc is not allowed or would synchronise, plug-ins
whose host owns all device memory).  Its scratch is a fixed 1 MiB array
inside the library.  Called straight through the C ABI, it must give the
same output as uw_matmul with a caller workspace, on two calls in a row
(the array keeps the previous call's contents, so the second call checks
that the library clears what has to start at zero).

This file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g(uw):
    from tests import _gpu
    return _gpu


def _call(uw, desc, blob_dev, xd, yd):
    so = ctypes.CDLL(uw.LIB_PATH)
    fn = so.uw_matmul_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(uw.Desc), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                   ctypes.c_void_p, ctypes.c_void_p]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = fn(ctypes.byref(desc), blob_dev.data_ptr(), xd.data_ptr(), xd.shape[0], yd.data_ptr(), stream)
    torch.cuda.synchronize()
    return status


# (64, 4096, 4): two row blocks, so the default row kernel splits K and the
# second call reuses arrival counters and partial sums the first one left;
# (1024, 1024, 16): the tensor-core kernel; (96, 100, 1) and (33, 4097, 3):
# ragged rows, whose zero-extended activations sit in the scratch too.
@pytest.mark.parametrize("rows,cols,batch", [(1024, 1024, 1), (4096, 14336, 1), (300, 640, 5), (64, 4096, 4),
                                             (1024, 1024, 16), (96, 100, 1), (33, 4097, 3)])
def test_noalloc_matches_workspace_entry_point_twice(g, uw, oracle, rows, cols, batch):
    w = wl.normal_weights(rows, cols, 0.02, seed=rows)
    x = wl.activations(batch, cols, seed=rows)
    c = g.Compressed(w)
    assert uw.workspace_size(c.desc, batch) <= (1 << 20)
    xd = g.dev_bits(x)
    expected = c.matmul(xd)                      # uw_matmul with a caller workspace, default plan
    y_ref, absum = oracle.matmul_f64(x, w)
    for _ in range(2):
        yd = g.empty_bits(batch, rows)
        yd.fill_(0x7FC0)                         # stale contents must not leak through
        assert _call(uw, c.desc, c.blob_dev, xd, yd) == 0
        y = g.host_bits(yd)
        g.assert_within_bound(y, y_ref, absum)
        assert np.array_equal(y, expected)


def test_noalloc_rejects_requests_beyond_its_scratch(g, uw):
    # 100,000 rows at batch 8 need ~3 MB of split partial sums: more than the
    # 1 MiB the library holds, so the call must refuse rather than overrun.
    w = wl.normal_weights(100_000, 64, 0.02, seed=1)
    c = g.Compressed(w)
    assert uw.workspace_size(c.desc, 8) > (1 << 20)
    xd = g.dev_bits(wl.activations(8, 64, seed=1))
    yd = g.empty_bits(8, 100_000)
    assert _call(uw, c.desc, c.blob_dev, xd, yd) == 7      # UW_ERR_UNSUPPORTED
