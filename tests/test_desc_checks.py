"""Every entry point that reads a blob checks the descriptor it is given
before any device work (uw_matmul_noalloc included): one filled by
uw_blob_info passes, one with
inconsistent sizes, sections or code lengths is refused with
UW_ERR_INVALID_ARG.  The calls get a zero-byte workspace, so a descriptor
that passes stops at UW_ERR_BUFFER_TOO_SMALL; no pointer is dereferenced
and nothing reaches the GPU."""
import ctypes

import numpy as np
import pytest

import workloads as wl

INVALID, TOO_SMALL = 1, 3
P = ctypes.c_void_p(4096)  # 16-byte aligned, never dereferenced


def _entry_points(L, uw, d):
    b = (ctypes.c_int64 * 1)(1)
    plans = (uw.Plan * 1)()
    r = ctypes.byref(d)
    return {
        "uw_decompress": lambda: L.uw_decompress(r, P, P, P, 0, None),
        "uw_matmul": lambda: L.uw_matmul(r, P, P, 1, P, None, P, 0, None),
        "uw_transcode_palette4": lambda: L.uw_transcode_palette4(r, P, P, P, 0, None),
        "uw_decode_exponents": lambda: L.uw_decode_exponents(r, P, P, P, 0, None),
        "uw_matmul_palette4": lambda: L.uw_matmul_palette4(r, P, P, P, 1, P, -1, P, 0, None),
        "uw_matmul_exponents": lambda: L.uw_matmul_exponents(r, P, P, P, 1, P, -1, P, 0, None),
        "uw_autotune": lambda: L.uw_autotune(r, P, b, 1, plans, P, 0, None),
    }


def _descs(uw):
    mats = [wl.normal_weights(96, 256, 0.02, seed=1), wl.heavy_tailed_weights(64, 512, seed=2),
            wl.all_bf16_patterns(), np.zeros((33, 128), np.uint16), wl.normal_weights(40, 100, 0.02, seed=3)]
    return [uw.blob_info(uw.compress(w)) for w in mats]


def test_descriptors_from_blob_info_pass(uw):
    L = uw.load()
    for d in _descs(uw):
        for name, call in _entry_points(L, uw, d).items():
            assert call() == TOO_SMALL, name


def _copy(d):
    c = type(d)()
    ctypes.memmove(ctypes.byref(c), ctypes.byref(d), ctypes.sizeof(d))
    return c


MUTATIONS = {
    "no rows": lambda d: setattr(d, "rows", 0),
    "cols beyond the group count": lambda d: setattr(d, "cols", d.cols + 32),
    "no cols": lambda d: setattr(d, "cols", 0),
    "rows beyond 2^31": lambda d: setattr(d, "rows", d.rows << 32),
    "tile count": lambda d: setattr(d, "n_tiles", d.n_tiles + 1),
    "group count": lambda d: setattr(d, "n_groups", d.n_groups - 1),
    "more escapes than groups": lambda d: setattr(d, "n_escaped", d.n_groups + 1),
    "escapes past the blob": lambda d: setattr(d, "blob_bytes", d.off_esc + 64 * d.n_escaped - 256),
    "section misaligned": lambda d: setattr(d, "off_tcode", d.off_tcode + 16),
    "sections out of order": lambda d: setattr(d, "off_code", d.off_tesc),
    "offset past the blob": lambda d: setattr(d, "off_esc", d.blob_bytes + 256),
    "huge blob size": lambda d: setattr(d, "blob_bytes", 1 << 62),
    "code longer than 5 bits": lambda d: d.code_len.__setitem__(0, 6),
    "code beyond the palette": lambda d: d.code_len.__setitem__(d.n_palette, 1) if d.n_palette < 16
    else setattr(d, "n_palette", 17),
    "Kraft sum above one": lambda d: [d.code_len.__setitem__(i, 1) for i in range(min(3, d.n_palette))]
    if d.n_palette >= 3 else setattr(d, "lmax", 4),
    "palette repeats an exponent": lambda d: d.palette.__setitem__(1, d.palette[0]) if d.n_palette >= 2
    else setattr(d, "n_palette", -1),
    "wrong length limit": lambda d: setattr(d, "lmax", 4),
    "palette too large": lambda d: setattr(d, "n_palette", 17),
}


@pytest.mark.parametrize("what", sorted(MUTATIONS))
def test_inconsistent_descriptors_are_refused(uw, what):
    L = uw.load()
    d0 = uw.blob_info(uw.compress(wl.heavy_tailed_weights(64, 512, seed=2)))
    assert d0.n_escaped > 0 and d0.n_palette == 16
    d = _copy(d0)
    MUTATIONS[what](d)
    for name, call in _entry_points(L, uw, d).items():
        assert call() == INVALID, (what, name)
    # the entry point without a workspace refuses it before it sizes or
    # clears any scratch (nothing is queued on a stream)
    assert L.uw_matmul_noalloc(ctypes.byref(d), P, P, ctypes.c_int64(1), P, None) == INVALID, what


def test_noalloc_refuses_unaligned_x_before_device_work(uw):
    L = uw.load()
    d = uw.blob_info(uw.compress(wl.normal_weights(96, 256, 0.02, seed=1)))
    assert L.uw_matmul_noalloc(ctypes.byref(d), P, ctypes.c_void_p(4096 + 8), ctypes.c_int64(1), P,
                               None) == INVALID


def test_uncompressed_twin_has_the_same_size_limit(uw):
    L = uw.load()
    assert L.uw_matmul_bf16(P, (1 << 31) + 32, 64, P, 1, P, -1, P, 0, None) == 7  # UW_ERR_UNSUPPORTED
    assert L.uw_matmul_bf16(P, 32, (1 << 31) + 64, P, 1, P, -1, P, 0, None) == 7
    assert L.uw_matmul_bf16(P, 32, 0, P, 1, P, -1, P, 0, None) == 2               # UW_ERR_SHAPE
    assert L.uw_matmul_bf16(P, 0, 64, P, 1, P, -1, P, 0, None) == 2
    assert L.uw_matmul_bf16(P, 32, 96, P, 1, P, -1, P, 0, None) == TOO_SMALL      # ragged rows are fine
    assert L.uw_matmul_bf16(P, 32, 128, P, 1, P, -1, P, 0, None) == TOO_SMALL


def test_ragged_workspaces_hold_the_zero_extended_rows(uw):
    # a ragged matmul needs room for x (and, uncompressed, W) at the stored width
    for rows, cols, batch in [(96, 100, 1), (64, 4097, 4), (33, 14335, 16)]:
        cp = -(-cols // 64) * 64
        whole = uw.workspace_size_bf16(rows, cp, batch)
        assert uw.workspace_size_bf16(rows, cols, batch) >= whole + 2 * batch * cp + 2 * rows * cp
        d = uw.blob_info(uw.compress(wl.normal_weights(rows, cols, 0.02, seed=rows)))
        assert d.cols == cols and d.n_groups == rows * cp // 64
        dw = uw.blob_info(uw.compress(wl.normal_weights(rows, cp, 0.02, seed=rows)))
        assert uw.workspace_size(d, batch) >= uw.workspace_size(dw, batch) + 2 * batch * cp
        assert uw.exponent_bytes(d) == rows * cp and uw.palette4_bytes(d) == rows * cp // 2
