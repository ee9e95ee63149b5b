"""The Python binding refuses buffers that are smaller than what a call reads
or writes, or not contiguous, before anything reaches the C ABI (which sees
plain pointers).  Checked on the CPU against a stand-in for the library that
records which entry points were reached."""
import pytest
import torch

import workloads as wl


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append(name)
            return 0
        return fn


@pytest.fixture
def fake(uw, monkeypatch):
    rec = _Recorder()
    monkeypatch.setattr(uw, "_lib", rec)
    return rec


@pytest.fixture(scope="module")
def mat(uw):
    w = wl.normal_weights(96, 256, 0.02, seed=2)
    blob = uw.compress(w)
    return uw.blob_info(blob), torch.from_numpy(blob)


def _bits(*shape):
    return torch.zeros(*shape, dtype=torch.int16)


def _refused(uw, fn, *args, **kw):
    with pytest.raises(uw.UwError) as e:
        fn(*args, **kw)
    assert e.value.status == uw.UW_ERR_BUFFER_TOO_SMALL


def test_matmul_passes_right_sized_buffers(uw, fake, mat):
    d, blob = mat
    ws = torch.zeros(4096, dtype=torch.uint8)
    uw.matmul(d, blob, _bits(4, 256), _bits(4, 96), ws, stream=0)
    uw.matmul(d, blob, _bits(256), _bits(96), ws, stream=0)  # batch 1 as vectors
    assert uw.matmul_status(d, blob, _bits(4, 256), _bits(4, 96), ws, stream=0) == 0
    assert uw.matmul_noalloc(d, blob, _bits(2, 256), _bits(2, 96), stream=0) == 0
    assert fake.calls == ["uw_matmul", "uw_matmul", "uw_matmul", "uw_matmul_noalloc"]


def test_matmul_refuses_short_or_strided_buffers(uw, fake, mat):
    d, blob = mat
    ws = torch.zeros(4096, dtype=torch.uint8)
    _refused(uw, uw.matmul, d, blob, _bits(4, 256), _bits(3, 96), ws, stream=0)       # y for 3 rows
    _refused(uw, uw.matmul, d, blob, _bits(4, 128), _bits(4, 96), ws, stream=0)       # x too narrow
    _refused(uw, uw.matmul, d, blob[:-16], _bits(1, 256), _bits(1, 96), ws, stream=0)  # cut blob
    _refused(uw, uw.matmul, d, blob, _bits(256, 4).t(), _bits(4, 96), ws, stream=0)   # x transposed view
    assert uw.matmul_status(d, blob, _bits(4, 256), _bits(96), ws, stream=0) == uw.UW_ERR_BUFFER_TOO_SMALL
    assert uw.matmul_noalloc(d, blob, _bits(4, 256), _bits(96), stream=0) == uw.UW_ERR_BUFFER_TOO_SMALL
    assert fake.calls == []


def test_decode_entry_points_check_their_outputs(uw, fake, mat):
    d, blob = mat
    ws = torch.zeros(4096, dtype=torch.uint8)
    n = d.rows * d.cols
    uw.decompress(d, blob, _bits(d.rows, d.cols), ws, stream=0)
    uw.transcode_palette4(d, blob, torch.zeros(n // 2, dtype=torch.uint8), ws, stream=0)
    uw.decode_exponents(d, blob, torch.zeros(n, dtype=torch.uint8), ws, stream=0)
    assert fake.calls == ["uw_decompress", "uw_transcode_palette4", "uw_decode_exponents"]
    _refused(uw, uw.decompress, d, blob, _bits(d.rows - 1, d.cols), ws, stream=0)
    _refused(uw, uw.transcode_palette4, d, blob, torch.zeros(n // 2 - 1, dtype=torch.uint8), ws, stream=0)
    _refused(uw, uw.decode_exponents, d, blob, torch.zeros(n // 2, dtype=torch.uint8), ws, stream=0)
    assert len(fake.calls) == 3


def test_form_matmuls_check_the_form(uw, fake, mat):
    d, blob = mat
    ws = torch.zeros(4096, dtype=torch.uint8)
    n = d.rows * d.cols
    x, y = _bits(16, 256), _bits(16, 96)
    p4, e = torch.zeros(n // 2, dtype=torch.uint8), torch.zeros(n, dtype=torch.uint8)
    assert uw.matmul_palette4_status(d, blob, p4, x, y, ws, stream=0) == 0
    assert uw.matmul_exponents_status(d, blob, e, x, y, ws, stream=0) == 0
    assert uw.matmul_palette4_status(d, blob, p4[:-1], x, y, ws, stream=0) == uw.UW_ERR_BUFFER_TOO_SMALL
    assert uw.matmul_exponents_status(d, blob, p4, x, y, ws, stream=0) == uw.UW_ERR_BUFFER_TOO_SMALL
    assert fake.calls == ["uw_matmul_palette4", "uw_matmul_exponents"]


def test_twin_and_swiglu_check_their_buffers(uw, fake):
    ws = torch.zeros(4096, dtype=torch.uint8)
    uw.matmul_bf16(_bits(96, 256), _bits(2, 256), _bits(2, 96), ws, stream=0)
    uw.swiglu(_bits(2, 64), _bits(2, 64), _bits(2, 64), stream=0)
    assert fake.calls == ["uw_matmul_bf16", "uw_swiglu"]
    _refused(uw, uw.matmul_bf16, _bits(96, 256), _bits(2, 256), _bits(1, 96), ws, stream=0)
    _refused(uw, uw.matmul_bf16, _bits(96, 256)[:, :128], _bits(2, 128), _bits(2, 96), ws, stream=0)
    _refused(uw, uw.swiglu, _bits(2, 64), _bits(2, 63), _bits(2, 64), stream=0)
    _refused(uw, uw.swiglu, _bits(2, 64), _bits(2, 64), _bits(64), stream=0)
    assert len(fake.calls) == 2


def test_chain_checks_activations_and_blobs(uw):
    # one SwiGLU layer, D = 256, F = 128: gate and up 128 x 256, down 256 x 128
    ents = []
    for (rows, cols), seed in zip([(128, 256), (128, 256), (256, 128)], (4, 5, 6)):
        b = uw.compress(wl.normal_weights(rows, cols, 0.02, seed=seed))
        ents.append((uw.blob_info(b), torch.from_numpy(b), None, None))
    d, blob = ents[0][0], ents[0][1]
    mats = uw.mlp_matrices(ents)
    with pytest.raises(uw.UwError):
        uw.mlp_matrices([(d, blob[:100], None, None)] + ents[1:])
    rec = _Recorder()
    real = uw._lib
    try:
        uw._lib = rec
        ws = torch.zeros(4096, dtype=torch.uint8)
        assert uw.mlp_forward_status(mats, _bits(2, 256), _bits(2, 256), ws, stream=0) == 0
        assert uw.mlp_forward_status(mats, _bits(2, 256), _bits(1, 256), ws, stream=0) == \
            uw.UW_ERR_BUFFER_TOO_SMALL
        assert uw.mlp_forward_status(mats, _bits(2, 255), _bits(2, 256), ws, stream=0) == \
            uw.UW_ERR_BUFFER_TOO_SMALL
        with pytest.raises(uw.UwError):
            uw.mlp_autotune(mats, _bits(2, 256), _bits(1, 256), ws, stream=0)
        assert rec.calls == ["uw_mlp_forward"]
    finally:
        uw._lib = real


@pytest.fixture(scope="module")
def ragged(uw):
    blob = uw.compress(wl.normal_weights(40, 100, 0.02, seed=4))
    return uw.blob_info(blob), torch.from_numpy(blob)


def test_ragged_forms_are_sized_for_the_stored_width(uw, ragged, fake):
    # 100 columns are stored as 128: the forms hold rows * 128 weights
    d, blob = ragged
    assert (d.rows, d.cols) == (40, 100)
    ws = torch.zeros(4096, dtype=torch.uint8)
    n = 40 * 128
    uw.transcode_palette4(d, blob, torch.zeros(n // 2, dtype=torch.uint8), ws, stream=0)
    uw.decode_exponents(d, blob, torch.zeros(n, dtype=torch.uint8), ws, stream=0)
    _refused(uw, uw.transcode_palette4, d, blob, torch.zeros(40 * 100 // 2, dtype=torch.uint8), ws, stream=0)
    _refused(uw, uw.decode_exponents, d, blob, torch.zeros(40 * 100, dtype=torch.uint8), ws, stream=0)
    x, y = _bits(2, 100), _bits(2, 40)
    assert uw.matmul_palette4_status(d, blob, torch.zeros(n // 2, dtype=torch.uint8), x, y, ws, stream=0) == 0
    assert uw.matmul_exponents_status(d, blob, torch.zeros(40 * 100, dtype=torch.uint8), x, y, ws,
                                      stream=0) == uw.UW_ERR_BUFFER_TOO_SMALL
    uw.decompress(d, blob, _bits(40, 100), ws, stream=0)   # the true columns only
    assert fake.calls == ["uw_transcode_palette4", "uw_decode_exponents", "uw_matmul_palette4", "uw_decompress"]
