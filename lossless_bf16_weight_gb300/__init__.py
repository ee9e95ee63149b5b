"""Python binding of the lossless BF16 weight compression library (libuw.so).

Every function here only marshals arguments into the C ABI declared in
include/uw.h and has the same name without the ``uw_`` prefix.  All compute
runs in the library's CUDA kernels (and its host compressor); PyTorch
tensors merely provide device memory and the current CUDA stream.  There is
no fallback: if libuw.so is missing, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libuw.so")

UW_OK = 0
UW_ERR_BUFFER_TOO_SMALL = 3
STATUS_NAMES = {0: "UW_OK", 1: "UW_ERR_INVALID_ARG", 2: "UW_ERR_SHAPE", 3: "UW_ERR_BUFFER_TOO_SMALL",
                4: "UW_ERR_CORRUPT", 5: "UW_ERR_CUDA", 6: "UW_ERR_TIMEOUT", 7: "UW_ERR_UNSUPPORTED",
                8: "UW_ERR_INTERNAL"}
STRATEGY_DEFAULT, STRATEGY_DECOMPRESS_GEMM, STRATEGY_FUSED, STRATEGY_PALETTE4, STRATEGY_EXPONENT = -1, 0, 1, 2, 3


class UwError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s: %s (%d)" % (what, STATUS_NAMES.get(status, "?"), status))
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
        ("blob_bytes", ctypes.c_uint64), ("code_bits", ctypes.c_uint64),
        ("n_groups", ctypes.c_uint64), ("n_escaped", ctypes.c_uint64), ("n_tiles", ctypes.c_uint64),
        ("n_palette", ctypes.c_int32), ("lmax", ctypes.c_int32),
        ("palette", ctypes.c_uint8 * 16), ("code_len", ctypes.c_uint8 * 16),
        ("off_sm", ctypes.c_uint64), ("off_glen", ctypes.c_uint64), ("off_tcode", ctypes.c_uint64),
        ("off_tesc", ctypes.c_uint64), ("off_code", ctypes.c_uint64), ("off_esc", ctypes.c_uint64),
        ("max_tile_bytes", ctypes.c_uint64),
    ]


class Plan(ctypes.Structure):
    _fields_ = [("strategy", ctypes.c_int32), ("variant", ctypes.c_int32),
                ("batch", ctypes.c_int64), ("us", ctypes.c_float)]

    def __repr__(self):
        return "Plan(strategy=%d, variant=%d, batch=%d, us=%.2f)" % (
            self.strategy, self.variant, self.batch, self.us)


class MlpMatrix(ctypes.Structure):
    """One weight matrix of an MLP chain (uw_mlp_matrix)."""
    _fields_ = [("desc", ctypes.POINTER(Desc)), ("blob_dev", ctypes.c_void_p), ("form_dev", ctypes.c_void_p),
                ("plan", Plan)]


class Schedule(ctypes.Structure):
    """Preprocess slots and SM split of an MLP chain (uw_schedule)."""
    _fields_ = [("slots", ctypes.c_int32), ("dec_ctas", ctypes.c_int32)]

    def __repr__(self):
        return "Schedule(slots=%d, dec_ctas=%d)" % (self.slots, self.dec_ctas)


_lib = None

# (name, restype, argtypes) of every symbol in include/uw.h
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
SIGNATURES = [
    ("uw_compress", ctypes.c_int, [_P, _I64, _I64, _P, ctypes.POINTER(_SZ)]),
    ("uw_blob_info", ctypes.c_int, [_P, _SZ, ctypes.POINTER(Desc)]),
    ("uw_workspace_size", ctypes.c_int, [ctypes.POINTER(Desc), _I64, ctypes.POINTER(Plan), ctypes.POINTER(_SZ)]),
    ("uw_workspace_size_bf16", ctypes.c_int, [_I64, _I64, _I64, _I32, ctypes.POINTER(_SZ)]),
    ("uw_workspace_init", ctypes.c_int, [_P, _SZ, _P]),
    ("uw_decompress", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _P, _SZ, _P]),
    ("uw_matmul", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _I64, _P, ctypes.POINTER(Plan), _P, _SZ, _P]),
    ("uw_matmul_bf16", ctypes.c_int, [_P, _I64, _I64, _P, _I64, _P, _I32, _P, _SZ, _P]),
    ("uw_autotune", ctypes.c_int, [ctypes.POINTER(Desc), _P, ctypes.POINTER(_I64), _I32, ctypes.POINTER(Plan),
                                   _P, _SZ, _P]),
    ("uw_autotune_workspace_size", ctypes.c_int, [ctypes.POINTER(Desc), ctypes.POINTER(_I64), _I32,
                                                  ctypes.POINTER(_SZ)]),
    ("uw_matmul_noalloc", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _I64, _P, _P]),
    ("uw_swiglu", ctypes.c_int, [_P, _P, _P, _I64, _P]),
    ("uw_palette4_bytes", ctypes.c_int, [ctypes.POINTER(Desc), ctypes.POINTER(_SZ)]),
    ("uw_transcode_palette4", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _P, _SZ, _P]),
    ("uw_matmul_palette4", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _P, _I64, _P, _I32, _P, _SZ, _P]),
    ("uw_exponent_bytes", ctypes.c_int, [ctypes.POINTER(Desc), ctypes.POINTER(_SZ)]),
    ("uw_decode_exponents", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _P, _SZ, _P]),
    ("uw_matmul_exponents", ctypes.c_int, [ctypes.POINTER(Desc), _P, _P, _P, _I64, _P, _I32, _P, _SZ, _P]),
    ("uw_mlp_workspace_size", ctypes.c_int, [ctypes.POINTER(MlpMatrix), _I32, _I64, ctypes.POINTER(Schedule),
                                             ctypes.POINTER(_SZ)]),
    ("uw_mlp_forward", ctypes.c_int, [ctypes.POINTER(MlpMatrix), _I32, _P, _I64, _P, ctypes.POINTER(Schedule),
                                      _P, _SZ, _P, _P]),
    ("uw_mlp_autotune", ctypes.c_int, [ctypes.POINTER(MlpMatrix), _I32, _P, _I64, _P, _I32, ctypes.POINTER(Plan),
                                       ctypes.POINTER(Schedule), _P, _SZ, _P, _P]),
    ("uw_mlp_autotune_workspace_size", ctypes.c_int, [ctypes.POINTER(MlpMatrix), _I32, _I64,
                                                      ctypes.POINTER(_SZ)]),
    ("uw_check_status", ctypes.c_int, [_P, _P]),
    ("uw_selftest_bounded_wait", ctypes.c_int, [_P, _SZ, ctypes.c_uint32, _P]),
    ("uw_variant_name", ctypes.c_char_p, [_I32, _I32]),
    ("uw_variant_count", ctypes.c_int32, [_I32]),
    ("uw_status_string", ctypes.c_char_p, [ctypes.c_int]),
]


def build(force: bool = False) -> str:
    from .build import build as _build
    return _build(force=force)


def load():
    """Load libuw.so (built beforehand by build()).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libuw.so is not built (run lossless_bf16_weight_gb300.build())")
        lib = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _check(status: int, what: str):
    if status != UW_OK:
        raise UwError(status, what)


def _ptr(t) -> int:
    """Device or host address of a torch tensor or numpy array."""
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _plan_ptr(plan):
    return None if plan is None else ctypes.byref(plan)


def _nbytes(t) -> int:
    return t.nbytes if isinstance(t, np.ndarray) else t.numel() * t.element_size()


def _contiguous(t) -> bool:
    return t.flags.c_contiguous if isinstance(t, np.ndarray) else t.is_contiguous()


def _short(*bufs) -> str | None:
    """The C ABI sees plain pointers, so a buffer smaller than what a call
    reads or writes would make a kernel run past its end.  Each argument is
    (buffer, bytes the call touches, name); returns why the first one that
    is not contiguous or too small is refused, or None."""
    for t, need, name in bufs:
        if not _contiguous(t):
            return "%s is not contiguous" % name
        if _nbytes(t) < need:
            return "%s holds %d bytes, the call needs %d" % (name, _nbytes(t), need)
    return None


def _refuse(why: str | None, what: str):
    if why is not None:
        raise UwError(UW_ERR_BUFFER_TOO_SMALL, "%s (%s)" % (what, why))


def _batch(x) -> int:
    return x.shape[0] if x.dim() == 2 else 1


def _form_bytes(desc) -> int:
    """Weights of a blob's stored width (rows extended to whole 64-column
    groups): the exponent form's bytes, twice the palette-4 form's."""
    return desc.rows * (-(-desc.cols // 64) * 64)


def _mm_bufs(desc, blob_dev, x, y):
    b = _batch(x)
    return [(blob_dev, desc.blob_bytes, "blob_dev"), (x, 2 * b * desc.cols, "x"), (y, 2 * b * desc.rows, "y")]


# ---------------------------------------------------------------- host side
def compress(w: np.ndarray) -> np.ndarray:
    """uw_compress: BF16 weight matrix (uint16 bits, [rows, cols]) -> blob bytes (uint8)."""
    w = np.ascontiguousarray(w)
    if w.dtype != np.uint16 or w.ndim != 2:
        raise TypeError("w must be a 2-D uint16 array of BF16 bit patterns")
    L = load()
    size = ctypes.c_size_t(0)
    s = L.uw_compress(w.ctypes.data, w.shape[0], w.shape[1], None, ctypes.byref(size))
    if s != 3:  # UW_ERR_BUFFER_TOO_SMALL answers the size query
        _check(s, "uw_compress")
    blob = np.empty(size.value, np.uint8)
    _check(L.uw_compress(w.ctypes.data, w.shape[0], w.shape[1], blob.ctypes.data, ctypes.byref(size)),
           "uw_compress")
    return blob


def blob_info(blob) -> Desc:
    """uw_blob_info on a host copy of the blob (numpy uint8 or bytes)."""
    b = np.frombuffer(blob, np.uint8) if isinstance(blob, (bytes, bytearray)) else np.ascontiguousarray(blob)
    d = Desc()
    _check(load().uw_blob_info(b.ctypes.data, b.size, ctypes.byref(d)), "uw_blob_info")
    return d


def blob_info_status(blob) -> int:
    b = np.frombuffer(blob, np.uint8) if isinstance(blob, (bytes, bytearray)) else np.ascontiguousarray(blob)
    d = Desc()
    return int(load().uw_blob_info(b.ctypes.data, b.size, ctypes.byref(d)))


def workspace_size(desc: Desc, batch: int = 0, plan: Plan | None = None) -> int:
    n = ctypes.c_size_t(0)
    _check(load().uw_workspace_size(ctypes.byref(desc), batch, _plan_ptr(plan), ctypes.byref(n)),
           "uw_workspace_size")
    return n.value


def workspace_size_bf16(rows: int, cols: int, batch: int = 1, variant: int = -1) -> int:
    """Workspace bytes of matmul_bf16 for this shape, batch and variant."""
    n = ctypes.c_size_t(0)
    _check(load().uw_workspace_size_bf16(rows, cols, batch, variant, ctypes.byref(n)), "uw_workspace_size_bf16")
    return n.value


def autotune_workspace_size(desc: Desc, batches) -> int:
    arr = (ctypes.c_int64 * len(batches))(*batches)
    n = ctypes.c_size_t(0)
    _check(load().uw_autotune_workspace_size(ctypes.byref(desc), arr, len(batches), ctypes.byref(n)),
           "uw_autotune_workspace_size")
    return n.value


def variant_count(strategy: int) -> int:
    return int(load().uw_variant_count(strategy))


def variant_name(strategy: int, variant: int) -> str | None:
    r = load().uw_variant_name(strategy, variant)
    return None if r is None else r.decode()


def status_string(status: int) -> str:
    return load().uw_status_string(status).decode()


# ---------------------------------------------------------------- device side
def workspace_init(ws, stream=None):
    _check(load().uw_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "uw_workspace_init")


def decompress(desc: Desc, blob_dev, w_out, ws, stream=None):
    _refuse(_short((blob_dev, desc.blob_bytes, "blob_dev"), (w_out, 2 * desc.rows * desc.cols, "w_out")),
            "uw_decompress")
    _check(load().uw_decompress(ctypes.byref(desc), _ptr(blob_dev), _ptr(w_out), _ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)), "uw_decompress")


def matmul(desc: Desc, blob_dev, x, y, ws, plan: Plan | None = None, stream=None):
    """y[batch, rows] = x[batch, cols] W^T with W compressed in blob_dev."""
    _refuse(_short(*_mm_bufs(desc, blob_dev, x, y)), "uw_matmul")
    batch = _batch(x)
    _check(load().uw_matmul(ctypes.byref(desc), _ptr(blob_dev), _ptr(x), batch, _ptr(y), _plan_ptr(plan),
                            _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "uw_matmul")


def matmul_status(desc: Desc, blob_dev, x, y, ws, plan: Plan | None = None, stream=None) -> int:
    if _short(*_mm_bufs(desc, blob_dev, x, y)):
        return UW_ERR_BUFFER_TOO_SMALL
    batch = _batch(x)
    return int(load().uw_matmul(ctypes.byref(desc), _ptr(blob_dev), _ptr(x), batch, _ptr(y), _plan_ptr(plan),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def matmul_noalloc(desc: Desc, blob_dev, x, y, stream=None) -> int:
    """uw_matmul_noalloc: fused matmul with library-held scratch; returns the status."""
    if _short(*_mm_bufs(desc, blob_dev, x, y)):
        return UW_ERR_BUFFER_TOO_SMALL
    batch = _batch(x)
    return int(load().uw_matmul_noalloc(ctypes.byref(desc), _ptr(blob_dev), _ptr(x), batch, _ptr(y),
                                        _stream(stream)))


def matmul_bf16(w, x, y, ws, variant: int = -1, stream=None):
    rows, cols = w.shape
    batch = _batch(x)
    _refuse(_short((w, 2 * rows * cols, "w"), (x, 2 * batch * cols, "x"), (y, 2 * batch * rows, "y")),
            "uw_matmul_bf16")
    _check(load().uw_matmul_bf16(_ptr(w), rows, cols, _ptr(x), batch, _ptr(y), variant, _ptr(ws),
                                 ws.numel() * ws.element_size(), _stream(stream)), "uw_matmul_bf16")


def autotune(desc: Desc, blob_dev, batches, ws, stream=None) -> list[Plan]:
    arr = (ctypes.c_int64 * len(batches))(*batches)
    plans = (Plan * len(batches))()
    _check(load().uw_autotune(ctypes.byref(desc), _ptr(blob_dev), arr, len(batches), plans, _ptr(ws),
                              ws.numel() * ws.element_size(), _stream(stream)), "uw_autotune")
    return list(plans)


def palette4_bytes(desc: Desc) -> int:
    n = _SZ(0)
    _check(load().uw_palette4_bytes(ctypes.byref(desc), ctypes.byref(n)), "uw_palette4_bytes")
    return int(n.value)


def transcode_palette4(desc: Desc, blob_dev, p4_out, ws, stream=None):
    """uw_transcode_palette4: the 4-bit palette index of every weight into p4_out."""
    _refuse(_short((blob_dev, desc.blob_bytes, "blob_dev"), (p4_out, _form_bytes(desc) // 2, "p4_out")),
            "uw_transcode_palette4")
    _check(load().uw_transcode_palette4(ctypes.byref(desc), _ptr(blob_dev), _ptr(p4_out), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)), "uw_transcode_palette4")


def matmul_palette4_status(desc: Desc, blob_dev, p4, x, y, ws, variant: int = -1, stream=None) -> int:
    if _short(*_mm_bufs(desc, blob_dev, x, y), (p4, _form_bytes(desc) // 2, "p4")):
        return UW_ERR_BUFFER_TOO_SMALL
    batch = _batch(x)
    return int(load().uw_matmul_palette4(ctypes.byref(desc), _ptr(blob_dev), _ptr(p4), _ptr(x), batch, _ptr(y),
                                         variant, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def matmul_palette4(desc: Desc, blob_dev, p4, x, y, ws, variant: int = -1, stream=None):
    """y[batch, rows] = x W^T from the palette-4 form p4 (plus the blob)."""
    _check(matmul_palette4_status(desc, blob_dev, p4, x, y, ws, variant, stream), "uw_matmul_palette4")


def exponent_bytes(desc: Desc) -> int:
    n = _SZ(0)
    _check(load().uw_exponent_bytes(ctypes.byref(desc), ctypes.byref(n)), "uw_exponent_bytes")
    return int(n.value)


def decode_exponents(desc: Desc, blob_dev, e_out, ws, stream=None):
    """uw_decode_exponents: the exponent byte of every weight into e_out."""
    _refuse(_short((blob_dev, desc.blob_bytes, "blob_dev"), (e_out, _form_bytes(desc), "e_out")),
            "uw_decode_exponents")
    _check(load().uw_decode_exponents(ctypes.byref(desc), _ptr(blob_dev), _ptr(e_out), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)), "uw_decode_exponents")


def matmul_exponents_status(desc: Desc, blob_dev, e, x, y, ws, variant: int = -1, stream=None) -> int:
    if _short(*_mm_bufs(desc, blob_dev, x, y), (e, _form_bytes(desc), "e")):
        return UW_ERR_BUFFER_TOO_SMALL
    batch = _batch(x)
    return int(load().uw_matmul_exponents(ctypes.byref(desc), _ptr(blob_dev), _ptr(e), _ptr(x), batch, _ptr(y),
                                          variant, _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def matmul_exponents(desc: Desc, blob_dev, e, x, y, ws, variant: int = -1, stream=None):
    """y[batch, rows] = x W^T from the exponent form e (plus the blob)."""
    _check(matmul_exponents_status(desc, blob_dev, e, x, y, ws, variant, stream), "uw_matmul_exponents")


def swiglu(g, u, h, stream=None):
    n = g.numel()
    _refuse(_short((g, 2 * n, "g"), (u, 2 * n, "u"), (h, 2 * n, "h")), "uw_swiglu")
    _check(load().uw_swiglu(_ptr(g), _ptr(u), _ptr(h), g.numel(), _stream(stream)), "uw_swiglu")


# ---------------------------------------------------------------- MLP chain
def mlp_matrices(entries) -> ctypes.Array:
    """uw_mlp_matrix array from (desc, blob_dev, form_dev or None, plan or None)
    entries, three per layer (gate, up, down).  Keep `entries` alive while
    the array is used."""
    arr = (MlpMatrix * len(entries))()
    for i, (d, blob, form, plan) in enumerate(entries):
        _refuse(_short((blob, d.blob_bytes, "blob_dev")), "uw_mlp_matrix %d" % i)
        arr[i].desc = ctypes.pointer(d)
        arr[i].blob_dev = _ptr(blob)
        arr[i].form_dev = None if form is None else _ptr(form)
        arr[i].plan = plan if plan is not None else Plan(STRATEGY_DEFAULT, -1, 0, 0.0)
    return arr


def _side(stream):
    if stream is None:
        return None
    return ctypes.c_void_p(stream if isinstance(stream, int) else stream.cuda_stream)


def _sched_ptr(sched):
    return None if sched is None else ctypes.byref(sched)


def mlp_workspace_size(mats, batch: int, sched: Schedule | None = None) -> int:
    n = _SZ(0)
    _check(load().uw_mlp_workspace_size(mats, len(mats) // 3, batch, _sched_ptr(sched), ctypes.byref(n)),
           "uw_mlp_workspace_size")
    return int(n.value)


def _chain_short(mats, x, y) -> str | None:
    if len(mats) < 3:
        return None  # the library refuses an empty chain itself
    dim_in, dim_out = mats[0].desc.contents.cols, mats[len(mats) // 3 * 3 - 1].desc.contents.rows
    return _short((x, 2 * x.shape[0] * dim_in, "x"), (y, 2 * x.shape[0] * dim_out, "y"))


def mlp_forward_status(mats, x, y, ws, sched: Schedule | None = None, stream=None, side_stream=None) -> int:
    """uw_mlp_forward: y = the chain of len(mats)//3 SwiGLU MLP layers applied to x."""
    if _chain_short(mats, x, y):
        return UW_ERR_BUFFER_TOO_SMALL
    return int(load().uw_mlp_forward(mats, len(mats) // 3, _ptr(x), x.shape[0], _ptr(y), _sched_ptr(sched),
                                     _ptr(ws), ws.numel() * ws.element_size(), _stream(stream),
                                     _side(side_stream)))


def mlp_forward(mats, x, y, ws, sched: Schedule | None = None, stream=None, side_stream=None):
    _check(mlp_forward_status(mats, x, y, ws, sched, stream, side_stream), "uw_mlp_forward")


def mlp_autotune_workspace_size(mats, batch: int) -> int:
    n = _SZ(0)
    _check(load().uw_mlp_autotune_workspace_size(mats, len(mats) // 3, batch, ctypes.byref(n)),
           "uw_mlp_autotune_workspace_size")
    return int(n.value)


def mlp_autotune(mats, x, y, ws, passes: int = 2, stream=None, side_stream=None):
    """uw_mlp_autotune: (6 plans: gate, up, down without a form, then with
    one; Schedule) by coordinate descent."""
    _refuse(_chain_short(mats, x, y), "uw_mlp_autotune")
    plans = (Plan * 6)()
    sched = Schedule()
    _check(load().uw_mlp_autotune(mats, len(mats) // 3, _ptr(x), x.shape[0], _ptr(y), passes, plans,
                                  ctypes.byref(sched), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream),
                                  _side(side_stream)), "uw_mlp_autotune")
    return list(plans), sched


def selftest_bounded_wait(ws, tries: int, stream=None) -> None:
    """uw_selftest_bounded_wait: a kernel whose bounded wait runs out; read
    the result with check_status."""
    _check(load().uw_selftest_bounded_wait(_ptr(ws), ws.numel() * ws.element_size(), int(tries), _stream(stream)),
           "uw_selftest_bounded_wait")


def check_status(ws, stream=None) -> int:
    """uw_check_status: synchronises and returns the device error status (0 = ok)."""
    return int(load().uw_check_status(_ptr(ws), _stream(stream)))
