"""CPU oracle for Unweight-style lossless BF16 weight compression.

TEST INFRASTRUCTURE ONLY.  The oracle checks the CUDA library; only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  It shares no code with the library (the library never imports
it, and it never imports the library).

The arithmetic lives in ``uw_oracle.c`` (plain single-threaded C); this
module only marshals numpy arrays through ctypes.  Every function names the
paragraph of the Unweight blog post it follows; see the C file's header for
the paragraph tags and the readings taken where the page is silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "uw_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

GROUP = 64
TILE_ROWS = 32
LMAX = 5
PALETTE = 16


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (plain -O2, no vector or
    architecture flags, so x86 and Arm hosts give the same results)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class Info(ctypes.Structure):
    _fields_ = [
        ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
        ("n_groups", ctypes.c_int64), ("n_escaped", ctypes.c_int64), ("n_tiles", ctypes.c_int64),
        ("code_bits", ctypes.c_int64), ("blob_bytes", ctypes.c_int64),
        ("n_palette", ctypes.c_int32), ("lmax", ctypes.c_int32),
        ("palette", ctypes.c_uint8 * 16), ("code_len", ctypes.c_uint8 * 16),
        ("off_sm", ctypes.c_uint64), ("off_glen", ctypes.c_uint64), ("off_tcode", ctypes.c_uint64),
        ("off_tesc", ctypes.c_uint64), ("off_code", ctypes.c_uint64), ("off_esc", ctypes.c_uint64),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["palette"] = list(self.palette)[: self.n_palette]
        d["code_len"] = list(self.code_len)
        return d


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.uwo_split.argtypes = [P, I64, P, P]
        lib.uwo_histogram.argtypes = [P, I64, P]
        lib.uwo_palette.argtypes = [P, P]
        lib.uwo_palette.restype = ctypes.c_int
        lib.uwo_escape_flags.argtypes = [P, I64, I64, P, ctypes.c_int, P]
        lib.uwo_code_lengths.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
        lib.uwo_code_lengths.restype = ctypes.c_int
        lib.uwo_canonical_codes.argtypes = [P, ctypes.c_int, P]
        lib.uwo_compress.argtypes = [P, I64, I64, P, P, I64, ctypes.POINTER(Info)]
        lib.uwo_compress.restype = I64
        lib.uwo_read_header.argtypes = [P, I64, ctypes.POINTER(Info)]
        lib.uwo_read_header.restype = ctypes.c_int
        lib.uwo_decompress.argtypes = [P, I64, P]
        lib.uwo_decompress.restype = ctypes.c_int
        lib.uwo_matmul_f64.argtypes = [P, I64, P, I64, I64, I64, I64, P, P]
        lib.uwo_swiglu_f64.argtypes = [P, P, I64, P]
        lib.uwo_palette4.argtypes = [P, I64, I64, P, ctypes.c_int, P]
        lib.uwo_exponents.argtypes = [P, I64, I64, P]
        lib.uwo_stored_cols.argtypes = [I64]
        lib.uwo_stored_cols.restype = I64
        lib.uwo_filler.argtypes = [P, ctypes.c_int]
        lib.uwo_filler.restype = ctypes.c_uint16
        lib.uwo_pad.argtypes = [P, I64, I64, P, ctypes.c_int, P]
        lib.uwo_join.argtypes = [ctypes.c_uint, ctypes.c_uint]
        lib.uwo_join.restype = ctypes.c_uint16
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns")
    return a


def split(w) -> tuple[np.ndarray, np.ndarray]:
    """[BF16] exponent bytes and raw sign+mantissa bytes of every weight."""
    w = _u16(w).ravel()
    e = np.empty(w.size, np.uint8)
    sm = np.empty(w.size, np.uint8)
    _L().uwo_split(_p(w), w.size, _p(e), _p(sm))
    return e, sm


def join(e: int, sm: int) -> int:
    """Inverse of the field split for one weight."""
    return int(_L().uwo_join(int(e), int(sm)))


def histogram(w) -> np.ndarray:
    """[SKEW] count of each of the 256 exponent values."""
    w = _u16(w).ravel()
    c = np.zeros(256, np.uint64)
    _L().uwo_histogram(_p(w), w.size, _p(c))
    return c


def palette(count) -> list[int]:
    """[SKEW]/[ROWS64] up to 16 most frequent exponents, ties to the smaller."""
    c = np.ascontiguousarray(count, dtype=np.uint64)
    out = np.zeros(16, np.uint8)
    n = _L().uwo_palette(_p(c), _p(out))
    return [int(v) for v in out[:n]]


def escape_flags(w, pal) -> np.ndarray:
    """[ROWS64] per group (row-major over (row, k/64)): 1 if escaped."""
    w = _u16(w)
    rows, cols = w.shape
    p = np.zeros(16, np.uint8)
    p[: len(pal)] = pal
    f = np.zeros(rows * (cols // GROUP), np.uint8)
    _L().uwo_escape_flags(_p(w), rows, cols, _p(p), len(pal), _p(f))
    return f


def code_lengths(freq, lmax: int = LMAX) -> list[int]:
    """[HUFFMAN] minimum-redundancy code lengths under a length limit."""
    f = np.ascontiguousarray(freq, dtype=np.uint64)
    out = np.zeros(f.size, np.uint8)
    r = _L().uwo_code_lengths(_p(f), f.size, lmax, _p(out))
    if r < 0:
        raise ValueError("no prefix code with these lengths")
    return [int(v) for v in out]


def canonical_codes(lengths) -> list[int]:
    """Canonical code values ordered by (length, symbol index)."""
    ln = np.ascontiguousarray(lengths, dtype=np.uint8)
    out = np.zeros(ln.size, np.uint16)
    _L().uwo_canonical_codes(_p(ln), ln.size, _p(out))
    return [int(v) for v in out]


def compress(w, len_override=None) -> tuple[bytes, dict]:
    """Whole encoder: W [rows, cols] bf16 bits -> (blob, header fields)."""
    w = _u16(w)
    rows, cols = w.shape
    info = Info()
    ov = None
    if len_override is not None:
        ov = np.zeros(16, np.uint8)
        ov[: len(len_override)] = len_override
    size = _L().uwo_compress(_p(w), rows, cols, None if ov is None else _p(ov), None, 0, ctypes.byref(info))
    if size < 0:
        raise ValueError("oracle compress failed (%d)" % size)
    blob = np.zeros(size, np.uint8)
    size2 = _L().uwo_compress(_p(w), rows, cols, None if ov is None else _p(ov), _p(blob), size, ctypes.byref(info))
    assert size2 == size
    return blob.tobytes(), info.as_dict()


def read_header(blob: bytes) -> dict:
    b = np.frombuffer(blob, np.uint8)
    info = Info()
    if _L().uwo_read_header(_p(b), b.size, ctypes.byref(info)) != 0:
        raise ValueError("not a valid blob header")
    return info.as_dict()


def decompress(blob: bytes) -> np.ndarray:
    """Whole decoder: blob -> W [rows, cols] bf16 bits (bit-by-bit decode)."""
    b = np.frombuffer(blob, np.uint8)
    info = read_header(blob)
    w = np.zeros((info["rows"], info["cols"]), np.uint16)
    r = _L().uwo_decompress(_p(b), b.size, _p(w))
    if r != 0:
        raise ValueError("oracle decompress failed (%d)" % r)
    return w


def decompress_status(blob: bytes) -> int:
    """Like decompress() but returns the oracle's status code (0 = ok)."""
    b = np.frombuffer(blob, np.uint8)
    info = Info()
    if _L().uwo_read_header(_p(b), b.size, ctypes.byref(info)) != 0:
        return -1
    w = np.zeros(max(info.rows * info.cols, 1), np.uint16)
    return int(_L().uwo_decompress(_p(b), b.size, _p(w)))


def matmul_f64(x, w, n0: int = 0, nr: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """[MATMUL] y = x W^T in fp64 over rows n0..n0+nr-1 of W, and the
    per-element magnitude sum sum_k |x_k w_k|."""
    x = _u16(x)
    w = _u16(w)
    if x.ndim == 1:
        x = x[None, :]
    B, K = x.shape
    N, K2 = w.shape
    assert K == K2
    if nr is None:
        nr = N - n0
    y = np.zeros((B, nr), np.float64)
    a = np.zeros((B, nr), np.float64)
    _L().uwo_matmul_f64(_p(x), B, _p(w), N, K, n0, nr, _p(y), _p(a))
    return y, a


def swiglu_f64(g, u) -> np.ndarray:
    """SwiGLU glue: silu(g) * u in fp64 from bf16 inputs."""
    g = _u16(g).ravel()
    u = _u16(u).ravel()
    h = np.zeros(g.size, np.float64)
    _L().uwo_swiglu_f64(_p(g), _p(u), g.size, _p(h))
    return h


def stored_cols(cols: int) -> int:
    """Columns the blob stores for a row of `cols` weights: the next multiple
    of 64 (a ragged row is extended with filler weights)."""
    return int(_L().uwo_stored_cols(int(cols)))


def filler(pal) -> int:
    """The filler weight (bf16 bits) of a matrix with this palette."""
    p = np.zeros(16, np.uint8)
    p[: len(pal)] = pal
    return int(_L().uwo_filler(_p(p), len(pal)))


def pad(w, pal) -> np.ndarray:
    """W [rows, cols] extended to [rows, stored_cols(cols)] with the filler."""
    w = _u16(w)
    rows, cols = w.shape
    p = np.zeros(16, np.uint8)
    p[: len(pal)] = pal
    out = np.zeros((rows, stored_cols(cols)), np.uint16)
    _L().uwo_pad(_p(w), rows, cols, _p(p), len(pal), _p(out))
    return out


def palette4(w, pal) -> np.ndarray:
    """[PALETTE] the 4-bit palette index of every weight in the library's
    palette-4 layout (rows*cols/2 bytes); escaped groups hold index 0."""
    w = _u16(w)
    rows, cols = w.shape
    p = np.zeros(16, np.uint8)
    p[: len(pal)] = pal
    out = np.zeros(rows * cols // 2, np.uint8)
    _L().uwo_palette4(_p(w), rows, cols, _p(p), len(pal), _p(out))
    return out


def exponents(w) -> np.ndarray:
    """[EXPONENT] the exponent byte of every weight in the library's exponent
    form (laid out like the sign+mantissa section; rows*cols bytes)."""
    w = _u16(w)
    rows, cols = w.shape
    out = np.zeros(rows * cols, np.uint8)
    _L().uwo_exponents(_p(w), rows, cols, _p(out))
    return out

