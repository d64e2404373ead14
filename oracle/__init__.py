"""Python handle on the plain-C oracle (``uw_oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the bench's
CPU-baseline leg may import this package.  The product library never links,
imports or calls it.

Every function follows the Cloudflare blog post "Unweight" (see the header of
``uw_oracle.c`` for the passages and for the readings taken where the post is
silent).  All pins are in ``tests/test_oracle_*.py``; no oracle function is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import struct
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "uw_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PALETTE, HUFFMAN = 0, 1
SECTIONS = ("sm", "bitmap", "prefix", "verb_exp", "idx", "chunk_off", "bits")
_VP, _U8, _U16, _I64, _U64, _DBL = (ctypes.c_void_p,) * 6


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` in place: plain C99, -O2, no FP contraction, no threads."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            c = ctypes
            L.or_sm_byte.argtypes = [c.c_uint16]; L.or_sm_byte.restype = c.c_uint8
            L.or_exp_byte.argtypes = [c.c_uint16]; L.or_exp_byte.restype = c.c_uint8
            L.or_rebuild.argtypes = [c.c_uint8, c.c_uint8]; L.or_rebuild.restype = c.c_uint16
            L.or_palette.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p]; L.or_palette.restype = c.c_int
            L.or_huffman_lengths.argtypes = [c.c_void_p, c.c_int, c.c_int, c.c_void_p]
            L.or_huffman_lengths.restype = c.c_int
            L.or_canonical_codes.argtypes = [c.c_void_p, c.c_int, c.c_void_p]; L.or_canonical_codes.restype = None
            L.or_encode.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_int, c.c_uint32, c.c_uint32,
                                    c.c_void_p, c.c_uint64, c.POINTER(c.c_uint64)]
            L.or_encode.restype = c.c_int
            L.or_decode.argtypes = [c.c_void_p, c.c_uint64, c.c_void_p]; L.or_decode.restype = c.c_int
            L.or_matmul_rows.argtypes = [c.c_void_p, c.c_int64, c.c_int64, c.c_void_p, c.c_int64,
                                         c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p]
            L.or_matmul_rows.restype = None
            L.or_split_many.argtypes = [c.c_void_p, c.c_int64, c.c_void_p, c.c_void_p]; L.or_split_many.restype = None
            L.or_rebuild_many.argtypes = [c.c_void_p, c.c_void_p, c.c_int64, c.c_void_p]
            L.or_rebuild_many.restype = None
            _lib = L
    return _lib


class OracleError(RuntimeError):
    pass


def split(h: np.ndarray):
    """sm byte (sign<<7 | mantissa) and exponent byte of every BF16 pattern."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    sm = np.empty(h.shape, np.uint8); e = np.empty(h.shape, np.uint8)
    _load().or_split_many(h.ctypes.data, h.size, sm.ctypes.data, e.ctypes.data)
    return sm, e


def rebuild(sm: np.ndarray, e: np.ndarray) -> np.ndarray:
    sm = np.ascontiguousarray(sm, np.uint8); e = np.ascontiguousarray(e, np.uint8)
    h = np.empty(sm.shape, np.uint16)
    _load().or_rebuild_many(sm.ctypes.data, e.ctypes.data, sm.size, h.ctypes.data)
    return h


def palette(w: np.ndarray):
    """(exponent histogram[256], palette list) of a BF16 array."""
    w = np.ascontiguousarray(w, np.uint16)
    counts = np.zeros(256, np.uint64); pal = np.zeros(16, np.uint8)
    n = _load().or_palette(w.ctypes.data, w.size, counts.ctypes.data, pal.ctypes.data)
    return counts, [int(v) for v in pal[:n]]


def huffman_lengths(counts, max_len: int):
    counts = np.ascontiguousarray(counts, np.uint64)
    lens = np.zeros(len(counts), np.uint8)
    rc = _load().or_huffman_lengths(counts.ctypes.data, len(counts), max_len, lens.ctypes.data)
    if rc:
        raise OracleError(f"or_huffman_lengths: {rc}")
    return [int(v) for v in lens]


def canonical_codes(lens):
    lens = np.ascontiguousarray(lens, np.uint8)
    codes = np.zeros(len(lens), np.uint32)
    _load().or_canonical_codes(lens.ctypes.data, len(lens), codes.ctypes.data)
    return [int(v) for v in codes]


def encode(w: np.ndarray, codec: int = PALETTE, chunk: int = 256, max_len: int = 12) -> bytes:
    w = np.ascontiguousarray(w, np.uint16)
    N, K = w.shape
    size = ctypes.c_uint64(0)
    L = _load()
    rc = L.or_encode(w.ctypes.data, N, K, codec, chunk, max_len, None, 0, ctypes.byref(size))
    if rc:
        raise OracleError(f"or_encode: {rc}")
    buf = np.zeros(size.value, np.uint8)
    rc = L.or_encode(w.ctypes.data, N, K, codec, chunk, max_len, buf.ctypes.data, size.value, ctypes.byref(size))
    if rc:
        raise OracleError(f"or_encode: {rc}")
    return buf.tobytes()


def decode(blob: bytes) -> np.ndarray:
    hdr = parse_header(blob)
    w = np.empty((hdr["N"], hdr["K"]), np.uint16)
    buf = np.frombuffer(blob, np.uint8)
    rc = _load().or_decode(buf.ctypes.data, len(blob), w.ctypes.data)
    if rc:
        raise OracleError(f"or_decode: {rc}")
    return w


def matmul(w: np.ndarray, x: np.ndarray, rows=None):
    """fp64 Y[B, n] = sum_k W[n, k] X[b, k] and A[B, n] = sum_k |W[n, k] X[b, k]| (rows subset optional)."""
    w = np.ascontiguousarray(w, np.uint16); x = np.ascontiguousarray(x, np.uint16)
    N, K = w.shape
    B = x.shape[0]
    assert x.shape[1] == K
    if rows is None:
        nr, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, np.int64); nr, rp = len(rows), rows.ctypes.data
    y = np.empty((B, nr), np.float64); a = np.empty((B, nr), np.float64)
    _load().or_matmul_rows(w.ctypes.data, N, K, x.ctypes.data, B, rp, nr, y.ctypes.data, a.ctypes.data)
    return y, a


def parse_header(blob: bytes) -> dict:
    """Field-by-field reading of the 256-byte blob header (format in ``uw_oracle.c``)."""
    if len(blob) < 256 or blob[:4] != b"UWB1":
        raise OracleError("bad magic")
    version, N, K, codec, block, chunk, max_len = struct.unpack_from("<IqqIIII", blob, 4)
    n_pal = blob[40]
    h = dict(version=version, N=N, K=K, codec=codec, block=block, chunk=chunk, max_len=max_len,
             n_pal=n_pal, palette=list(blob[41:57]), code_len=list(blob[57:73]))
    h["n_blocks"], h["n_verbatim"], h["n_chunks"], h["total_bits"], h["blob_bytes"] = \
        struct.unpack_from("<QQQQQ", blob, 80)
    h["sections"] = {}
    for i, name in enumerate(SECTIONS):
        off, nb = struct.unpack_from("<QQ", blob, 128 + 16 * i)
        h["sections"][name] = (off, nb)
    return h


def section(blob: bytes, name: str) -> bytes:
    off, nb = parse_header(blob)["sections"][name]
    return blob[off:off + nb]
