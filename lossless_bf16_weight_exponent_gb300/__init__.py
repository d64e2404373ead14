"""Python binding of ``libuw.so`` - the C ABI declared in ``include/uw.h``.

Argument marshalling only: every step of the codec and the matmul runs in the
library's own host code and CUDA kernels.  PyTorch is used by callers for device
memory and streams; this module accepts torch tensors (or raw integer device
addresses) and passes plain pointers.  There is no CPU fallback: if the library
is missing, importing works but the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libuw.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "uw.h")

# enums (mirrors of include/uw.h)
OK, ERR_INVALID_ARG, ERR_SHAPE, ERR_UNSUPPORTED, ERR_CORRUPT = 0, 1, 2, 3, 4
ERR_NO_MEMORY, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_BUFFER_TOO_SMALL = 5, 6, 7, 8, 9
CODEC_PALETTE, CODEC_HUFFMAN = 0, 1
STRAT_AUTO, STRAT_FULL_DECODE, STRAT_EXP_ONLY, STRAT_PALETTE_TRANSCODE, STRAT_DIRECT_PALETTE = 0, 1, 2, 3, 4
STRAT_HUFFMAN_DIRECT = 5
STRATEGIES = {"full_decode": 1, "exp_only": 2, "palette_transcode": 3, "direct_palette": 4, "huffman_direct": 5}
OUT_F32, OUT_BF16 = 0, 1
KERNEL_AUTO, KERNEL_GEMV, KERNEL_TC = 0, 1, 2
RESIDENT_HUFFMAN, RESIDENT_BOTH, RESIDENT_PALETTE = 0, 1, 2
RESIDENT = {"huffman": RESIDENT_HUFFMAN, "both": RESIDENT_BOTH, "palette": RESIDENT_PALETTE}
SEQ_DIRECT = -1  # uw_sequence_run schedule: no side-stream transcode, every step its own AUTO plan
STEP_CONCURRENT = 1  # uw_step flag: the step may overlap the step before it
SEQ_GROUPS = 65536  # added to a uw_sequence_run schedule: overlap the groups of STEP_CONCURRENT steps


class UwError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status} ({message})")
        self.status = status
        self.message = message


class EncodeOpts(ctypes.Structure):
    _fields_ = [("codec", ctypes.c_uint32), ("chunk_weights", ctypes.c_uint32), ("max_code_len", ctypes.c_uint32)]


class Plan(ctypes.Structure):
    _fields_ = [("strategy", ctypes.c_int32), ("kernel", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("variant", ctypes.c_int32)]

    def as_tuple(self):
        return (self.strategy, self.kernel, self.split_k, self.variant)

    def __repr__(self):
        return f"Plan(strategy={self.strategy}, kernel={self.kernel}, split_k={self.split_k}, variant={self.variant})"


class Step(ctypes.Structure):
    _fields_ = [("m", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("out_dtype", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class Info(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("K", ctypes.c_int64), ("codec", ctypes.c_uint32), ("n_pal", ctypes.c_uint32),
                ("palette", ctypes.c_uint8 * 16), ("code_len", ctypes.c_uint8 * 16),
                ("n_blocks", ctypes.c_uint64), ("n_verbatim", ctypes.c_uint64), ("n_chunks", ctypes.c_uint64),
                ("total_bits", ctypes.c_uint64), ("blob_bytes", ctypes.c_uint64), ("device_bytes", ctypes.c_uint64),
                ("has_palette_form", ctypes.c_int32), ("chunk_weights", ctypes.c_int32),
                ("max_code_len", ctypes.c_int32), ("has_huffman_stream", ctypes.c_int32)]

    def as_dict(self):
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["palette"] = list(self.palette)
        d["code_len"] = list(self.code_len)
        return d


_lib = None
_VP, _SZ, _I64, _INT = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_int

_SIGS = {
    "uw_encode": [_VP, _I64, _I64, ctypes.POINTER(EncodeOpts), _VP, _SZ, ctypes.POINTER(_SZ)],
    "uw_load": [_VP, _SZ, _INT, _VP, ctypes.POINTER(_VP)],
    "uw_blob_validate": [_VP, _SZ, ctypes.POINTER(Info)],
    "uw_free": [_VP],
    "uw_get_info": [_VP, ctypes.POINTER(Info)],
    "uw_decode": [_VP, _VP, _VP],
    "uw_workspace_size": [_VP, _I64, _INT, ctypes.POINTER(_SZ)],
    "uw_matmul": [_VP, _VP, _I64, _VP, _INT, _INT, _VP, _SZ, _VP],
    "uw_matmul_plan": [_VP, _VP, _I64, _VP, _INT, ctypes.POINTER(Plan), _VP, _SZ, _VP],
    "uw_plan_workspace_size": [_VP, _I64, ctypes.POINTER(Plan), ctypes.POINTER(_SZ)],
    "uw_plan_for": [_VP, _I64, ctypes.POINTER(Plan)],
    "uw_matmul_host": [_VP, _VP, _I64, _VP, _INT, _VP, _SZ, _VP],
    "uw_matmul_host_async": [_VP, _VP, _I64, _VP, _INT, _VP, _SZ, _VP],
    "uw_host_workspace_size": [_VP, _I64, _INT, ctypes.POINTER(_SZ)],
    "uw_autotune": [_VP, ctypes.POINTER(_I64), _INT, _VP, _SZ, _VP],
    "uw_autotune_workspace_size": [_VP, ctypes.POINTER(_I64), _INT, ctypes.POINTER(_SZ)],
    "uw_tune_save": [_VP, ctypes.c_char_p, _SZ, ctypes.POINTER(_SZ)],
    "uw_tune_load": [_VP, ctypes.c_char_p],
    "uw_check": [_VP, _VP],
    "uw_matmul_noalloc": [_VP, _VP, _I64, _VP, _INT, _VP],
    "uw_sequence_workspace_size": [ctypes.POINTER(Step), _INT, _I64, ctypes.POINTER(_SZ)],
    "uw_sequence_run": [ctypes.POINTER(Step), _INT, _I64, _VP, _SZ, _VP, _VP, _INT],
    "uw_sequence_tune": [ctypes.POINTER(Step), _INT, _I64, _VP, _SZ, _VP, _VP, ctypes.POINTER(_INT)],
    "uw_status_string": [_INT],
    "uw_last_error": [],
    "uw_version": [],
}


def lib():
    """The loaded ``libuw.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _INT
        L.uw_free.restype = None
        L.uw_status_string.restype = ctypes.c_char_p
        L.uw_last_error.restype = ctypes.c_char_p
        L.uw_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def header_symbols():
    """Entry points declared in include/uw.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(uw_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, where: str):
    if status != OK:
        raise UwError(status, where, lib().uw_last_error().decode(errors="replace"))


def _ptr(t) -> int:
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def encode(w: np.ndarray, codec: int = CODEC_PALETTE, chunk: int = 256, max_len: int = 12) -> bytes:
    """Host encode of W[N,K] (numpy uint16 bf16 bit patterns)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    N, K = w.shape
    opts = EncodeOpts(codec, chunk, max_len)
    size = ctypes.c_size_t(0)
    _check(lib().uw_encode(w.ctypes.data, N, K, ctypes.byref(opts), None, 0, ctypes.byref(size)), "uw_encode")
    out = np.empty(size.value, np.uint8)
    _check(lib().uw_encode(w.ctypes.data, N, K, ctypes.byref(opts), out.ctypes.data, size.value, ctypes.byref(size)),
           "uw_encode")
    return out.tobytes()


def validate(blob: bytes) -> dict:
    info = Info()
    buf = np.frombuffer(blob, np.uint8)
    _check(lib().uw_blob_validate(buf.ctypes.data if len(blob) else None, len(blob), ctypes.byref(info)),
           "uw_blob_validate")
    return info.as_dict()


class Matrix:
    """A compressed matrix resident on the current CUDA device (owns a ``uw_matrix``)."""

    def __init__(self, blob: bytes, want_palette_form: bool = False, stream=None, resident=None):
        """resident: "huffman", "both" or "palette" (uw_resident); if None, want_palette_form picks "both" (True)
        or "huffman" (False)."""
        mode = RESIDENT[resident] if resident is not None else (RESIDENT_BOTH if want_palette_form else RESIDENT_HUFFMAN)
        buf = np.frombuffer(blob, np.uint8)
        h = ctypes.c_void_p()
        _check(lib().uw_load(buf.ctypes.data, len(blob), mode, _stream(stream), ctypes.byref(h)), "uw_load")
        self._h = h
        info = Info()
        _check(lib().uw_get_info(self._h, ctypes.byref(info)), "uw_get_info")
        self.info = info.as_dict()
        self.N, self.K = self.info["N"], self.info["K"]

    def close(self):
        if getattr(self, "_h", None):
            lib().uw_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def decode(self, out, stream=None):
        _check(lib().uw_decode(self._h, _ptr(out), _stream(stream)), "uw_decode")

    def workspace_size(self, B: int, strategy: int = STRAT_AUTO) -> int:
        n = ctypes.c_size_t(0)
        _check(lib().uw_workspace_size(self._h, B, strategy, ctypes.byref(n)), "uw_workspace_size")
        return n.value

    def plan_workspace_size(self, B: int, plan: Plan) -> int:
        n = ctypes.c_size_t(0)
        _check(lib().uw_plan_workspace_size(self._h, B, ctypes.byref(plan), ctypes.byref(n)), "uw_plan_workspace_size")
        return n.value

    def matmul(self, x, B: int, y, out_dtype: int = OUT_F32, strategy: int = STRAT_AUTO, workspace=None,
               ws_bytes: int = 0, stream=None):
        _check(lib().uw_matmul(self._h, _ptr(x), B, _ptr(y), out_dtype, strategy, _ptr(workspace), ws_bytes,
                               _stream(stream)), "uw_matmul")

    def matmul_plan(self, x, B: int, y, plan: Plan, out_dtype: int = OUT_F32, workspace=None, ws_bytes: int = 0,
                    stream=None):
        _check(lib().uw_matmul_plan(self._h, _ptr(x), B, _ptr(y), out_dtype, ctypes.byref(plan), _ptr(workspace),
                                    ws_bytes, _stream(stream)), "uw_matmul_plan")

    def plan_for(self, B: int) -> Plan:
        p = Plan()
        _check(lib().uw_plan_for(self._h, B, ctypes.byref(p)), "uw_plan_for")
        return p

    def host_workspace_size(self, B: int, out_dtype: int = OUT_F32) -> int:
        n = ctypes.c_size_t(0)
        _check(lib().uw_host_workspace_size(self._h, B, out_dtype, ctypes.byref(n)), "uw_host_workspace_size")
        return n.value

    def matmul_host(self, x_host, B: int, y_host, out_dtype: int, workspace, ws_bytes: int, stream=None):
        _check(lib().uw_matmul_host(self._h, _ptr(x_host), B, _ptr(y_host), out_dtype, _ptr(workspace), ws_bytes,
                                    _stream(stream)), "uw_matmul_host")

    def matmul_host_async(self, x_host, B: int, y_host, out_dtype: int, workspace, ws_bytes: int, stream=None):
        _check(lib().uw_matmul_host_async(self._h, _ptr(x_host), B, _ptr(y_host), out_dtype, _ptr(workspace),
                                          ws_bytes, _stream(stream)), "uw_matmul_host_async")

    def autotune_workspace_size(self, batches) -> int:
        arr = (ctypes.c_int64 * len(batches))(*batches)
        n = ctypes.c_size_t(0)
        _check(lib().uw_autotune_workspace_size(self._h, arr, len(batches), ctypes.byref(n)), "uw_autotune_workspace_size")
        return n.value

    def autotune(self, batches, workspace, ws_bytes: int, stream=None):
        arr = (ctypes.c_int64 * len(batches))(*batches)
        _check(lib().uw_autotune(self._h, arr, len(batches), _ptr(workspace), ws_bytes, _stream(stream)), "uw_autotune")

    def tune_save(self) -> str:
        n = ctypes.c_size_t(0)
        _check(lib().uw_tune_save(self._h, None, 0, ctypes.byref(n)), "uw_tune_save")
        buf = ctypes.create_string_buffer(n.value + 1)
        _check(lib().uw_tune_save(self._h, buf, n.value + 1, ctypes.byref(n)), "uw_tune_save")
        return buf.value.decode()

    def tune_load(self, text: str):
        _check(lib().uw_tune_load(self._h, text.encode()), "uw_tune_load")

    def matmul_noalloc(self, x, B: int, y, out_dtype: int = OUT_F32, stream=None):
        _check(lib().uw_matmul_noalloc(self._h, _ptr(x), B, _ptr(y), out_dtype, _stream(stream)), "uw_matmul_noalloc")

    def check(self, stream=None):
        _check(lib().uw_check(self._h, _stream(stream)), "uw_check")


def _steps(steps):
    arr = (Step * max(1, len(steps)))()
    for i, st in enumerate(steps):
        m, x, y = st[0], st[1], st[2]
        od = st[3] if len(st) > 3 else OUT_F32
        fl = st[4] if len(st) > 4 else 0
        arr[i] = Step(m.handle.value if isinstance(m, Matrix) else m, _ptr(x), _ptr(y), od, fl)
    return arr


def sequence_workspace_size(steps, B: int) -> int:
    """Workspace bytes of uw_sequence_run; steps: (Matrix, x, y[, out_dtype[, flags]]) tuples."""
    n = ctypes.c_size_t(0)
    _check(lib().uw_sequence_workspace_size(_steps(steps), len(steps), B, ctypes.byref(n)), "uw_sequence_workspace_size")
    return n.value


def sequence_run(steps, B: int, workspace, ws_bytes: int, stream=None, side_stream=None, decode_sms: int = 0):
    """uw_sequence_run: the steps in order on `stream`, hard steps' transcodes on `side_stream` (on `decode_sms`
    SMs beside the matmuls when it is > 0; SEQ_DIRECT: no transcode, every step its own AUTO plan)."""
    _check(lib().uw_sequence_run(_steps(steps), len(steps), B, _ptr(workspace), ws_bytes, _stream(stream),
                                 _stream(side_stream), decode_sms), "uw_sequence_run")


def sequence_tune(steps, B: int, workspace, ws_bytes: int, stream=None, side_stream=None) -> int:
    """uw_sequence_tune: the fastest decode SM split for these steps."""
    d = ctypes.c_int(0)
    _check(lib().uw_sequence_tune(_steps(steps), len(steps), B, _ptr(workspace), ws_bytes, _stream(stream),
                                  _stream(side_stream), ctypes.byref(d)), "uw_sequence_tune")
    return d.value
