"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

Only random draws and BF16 rounding live here (see ``synth.c``); nothing of the
codec or the matmul.  Every tensor is returned as a numpy ``uint16`` array of
BF16 bit patterns.

Workload recipes stand in for the trained Llama-3.1-8B / 70B MLP weights the
Unweight post measured on (Cloudflare blog, "Unweight", results section); no
trained weights are used.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

NORMAL, STUDENT_T3 = 0, 1
SEED_BASE = 0x55574D00


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` in place (gcc, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.synth_fill_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int,
                                            ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                            ctypes.c_double, ctypes.c_double]
            lib.synth_fill_bf16.restype = None
            lib.synth_fill_u16_bits.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64]
            lib.synth_fill_u16_bits.restype = None
            _lib = lib
    return _lib


def fill(shape, seed: int, kind: int = NORMAL, scale: float = 1.0,
         p1: float = 0.0, f1: float = 1.0, p2: float = 0.0, f2: float = 1.0) -> np.ndarray:
    """BF16 bit patterns of ``scale * Z`` (or ``scale * t_3``) with two optional outlier classes."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_fill_bf16(out.ctypes.data, out.size, seed & (2**64 - 1), kind, scale, p1, f1, p2, f2)
    return out


def random_bits(shape, seed: int) -> np.ndarray:
    """Uniformly random 16-bit patterns (every BF16 class, NaNs and infinities included)."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_fill_u16_bits(out.ctypes.data, out.size, seed & (2**64 - 1))
    return out


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# Workload recipes.  Seeds: SEED_BASE + config_id*1000 + layer*3 + {0 gate, 1 up, 2 down};
# activations use the matrix seed + 500.
# ---------------------------------------------------------------------------
class Matrix:
    def __init__(self, name, N, K, seed, kind=NORMAL, scale=0.02, p1=0.0, f1=1.0, p2=0.0, f2=1.0):
        self.name, self.N, self.K, self.seed = name, N, K, seed
        self.kind, self.scale, self.p1, self.f1, self.p2, self.f2 = kind, scale, p1, f1, p2, f2

    def weights(self) -> np.ndarray:
        return fill((self.N, self.K), self.seed, self.kind, self.scale, self.p1, self.f1, self.p2, self.f2)

    def activations(self, B: int) -> np.ndarray:
        return fill((B, self.K), self.seed + 500, NORMAL, 1.0)

    def __repr__(self):
        return f"Matrix({self.name}, N={self.N}, K={self.K}, seed={self.seed:#x})"


def _seed(cfg, layer, proj):
    return SEED_BASE + cfg * 1000 + layer * 3 + proj


def tiny() -> Matrix:
    """W[256,512] ~ N(0,0.02); 0.1% of entries x64, 0.1% x2^-20 (out-of-palette exponents)."""
    return Matrix("tiny", 256, 512, _seed(0, 0, 0), NORMAL, 0.02, 1e-3, 64.0, 1e-3, 2.0 ** -20)


def gate_8b() -> Matrix:
    """Llama-3.1-8B-shaped gate_proj W[14336,4096] ~ N(0,0.02) with 1e-4 of entries x100."""
    return Matrix("gate_8b", 14336, 4096, _seed(1, 0, 0), NORMAL, 0.02, 1e-4, 100.0)


def stack_8b(layers: int = 32):
    """32 layers x (gate, up W[14336,4096]; down W[4096,14336]) ~ N(0,0.02), per-layer seeds."""
    out = []
    for l in range(layers):
        out.append(Matrix(f"stack_8b.l{l}.gate", 14336, 4096, _seed(2, l, 0)))
        out.append(Matrix(f"stack_8b.l{l}.up", 14336, 4096, _seed(2, l, 1)))
        out.append(Matrix(f"stack_8b.l{l}.down", 4096, 14336, _seed(2, l, 2)))
    return out


def heavy_tail() -> Matrix:
    """W[8192,8192] = 0.02 * Student-t(nu=3)."""
    return Matrix("heavy_tail", 8192, 8192, _seed(3, 0, 0), STUDENT_T3, 0.02)


def mlp_70b():
    """70B-shaped MLP: gate/up W[28672,8192], down W[8192,28672] ~ N(0,0.015), 1e-4 x100."""
    return [Matrix("mlp_70b.gate", 28672, 8192, _seed(4, 0, 0), NORMAL, 0.015, 1e-4, 100.0),
            Matrix("mlp_70b.up", 28672, 8192, _seed(4, 0, 1), NORMAL, 0.015, 1e-4, 100.0),
            Matrix("mlp_70b.down", 8192, 28672, _seed(4, 0, 2), NORMAL, 0.015, 1e-4, 100.0)]


BATCHES = {"tiny": [1], "gate_8b": [1, 4, 16], "stack_8b": [1, 8, 32, 128],
           "heavy_tail": [1, 16, 64], "mlp_70b": [1, 32, 256, 512]}
