"""CPU oracle for the MoE routing step (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library path never does: the CUDA
library and this oracle share no code.

The oracle itself is plain C in ``oracle.c``; this module compiles it with gcc
into ``liboracle.so`` next to the source and wraps it with ctypes, converting
numpy arrays to pointers and nothing else.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

DT = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_sigmoid.argtypes = [ctypes.c_float]
    lib.oracle_sigmoid.restype = ctypes.c_float
    lib.oracle_sigmoid_array.argtypes = [P, I, P, ctypes.c_long]
    lib.oracle_sigmoid_array.restype = None
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_num_experts.argtypes = [I, I, I, I]
    lib.oracle_num_experts.restype = I
    lib.oracle_route.argtypes = [P, I, P, I, I, I, I, I, ctypes.c_float, I, I, P, P, P, P, P]
    lib.oracle_route.restype = I
    lib.oracle_router_gemm.argtypes = [P, P, I, I, I, P]
    lib.oracle_router_gemm.restype = None
    lib.oracle_route_layout.argtypes = [P, P, P, I, I, I, I, P, P, P, P]
    lib.oracle_route_layout.restype = I
    lib.oracle_route_index.argtypes = [P, I, I, I, P, P, P]
    lib.oracle_route_index.restype = I
    lib.oracle_dispatch_counts.argtypes = [P, I, I, I, P, P]
    lib.oracle_dispatch_counts.restype = I
    lib.oracle_alltoall_layout.argtypes = [P, I, I, P, P, P]
    lib.oracle_alltoall_layout.restype = I
    lib.oracle_mxfp4_quant.argtypes = [P, I, I, P, P]
    lib.oracle_mxfp4_quant.restype = I
    lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
    lib.oracle_e2m1_encode.restype = ctypes.c_uint8
    return lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_experts(E: int, k: int, off: int, cnt: int, lib=None) -> int:
    return (lib or load()).oracle_num_experts(E, k, off, cnt)


def sigmoid(x: np.ndarray, dtype: str = "f32", lib=None) -> np.ndarray:
    """Oracle scores of an array of float32 values or bf16 bit patterns (same shape)."""
    lib = lib or load()
    xa = np.ascontiguousarray(x, dtype=np.float32 if dtype == "f32" else np.uint16)
    s = np.empty(xa.shape, dtype=np.float32)
    lib.oracle_sigmoid_array(_ptr(xa), DT[dtype], _ptr(s), xa.size)
    return s


def f32_to_bf16(x: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)


def route(logits: np.ndarray, dtype: str, bias: np.ndarray, T: int, E: int, k: int, G: int,
          Kg: int, scale: float, off: int = 0, cnt: int = 0, lib=None, **_ignored) -> dict:
    """Run the oracle router; returns packed, counts, offsets, perm, ids (global), NE."""
    lib = lib or load()
    want = np.float32 if dtype == "f32" else np.uint16
    lg = np.ascontiguousarray(logits, dtype=want)
    bs = np.ascontiguousarray(bias, dtype=np.float32)
    NE = lib.oracle_num_experts(E, k, off, cnt)
    packed = np.zeros(max(T * k, 1), dtype=np.int32)
    ids = np.zeros(max(T * k, 1), dtype=np.int32)
    perm = np.zeros(max(T * k, 1), dtype=np.int32)
    counts = np.zeros(max(NE, 1), dtype=np.int32)
    offsets = np.zeros(max(NE, 0) + 1, dtype=np.int32)
    rc = lib.oracle_route(_ptr(lg), DT[dtype], _ptr(bs), T, E, k, G, Kg, float(scale), off, cnt,
                          _ptr(packed), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(ids))
    if rc != 0:
        raise ValueError(f"oracle_route rejected the arguments (rc={rc})")
    return dict(packed=packed[:T * k].reshape(T, k), ids=ids[:T * k].reshape(T, k),
                perm=perm[:T * k], counts=counts[:NE], offsets=offsets[:NE + 1], NE=NE)


def route_cfg(cfg: dict, lib=None) -> dict:
    return route(cfg["logits"], cfg["dtype"], cfg["bias"], cfg["T"], cfg["E"], cfg["k"], cfg["G"],
                 cfg["Kg"], cfg["scale"], cfg.get("off", 0), cfg.get("cnt", 0), lib=lib)


def router_gemm(hidden: np.ndarray, w: np.ndarray, lib=None) -> np.ndarray:
    lib = lib or load()
    h = np.ascontiguousarray(hidden, dtype=np.uint16)
    ww = np.ascontiguousarray(w, dtype=np.uint16)
    T, H = h.shape
    E = ww.shape[0]
    out = np.zeros((T, E), dtype=np.float64)
    lib.oracle_router_gemm(_ptr(h), _ptr(ww), T, H, E, _ptr(out))
    return out


def route_layout(counts: np.ndarray, offsets: np.ndarray, perm: np.ndarray, tile: int,
                 capacity: int | None = None, lib=None) -> dict:
    """Inverse permutation, padded offsets, padded rows and m_indices of a routing
    result (see oracle_route_layout).  capacity defaults to the padded total's bound
    n + NE * (tile - 1)."""
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    perm = np.ascontiguousarray(perm, dtype=np.int32).ravel()
    NE, n = counts.size, perm.size
    cap = n + NE * (tile - 1) if capacity is None else capacity
    inv = np.empty(n, np.int32)
    poff = np.empty(NE + 1, np.int32)
    rows = np.empty(max(cap, 0), np.int32)
    mind = np.empty(max(cap, 0), np.int32)
    total = (lib or load()).oracle_route_layout(_ptr(counts), _ptr(offsets), _ptr(perm), n, NE,
                                                tile, cap, _ptr(inv), _ptr(poff), _ptr(rows),
                                                _ptr(mind))
    if total < 0:
        raise ValueError("oracle_route_layout rejected its arguments")
    return dict(inv_perm=inv, padded_offsets=poff, padded_rows=rows, m_indices=mind, total=total)


def route_index(packed: np.ndarray, NE: int, lib=None) -> dict:
    """counts, offsets and perm of packed values [T, k] (steps 10-12 alone)."""
    packed = np.ascontiguousarray(packed, dtype=np.int32)
    T, k = packed.shape
    counts = np.empty(NE, np.int32)
    offsets = np.empty(NE + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    rc = (lib or load()).oracle_route_index(_ptr(packed), T, k, NE, _ptr(counts), _ptr(offsets),
                                            _ptr(perm))
    if rc != 0:
        raise ValueError("oracle_route_index rejected its arguments")
    return dict(counts=counts, offsets=offsets, perm=perm)


def dispatch_counts(ids: np.ndarray, E: int, R: int, lib=None) -> dict:
    """Entries per destination rank for global expert ids (R ranks, E / R experts each)."""
    ids = np.ascontiguousarray(ids, dtype=np.int32).ravel()
    sc = np.empty(R, np.int32)
    so = np.empty(R + 1, np.int32)
    rc = (lib or load()).oracle_dispatch_counts(_ptr(ids), ids.size, E, R, _ptr(sc), _ptr(so))
    if rc != 0:
        raise ValueError("oracle_dispatch_counts rejected its arguments")
    return dict(send_counts=sc, send_offsets=so)


def alltoall_layout(matrix: np.ndarray, me: int, lib=None) -> dict:
    """send displacements, receive counts and displacements of rank `me`."""
    m = np.ascontiguousarray(matrix, dtype=np.int32)
    R = m.shape[0]
    sd = np.empty(R + 1, np.int32)
    rcnt = np.empty(R, np.int32)
    rd = np.empty(R + 1, np.int32)
    rc = (lib or load()).oracle_alltoall_layout(_ptr(m), R, me, _ptr(sd), _ptr(rcnt), _ptr(rd))
    if rc != 0:
        raise ValueError("oracle_alltoall_layout rejected its arguments")
    return dict(send_displs=sd, recv_counts=rcnt, recv_displs=rd)


def mxfp4_quant(x: np.ndarray, lib=None) -> dict:
    """MXFP4 codes q [T, H / 2] (two E2M1 codes per byte, even element low) and E8M0
    scales [T, H / 32] of bf16 activations x [T, H] (see oracle_mxfp4_quant)."""
    xa = np.ascontiguousarray(x, dtype=np.uint16)
    T, H = xa.shape
    q = np.empty((T, H // 2), np.uint8)
    sc = np.empty((T, H // 32), np.uint8)
    rc = (lib or load()).oracle_mxfp4_quant(_ptr(xa), T, H, _ptr(q), _ptr(sc))
    if rc != 0:
        raise ValueError("oracle_mxfp4_quant rejected its arguments")
    return dict(q=q, scales=sc)


def e2m1_encode(v: float, lib=None) -> int:
    return int((lib or load()).oracle_e2m1_encode(float(v)))
