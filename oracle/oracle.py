"""Python access to the CPU oracle (qk_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the package smoke check and
the benchmark's CPU-baseline leg, never by the product path.  The C source is
compiled with gcc -O2 (no -ffast-math) into oracle/_build/ on first use.

Every function returns f64 results.  Rows are addressed by an explicit index
list so that a full-size tensor can be checked on sampled rows.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qk_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libqk_oracle.so")

FMT = {"q8_0": 0, "q4_k": 1, "q6_k": 2}
QK = {"q8_0": 32, "q4_k": 256, "q6_k": 256}
BLOCK_BYTES = {"q8_0": 34, "q4_k": 144, "q6_k": 210}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall",
                               "-fno-fast-math", "-ffp-contract=off", SRC, "-o", tmp, "-lm"])
        os.replace(tmp, LIB)
    return LIB


def _load(path: str | None = None):
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using(path: str):
    """Temporarily route every call through another build of the oracle
    (used by the tests that check the pins reject planted mistakes)."""
    global _lib
    with _lock:
        old = _lib
        _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        with _lock:
            _lib = old


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.qko_fp16_to_f64.argtypes = [ctypes.c_uint16]
    lib.qko_fp16_to_f64.restype = ctypes.c_double
    lib.qko_f64_to_fp16.argtypes = [ctypes.c_double]
    lib.qko_f64_to_fp16.restype = ctypes.c_uint16
    lib.qko_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.qko_f32_to_bf16.restype = ctypes.c_uint16
    lib.qko_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.qko_bf16_to_f64.restype = ctypes.c_double
    lib.qko_decode_rows.argtypes = [ctypes.c_int, P, I64, P, I64, P]
    lib.qko_decode_rows.restype = ctypes.c_int
    lib.qko_gemv.argtypes = [ctypes.c_int, P, I64, P, I64, P, I64, P, P]
    lib.qko_gemv.restype = ctypes.c_int
    lib.qko_gemm_bf16.argtypes = [ctypes.c_int, P, I64, P, I64, P, I64, P, P]
    lib.qko_swiglu.argtypes = [ctypes.c_int, P, I64, P, P, I64, P, I64, P, P, P, P, P]
    lib.qko_experts.argtypes = [ctypes.c_int, P, I64, I64, I64, P, I64, P, I64, P, P]
    lib.qko_swiglu_gemm_bf16.argtypes = [ctypes.c_int, P, I64, P, P, I64, P, I64, P, P, P, P, P]
    lib.qko_swiglu_gemm_bf16.restype = ctypes.c_int
    lib.qko_experts.restype = ctypes.c_int
    lib.qko_swiglu.restype = ctypes.c_int
    lib.qko_gemm_bf16.restype = ctypes.c_int
    lib.qko_quantise_q8_0_row.argtypes = [P, I64, P]
    lib.qko_quantise_q8_0_row.restype = None
    lib.qko_quantise_q4_k_row.argtypes = [P, I64, P]
    lib.qko_quantise_q4_k_row.restype = None
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def row_bytes(fmt: str, K: int) -> int:
    return ((K + QK[fmt] - 1) // QK[fmt]) * BLOCK_BYTES[fmt]


def _rows_arg(rows, n_total=None):
    if rows is None:
        rows = np.arange(n_total, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


# ------------------------------------------------------------------ scalars

def fp16_to_f64(bits: int, lib=None) -> float:
    return (lib or _load()).qko_fp16_to_f64(int(bits))


def f64_to_fp16(v: float, lib=None) -> int:
    return int((lib or _load()).qko_f64_to_fp16(float(v)))


def f32_to_bf16(v: float, lib=None) -> int:
    return int((lib or _load()).qko_f32_to_bf16(float(np.float32(v))))


def bf16_to_f64(bits: int, lib=None) -> float:
    return (lib or _load()).qko_bf16_to_f64(int(bits))


# ------------------------------------------------------------------ tensors

def decode(fmt: str, wq: np.ndarray, K: int, rows=None, n_rows_total=None, lib=None) -> np.ndarray:
    """Decoded weights W[rows][K] as f64."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    if rows is None:
        n_rows_total = wq.size // row_bytes(fmt, K)
    r = _rows_arg(rows, n_rows_total)
    out = np.empty((r.size, K), dtype=np.float64)
    rc = (lib or _load()).qko_decode_rows(FMT[fmt], _ptr(wq), K, _ptr(r), r.size, _ptr(out))
    assert rc == 0
    return out


def gemv(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, rows=None, lib=None):
    """(y, S): y[b][i] = sum_c W[rows[i]][c] x[b][c], S = sum |W x|, both f64."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == K
    r = _rows_arg(rows, wq.size // row_bytes(fmt, K))
    B = x.shape[0]
    y = np.empty((B, r.size), dtype=np.float64)
    s = np.empty((B, r.size), dtype=np.float64)
    rc = (lib or _load()).qko_gemv(FMT[fmt], _ptr(wq), K, _ptr(r), r.size, _ptr(x), B,
                                    _ptr(y), _ptr(s))
    assert rc == 0
    return y, s


def swiglu(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, gate_rows, up_rows, lib=None):
    """(h, g, u, Sg, Su), all f64 [batch][n]: g and u the matvecs of the gate and
    up rows, h = silu(g) * u with silu(z) = z / (1 + e^-z)."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == K
    nr = wq.size // row_bytes(fmt, K)
    gr = _rows_arg(gate_rows, nr)
    ur = _rows_arg(up_rows, nr)
    assert gr.size == ur.size
    B, n = x.shape[0], gr.size
    out = [np.empty((B, n), dtype=np.float64) for _ in range(5)]
    rc = (lib or _load()).qko_swiglu(FMT[fmt], _ptr(wq), K, _ptr(gr), _ptr(ur), n, _ptr(x), B,
                                     *[_ptr(o) for o in out])
    assert rc == 0
    return tuple(out)


def swiglu_gemm_bf16(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, gate_rows, up_rows, lib=None):
    """(h, g, u, Sg, Su), f64 [M][n]: g, u the bf16 GEMM references of the gate and
    up rows, h = silu(g) * u."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == K
    nr = wq.size // row_bytes(fmt, K)
    gr = _rows_arg(gate_rows, nr)
    ur = _rows_arg(up_rows, nr)
    assert gr.size == ur.size
    M, n = x.shape[0], gr.size
    out = [np.empty((M, n), dtype=np.float64) for _ in range(5)]
    rc = (lib or _load()).qko_swiglu_gemm_bf16(FMT[fmt], _ptr(wq), K, _ptr(gr), _ptr(ur), n, _ptr(x), M,
                                               *[_ptr(o) for o in out])
    assert rc == 0
    return tuple(out)


def experts(fmt: str, wq: np.ndarray, n_experts: int, rows: int, K: int, x: np.ndarray, xk: int,
            expid, lib=None):
    """(y, S), f64 [n_assign][rows]: y[a][r] = sum_c W[expid[a]*rows + r][c] x[a // xk][c]."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == K
    ids = np.ascontiguousarray(expid, dtype=np.int32)
    n = ids.size
    assert x.shape[0] * xk >= n
    y = np.empty((n, rows), dtype=np.float64)
    s = np.empty((n, rows), dtype=np.float64)
    rc = (lib or _load()).qko_experts(FMT[fmt], _ptr(wq), n_experts, rows, K, _ptr(x), xk, _ptr(ids), n,
                                      _ptr(y), _ptr(s))
    assert rc == 0, rc
    return y, s


def gemm_bf16(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, rows=None, lib=None):
    """(y, S) of the bf16-rounded reference: y[m][i] = sum_c bf16(fp32(W)) bf16(x)."""
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    assert x.shape[1] == K
    r = _rows_arg(rows, wq.size // row_bytes(fmt, K))
    M = x.shape[0]
    y = np.empty((M, r.size), dtype=np.float64)
    s = np.empty((M, r.size), dtype=np.float64)
    rc = (lib or _load()).qko_gemm_bf16(FMT[fmt], _ptr(wq), K, _ptr(r), r.size, _ptr(x), M,
                                         _ptr(y), _ptr(s))
    assert rc == 0
    return y, s


def quantise(fmt: str, w: np.ndarray, lib=None) -> np.ndarray:
    """Encode f64 weights W[rows][K] into raw block bytes (round-trip checks)."""
    w = np.ascontiguousarray(np.atleast_2d(w), dtype=np.float64)
    rows, K = w.shape
    rb = row_bytes(fmt, K)
    out = np.zeros(rows * rb, dtype=np.uint8)
    L = lib or _load()
    fn = L.qko_quantise_q8_0_row if fmt == "q8_0" else L.qko_quantise_q4_k_row
    for r in range(rows):
        fn(_ptr(w[r]), K, ctypes.c_void_p(out.ctypes.data + r * rb))
    return out


def gemv_threaded(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, rows, threads: int,
                  lib=None):
    """The same oracle GEMV, run on `threads` host threads over contiguous row
    bands (ctypes releases the GIL during the call).  Each output is computed
    by the same code in the same order, so results equal the serial run."""
    rows = _rows_arg(rows)
    bands = np.array_split(rows, max(1, threads))
    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        parts = list(ex.map(lambda b: gemv(fmt, wq, K, x, b, lib=lib), bands))
    y = np.concatenate([p[0] for p in parts], axis=1)
    s = np.concatenate([p[1] for p in parts], axis=1)
    return y, s


def gemm_bf16_threaded(fmt: str, wq: np.ndarray, K: int, x: np.ndarray, rows, threads: int, lib=None):
    """gemm_bf16 on `threads` host threads over contiguous row bands (same
    code and order per output as the serial call)."""
    rows = _rows_arg(rows)
    bands = np.array_split(rows, max(1, threads))
    with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
        parts = list(ex.map(lambda b: gemm_bf16(fmt, wq, K, x, b, lib=lib), bands))
    return np.concatenate([p[0] for p in parts], axis=1), np.concatenate([p[1] for p in parts], axis=1)


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
