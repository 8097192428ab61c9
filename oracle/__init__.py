"""fp64 CPU oracle for D = alpha*(A*B) + beta*C + x_factor*X and Y = A*B.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  Nothing in the CUDA
library or its Python binding imports this package, and this package imports
nothing from them.

The arithmetic lives in ``oracle.c`` (plain C, fp64, no fast-math); this file
only compiles it with gcc and marshals numpy arrays.  See ``oracle.c`` for the
definition, the page citations and the layout conventions.

Type codes here are the oracle's own: ``"f32"``, ``"f16"``, ``"bf16"``,
``"e4m3"``, ``"e5m2"``.  Input buffers are numpy arrays holding the raw storage
(float32, uint16 bit patterns for f16/bf16, uint8 codes for fp8), laid out as
``oracle.c`` describes.  Outputs come back in logical [L, M, N] order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"f32": 0, "f16": 1, "bf16": 2, "e4m3": 3, "e5m2": 4, "tf32": 5}
STORAGE = {"f32": np.float32, "f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8,
           "e5m2": np.uint8, "tf32": np.float32}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, -O2,
    contraction off so results do not depend on the host's FMA use)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB_OVERRIDE: a deliberately broken copy, built by the
            # mutation tests to show that the pins catch planted mistakes.
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            lib = ctypes.CDLL(override if override else build())
            i64, i32, f64, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.oracle_decode.restype = f64
            lib.oracle_decode.argtypes = [i32, ctypes.c_uint32]
            lib.oracle_round.restype = None
            lib.oracle_round.argtypes = [i32, vp, i64, vp]
            common = [i64, i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, vp, i32, i32, i32, i32,
                      i32, f64, f64, f64, i32, i32, i32, i64]
            lib.oracle_gemm_rows.restype = i32
            lib.oracle_gemm_rows.argtypes = common + [i64, i64, vp, vp, vp, vp, i32]
            lib.oracle_gemm_entries.restype = i32
            lib.oracle_gemm_entries.argtypes = common + [vp, vp, vp, i64, vp, vp, vp, vp, i32]
            lib.oracle_max_threads.restype = i32
            lib.oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return _load().oracle_max_threads()


def decode(dtype: str, codes) -> np.ndarray:
    """Exact fp64 value of each storage code (bit pattern) of `dtype`."""
    lib = _load()
    codes = np.asarray(codes).astype(np.uint64).ravel()
    return np.array([lib.oracle_decode(DTYPES[dtype], int(c)) for c in codes], dtype=np.float64)


def round_to(dtype: str, values) -> np.ndarray:
    """Round fp64 values once (RNE) into `dtype` storage (f32, f16 or bf16)."""
    lib = _load()
    v = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(v.shape, dtype=STORAGE[dtype])
    lib.oracle_round(DTYPES[dtype], v.ctypes.data, v.size, out.ctypes.data)
    return out


class Problem:
    """Raw storage buffers plus the shape, layout, type and scalar arguments.

    a_mn_major: A stored M-major ([L][K][lda]) instead of K-major ([L][M][lda]).
    b_mn_major: B stored N-major ([L][K][ldb]) instead of K-major ([L][N][ldb]).
    cd_m_major: C/X stored M-major ([L][N][M]) instead of N-major ([L][M][N]).
    use_c / use_x: whether beta*C / x_factor*X take part (C, X may be None).
    b_dtype: B's type when it differs from A's (fp8 pairs); None = ab_dtype.
    relu: D = max(alpha*acc + beta*C, 0) + x_factor*X.
    acc_chunk: > 0 makes gemm_rows / gemm_entries also return P, the sum over
        the chunk boundaries (every acc_chunk k, and k = K) of the magnitude of
        the exact running sum: the scale of the error a half-precision
        accumulator, rounded once per chunk, may add.  P is not part of the result.
    """

    def __init__(self, M, N, K, L, A, lda, a_mn_major, B, ldb, b_mn_major, C, X,
                 ab_dtype, c_dtype="f32", x_dtype="f32", cd_m_major=False,
                 alpha=1.0, beta=0.0, x_factor=0.0, use_c=None, use_x=None, b_dtype=None,
                 relu=False, acc_chunk=0):
        self.M, self.N, self.K, self.L = int(M), int(N), int(K), int(L)
        self.A = None if A is None else np.ascontiguousarray(A)
        self.B = None if B is None else np.ascontiguousarray(B)
        self.C = None if C is None else np.ascontiguousarray(C)
        self.X = None if X is None else np.ascontiguousarray(X)
        self.lda, self.ldb = int(lda), int(ldb)
        self.a_mn_major, self.b_mn_major = bool(a_mn_major), bool(b_mn_major)
        self.ab_dtype, self.c_dtype, self.x_dtype = ab_dtype, c_dtype, x_dtype
        self.b_dtype = ab_dtype if b_dtype is None else b_dtype
        self.relu = bool(relu)
        self.acc_chunk = int(acc_chunk)
        self.cd_m_major = bool(cd_m_major)
        self.alpha, self.beta, self.x_factor = float(alpha), float(beta), float(x_factor)
        self.use_c = (self.C is not None and self.beta != 0.0) if use_c is None else bool(use_c)
        self.use_x = (self.X is not None and self.x_factor != 0.0) if use_x is None else bool(use_x)

    def _common(self):
        ptr = lambda a: None if a is None else a.ctypes.data
        return [self.M, self.N, self.K, self.L, ptr(self.A), self.lda, int(self.a_mn_major),
                ptr(self.B), self.ldb, int(self.b_mn_major), ptr(self.C), ptr(self.X),
                DTYPES[self.ab_dtype], DTYPES[self.b_dtype], DTYPES[self.c_dtype],
                DTYPES[self.x_dtype], int(self.cd_m_major), self.alpha, self.beta, self.x_factor,
                int(self.use_c), int(self.use_x), int(self.relu), self.acc_chunk]


def gemm_rows(p: Problem, m0: int = 0, m1: int | None = None, nthreads: int = 0):
    """Exact (fp64) D, Y and sum|a*b| for rows [m0, m1) of every batch.

    Returns three float64 arrays of shape [L, m1-m0, N] -- four (P last) when
    p.acc_chunk > 0."""
    lib = _load()
    m1 = p.M if m1 is None else int(m1)
    shape = (p.L, m1 - m0, p.N)
    D = np.empty(shape, np.float64)
    Y = np.empty(shape, np.float64)
    S = np.empty(shape, np.float64)
    P = np.empty(shape, np.float64) if p.acc_chunk > 0 else None
    rc = lib.oracle_gemm_rows(*p._common(), int(m0), m1, D.ctypes.data, Y.ctypes.data,
                              S.ctypes.data, None if P is None else P.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_rows: bad arguments")
    return (D, Y, S) if P is None else (D, Y, S, P)


def gemm(p: Problem, nthreads: int = 0):
    """Exact D, Y and sum|a*b| (and P, see Problem) for the whole problem, each
    [L, M, N] float64."""
    return gemm_rows(p, 0, p.M, nthreads)


def gemm_entries(p: Problem, ms, ns, ls, nthreads: int = 0):
    """Exact D, Y and sum|a*b| (and P, see Problem) at the listed (m, n, l)
    entries (1-D arrays)."""
    lib = _load()
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    ls = np.ascontiguousarray(ls, dtype=np.int64)
    n = ms.size
    D = np.empty(n, np.float64)
    Y = np.empty(n, np.float64)
    S = np.empty(n, np.float64)
    P = np.empty(n, np.float64) if p.acc_chunk > 0 else None
    rc = lib.oracle_gemm_entries(*p._common(), ms.ctypes.data, ns.ctypes.data, ls.ctypes.data,
                                 n, D.ctypes.data, Y.ctypes.data, S.ctypes.data,
                                 None if P is None else P.ctypes.data, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_entries: bad arguments")
    return (D, Y, S) if P is None else (D, Y, S, P)
