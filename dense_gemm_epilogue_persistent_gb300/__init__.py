"""Python binding of the GB300 persistent batched GEMM with fused epilogue.

Thin ctypes layer over ``libgemm_gb300.so`` (C ABI in ``include/gemm_gb300.h``):
the functions below carry the C entry points' names and only marshal
arguments.  Every step of the computation runs in the library's CUDA kernel;
there is no fallback, and a missing library raises immediately.

    Y = A*B,   D = alpha*(A*B) + beta*C + x_factor*X

Tensor arguments may be raw device addresses (int) or objects with a
``data_ptr()`` method (e.g. torch CUDA tensors); streams may be an int handle
or an object with a ``cuda_stream`` attribute.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# The library for a process that drives one GPU (every kernel variant), and
# the one for processes that drive several GPUs (no multicast kernels).
LIB_PATH = os.path.join(_HERE, "libgemm_gb300.so")
NOMC_LIB_PATH = os.path.join(_HERE, "libgemm_gb300_nomc.so")

# enums (include/gemm_gb300.h)
GEMM_OK = 0
GEMM_ERR_INVALID_ARG = 1
GEMM_ERR_UNSUPPORTED_DTYPE = 2
GEMM_ERR_MISALIGNED = 3
GEMM_ERR_UNSUPPORTED_ARCH = 4
GEMM_ERR_CUDA = 5
GEMM_ERR_DEVICE_TIMEOUT = 6
GEMM_ERR_UNSUPPORTED_CONFIG = 7
GEMM_ERR_DEVICE_CHECK = 8

GEMM_F32, GEMM_F16, GEMM_BF16, GEMM_E4M3, GEMM_E5M2, GEMM_TF32 = 0, 1, 2, 3, 4, 5
GEMM_K_MAJOR, GEMM_MN_MAJOR = 0, 1
GEMM_EPI_LINEAR, GEMM_EPI_RELU = 0, 1
GEMM_RING_STAT_WORDS = 16

DTYPE_CODES = {"f32": GEMM_F32, "f16": GEMM_F16, "bf16": GEMM_BF16, "e4m3": GEMM_E4M3,
               "e5m2": GEMM_E5M2, "tf32": GEMM_TF32}


class gemm_dtypes_t(ctypes.Structure):
    _fields_ = [("ab", ctypes.c_int), ("c", ctypes.c_int), ("d", ctypes.c_int),
                ("x", ctypes.c_int), ("y", ctypes.c_int), ("cdxy_major", ctypes.c_int),
                ("b", ctypes.c_int), ("epilogue", ctypes.c_int), ("acc", ctypes.c_int)]


class gemm_config_t(ctypes.Structure):
    _fields_ = [("cta_group", ctypes.c_int), ("tile_n", ctypes.c_int), ("stages", ctypes.c_int),
                ("group_m", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_k", ctypes.c_int),
                ("acc_stages", ctypes.c_int), ("ring_bytes", ctypes.c_int),
                ("smem_bytes", ctypes.c_int), ("tiles", ctypes.c_int64),
                ("grid_ctas", ctypes.c_int), ("epi_slots", ctypes.c_int),
                ("epi_slot_bytes", ctypes.c_int), ("cluster_m", ctypes.c_int),
                ("l2_hints", ctypes.c_int), ("epi_wait_ns", ctypes.c_int),
                ("inject_stall", ctypes.c_int), ("tail_split", ctypes.c_int),
                ("cluster_n", ctypes.c_int),
                ("epi_warps", ctypes.c_int),
                ("stream_k", ctypes.c_int)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class gemm_problem_t(ctypes.Structure):
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("L", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64), ("layoutA", ctypes.c_int),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64), ("layoutB", ctypes.c_int),
                ("C", ctypes.c_void_p), ("X", ctypes.c_void_p), ("D", ctypes.c_void_p),
                ("Y", ctypes.c_void_p),
                ("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("x_factor", ctypes.c_float),
                ("dtypes", gemm_dtypes_t)]


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {gemm_status_string(status)}" if what else
                         gemm_status_string(status))


_lock = threading.Lock()
_lib = None


def select_library(path: str) -> None:
    """Load the library at `path` instead of the product one (the
    ring-statistics build, for instance).  Must precede the first call."""
    global LIB_PATH
    with _lock:
        if _lib is not None and os.path.abspath(path) != os.path.abspath(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is already loaded")
        LIB_PATH = path


def library():
    """Load libgemm_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            lib = ctypes.CDLL(LIB_PATH)
            i32, i64, f32, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
            lib.gemm_create.argtypes = [ctypes.POINTER(vp), i32]
            lib.gemm_destroy.argtypes = [vp]
            lib.gemm_run.argtypes = [vp, i64, i64, i64, i64, vp, i64, i32, vp, i64, i32, vp, vp,
                                     vp, vp, f32, f32, f32, ctypes.POINTER(gemm_dtypes_t), vp]
            lib.gemm_run_host.argtypes = list(lib.gemm_run.argtypes)
            lib.gemm_ring_stats.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint64), i32,
                                            ctypes.POINTER(ctypes.c_int)]
            lib.gemm_sync_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_uint32)]
            lib.gemm_run_noalloc.argtypes = [i64, i64, i64, i64, vp, i64, i32, vp, i64, i32, vp,
                                             vp, vp, vp, f32, f32, f32,
                                             ctypes.POINTER(gemm_dtypes_t), vp,
                                             ctypes.POINTER(ctypes.c_uint32)]
            lib.gemm_status_string.argtypes = [i32]
            lib.gemm_status_string.restype = ctypes.c_char_p
            lib.gemm_check.argtypes = [ctypes.POINTER(gemm_problem_t)]
            lib.gemm_plan.argtypes = [ctypes.POINTER(gemm_problem_t), i32, i32,
                                      ctypes.POINTER(gemm_config_t), ctypes.POINTER(gemm_config_t)]
            lib.gemm_set_config.argtypes = [vp, ctypes.POINTER(gemm_config_t)]
            lib.gemm_last_config.argtypes = [vp, ctypes.POINTER(gemm_config_t)]
            lib.gemm_tmem_columns.argtypes = [i32, i32]
            lib.gemm_set_timeout_ns.argtypes = [vp, ctypes.c_uint64]
            for name in ("gemm_create", "gemm_destroy", "gemm_run", "gemm_run_noalloc",
                         "gemm_sync_status",
                         "gemm_check", "gemm_plan", "gemm_set_config", "gemm_last_config",
                         "gemm_tmem_columns", "gemm_set_timeout_ns"):
                getattr(lib, name).restype = i32
            _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t or None
    return int(t.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return int(s.cuda_stream)


def make_dtypes(ab, c="f32", d="f32", x="f32", y="f32", cdxy_major=GEMM_K_MAJOR, b=None,
                epilogue=GEMM_EPI_LINEAR, acc="f32") -> gemm_dtypes_t:
    """b: B's type when it differs from A's (fp8 pairs); epilogue: GEMM_EPI_*;
    acc: the tensor-core accumulator type, "f32" or "f16"."""
    code = lambda v: DTYPE_CODES[v] if isinstance(v, str) else int(v)
    return gemm_dtypes_t(code(ab), code(c), code(d), code(x), code(y), int(cdxy_major),
                         GEMM_F32 if b is None or b == ab else code(b), int(epilogue), code(acc))


# ------------------------------------------------------------------ C entry points

def gemm_status_string(status: int) -> str:
    return library().gemm_status_string(int(status)).decode()


def gemm_create(device: int = 0) -> int:
    h = ctypes.c_void_p()
    st = library().gemm_create(ctypes.byref(h), int(device))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_create")
    return h.value


def gemm_destroy(handle: int) -> None:
    st = library().gemm_destroy(handle)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_destroy")


def gemm_run(handle, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y,
             alpha, beta, x_factor, dtypes: gemm_dtypes_t, stream=None, check=True) -> int:
    st = library().gemm_run(handle, M, N, K, L, _ptr(A), lda, layoutA, _ptr(B), ldb, layoutB,
                            _ptr(C), _ptr(X), _ptr(D), _ptr(Y), alpha, beta, x_factor,
                            ctypes.byref(dtypes), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_run")
    return st


def gemm_run_host(handle, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y,
                  alpha, beta, x_factor, dtypes: gemm_dtypes_t, stream=None,
                  check=True) -> int:
    """gemm_run on HOST buffers (CPU tensors, pinned for overlap): the library
    copies the inputs in, runs the GEMM and copies D and Y back, all enqueued
    on `stream` (see the C header)."""
    st = library().gemm_run_host(handle, M, N, K, L, _ptr(A), lda, layoutA, _ptr(B), ldb,
                                 layoutB, _ptr(C), _ptr(X), _ptr(D), _ptr(Y), alpha, beta,
                                 x_factor, ctypes.byref(dtypes), _stream(stream))
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_run_host")
    return st


def gemm_run_noalloc(M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y, alpha, beta,
                     x_factor, dtypes: gemm_dtypes_t, stream=None, check=True,
                     watchdog=False) -> tuple[int, int]:
    """gemm_run without a handle and without allocating device memory (the
    watchdog status word lives in a static device array); see the C header.
    watchdog=True makes the call synchronise and report the status word.
    Returns (status, watchdog word)."""
    word = ctypes.c_uint32(0)
    st = library().gemm_run_noalloc(M, N, K, L, _ptr(A), lda, layoutA, _ptr(B), ldb, layoutB,
                                    _ptr(C), _ptr(X), _ptr(D), _ptr(Y), alpha, beta, x_factor,
                                    ctypes.byref(dtypes), _stream(stream),
                                    ctypes.byref(word) if watchdog else None)
    if check and st != GEMM_OK:
        raise GemmError(st, "gemm_run_noalloc")
    return st, word.value


def gemm_sync_status(handle, stream=None) -> tuple[int, int]:
    detail = ctypes.c_uint32(0)
    st = library().gemm_sync_status(handle, _stream(stream), ctypes.byref(detail))
    return st, detail.value


def gemm_check(problem: gemm_problem_t) -> int:
    return library().gemm_check(ctypes.byref(problem))


def gemm_plan(problem: gemm_problem_t, sm_count: int, smem_optin: int,
              forced: gemm_config_t | None = None) -> tuple[int, gemm_config_t]:
    out = gemm_config_t()
    st = library().gemm_plan(ctypes.byref(problem), sm_count, smem_optin,
                             ctypes.byref(forced) if forced is not None else None,
                             ctypes.byref(out))
    return st, out


def gemm_set_config(handle, cfg: gemm_config_t | None) -> None:
    st = library().gemm_set_config(handle, ctypes.byref(cfg) if cfg is not None else None)
    if st != GEMM_OK:
        raise GemmError(st, "gemm_set_config")


def gemm_last_config(handle) -> gemm_config_t:
    out = gemm_config_t()
    st = library().gemm_last_config(handle, ctypes.byref(out))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_last_config")
    return out


def gemm_tmem_columns(tile_m: int, tile_n: int) -> int:
    return library().gemm_tmem_columns(tile_m, tile_n)


def gemm_set_timeout_ns(handle, ns: int) -> None:
    st = library().gemm_set_timeout_ns(handle, int(ns))
    if st != GEMM_OK:
        raise GemmError(st, "gemm_set_timeout_ns")


def make_problem(M, N, K, L, A=None, lda=0, layoutA=GEMM_K_MAJOR, B=None, ldb=0,
                 layoutB=GEMM_K_MAJOR, C=None, X=None, D=None, Y=None, alpha=1.0, beta=0.0,
                 x_factor=0.0, dtypes: gemm_dtypes_t | None = None) -> gemm_problem_t:
    """A gemm_problem_t for the host-only calls (pointers may be plain ints)."""
    return gemm_problem_t(M, N, K, L, _ptr(A), lda, layoutA, _ptr(B), ldb, layoutB, _ptr(C),
                          _ptr(X), _ptr(D), _ptr(Y), alpha, beta, x_factor,
                          dtypes if dtypes is not None else make_dtypes("f16"))


class Gemm:
    """Owns one library handle on `device`."""

    def __init__(self, device: int = 0):
        self.handle = gemm_create(device)

    def close(self):
        if self.handle:
            gemm_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def run(self, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y, alpha, beta,
            x_factor, dtypes, stream=None):
        return gemm_run(self.handle, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y,
                        alpha, beta, x_factor, dtypes, stream)

    def run_host(self, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D, Y, alpha, beta,
                 x_factor, dtypes, stream=None):
        return gemm_run_host(self.handle, M, N, K, L, A, lda, layoutA, B, ldb, layoutB, C, X, D,
                             Y, alpha, beta, x_factor, dtypes, stream)

    def ring_stats(self, stream=None):
        """Per-CTA ring counters of the last launch (statistics build only):
        a list of GEMM_RING_STAT_WORDS-long lists, CTA by CTA."""
        max_ctas = 1024
        buf = (ctypes.c_uint64 * (max_ctas * GEMM_RING_STAT_WORDS))()
        n = ctypes.c_int(0)
        st = library().gemm_ring_stats(self.handle, _stream(stream), buf, max_ctas,
                                       ctypes.byref(n))
        if st != GEMM_OK:
            raise GemmError(st, "gemm_ring_stats")
        w = GEMM_RING_STAT_WORDS
        return [list(buf[i * w:(i + 1) * w]) for i in range(n.value)]

    def sync_status(self, stream=None):
        return gemm_sync_status(self.handle, stream)

    def set_config(self, cfg=None, **fields):
        if cfg is None and fields:
            cfg = gemm_config_t(**fields)
        gemm_set_config(self.handle, cfg)

    def last_config(self):
        return gemm_last_config(self.handle)
