"""CPU oracle for the skinny BF16 GEMM ``Y[M,N] = X[M,K] . W[N,K]^T``.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``latency_skinny_bf16_gb300``) neither imports it nor shares any
code with it; the two meet only in the seeded input generators of
``skinny_inputs``.

The arithmetic lives in ``skinny_oracle.c`` (plain C, fp64, ascending k) and
follows the definition of the router / projection GEMM on the pages
("[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)", section
"Implementation breakdown" item 1 and the ``_vector_dotprod`` snippet: bf16
inputs widened, multiplied and added into a wide accumulator; "GLM-5.2
Blackwell decode optimizations", "Implementation breakdown" item 3: the bf16
A x B^T decode projections).  This module only compiles the C file with the
host compiler and marshals numpy arrays.

``rmsnorm`` is the RMS norm of the query latent that precedes the q_b
projection (the fused prologue).  ``gemm_f32w`` is the same definition with fp32 weights (the router GEMM
for models that keep fp32 router weights).  It also holds the router
epilogue that consumes the router logits: a
softmax over each token's N logits and its k largest entries
(``router_topk``); the pages print no epilogue, so the oracle takes the
plainest one (see ``skinny_oracle.c``).

Every function here is pinned by ``tests/test_oracle_pins.py`` to results that
do not come from the oracle itself (hand-worked values under
``tests/golden/``, exact rational brute force, one-hot / identity / linearity /
row-independence / zero-padding invariants, and a float64 library matmul).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "skinny_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libskinny_oracle.so")

_lock = threading.Lock()
_lib = None

# -O2 without -ffast-math: IEEE fp64 semantics are part of the oracle's
# definition.  Contraction is switched off so every product is rounded on its
# own (it is exact in fp64 anyway) before the add.
CFLAGS = ["-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(src: str = _SRC, out: str = _LIB_PATH, cc: str = "gcc") -> str:
    """Compile the oracle into a shared library (host compiler, no CUDA)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = [cc, *CFLAGS, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    return os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64 = ctypes.c_int64
    lib.skinny_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.skinny_oracle_bf16_to_f64.restype = ctypes.c_double
    lib.skinny_oracle_gemm.argtypes = [u16p, i64, u16p, i64, f64p, i64, f64p, i64,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.skinny_oracle_gemm.restype = None
    lib.skinny_oracle_gemm_points.argtypes = [u16p, i64, u16p, i64, ctypes.c_int,
                                              i32p, i32p, ctypes.c_int, f64p, f64p]
    lib.skinny_oracle_gemm_points.restype = None
    f32p = ctypes.POINTER(ctypes.c_float)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.skinny_oracle_gemm_f32w.argtypes = [u16p, i64, f32p, i64, f64p, i64, f64p, i64,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.skinny_oracle_gemm_f32w.restype = None
    lib.skinny_oracle_rmsnorm.argtypes = [u16p, i64, u16p, ctypes.c_double, ctypes.c_int, ctypes.c_int, f64p, i64]
    lib.skinny_oracle_rmsnorm.restype = None
    lib.skinny_oracle_router_topk.argtypes = [f32p, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              f64p, i64, i32p, i64, u8p]
    lib.skinny_oracle_router_topk.restype = None
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.

    ``path`` loads a specific build, e.g. a deliberately mutated copy that a
    test compiles to show that the pins catch a planted mistake."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = _bind(ctypes.CDLL(_LIB_PATH))
        return _lib


def _u16(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 bit patterns must be uint16, got {a.dtype}")
    return a


def bf16_to_f64(bits, lib: ctypes.CDLL | None = None) -> float:
    """Exact value of one bf16 bit pattern."""
    return (lib or load()).skinny_oracle_bf16_to_f64(int(bits) & 0xFFFF)


def gemm(X: np.ndarray, W: np.ndarray, M: int, N: int, K: int,
         ldx: int | None = None, ldw: int | None = None,
         Y_init: np.ndarray | None = None, ldy: int | None = None,
         lib: ctypes.CDLL | None = None):
    """fp64 ``Y = X . W^T`` and ``A = |X| . |W|^T`` (elementwise-abs products).

    ``X`` and ``W`` are flat or 2-D uint16 arrays of bf16 bit patterns with row
    strides ``ldx`` / ``ldw`` (elements; default K).  Returns ``(Y, A)`` as
    float64 arrays of shape ``[M, ldy]`` (``ldy`` defaults to N); columns
    ``n >= N`` keep the values of ``Y_init`` (default NaN) so tests can see the
    oracle leave the gaps of a strided output alone.
    """
    lib = lib or load()
    ldx = K if ldx is None else ldx
    ldw = K if ldw is None else ldw
    ldy = N if ldy is None else ldy
    Xf = _u16(X).reshape(-1)
    Wf = _u16(W).reshape(-1)
    if M > 0 and K > 0 and Xf.size < (M - 1) * ldx + K:
        raise ValueError("X buffer too small")
    if N > 0 and K > 0 and Wf.size < (N - 1) * ldw + K:
        raise ValueError("W buffer too small")
    if Y_init is None:
        Y = np.full((max(M, 0), ldy), np.nan, dtype=np.float64)
    else:
        Y = np.array(Y_init, dtype=np.float64).reshape(max(M, 0), ldy).copy()
    A = np.full((max(M, 0), ldy), np.nan, dtype=np.float64)
    if Xf.size == 0:
        Xf = np.zeros(1, np.uint16)
    if Wf.size == 0:
        Wf = np.zeros(1, np.uint16)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.skinny_oracle_gemm(Xf.ctypes.data_as(u16p), ldx, Wf.ctypes.data_as(u16p), ldw,
                           Y.ctypes.data_as(f64p), ldy, A.ctypes.data_as(f64p), ldy,
                           M, N, K)
    return Y, A


def gemm_points(X: np.ndarray, W: np.ndarray, K: int, rows, cols,
                ldx: int | None = None, ldw: int | None = None,
                lib: ctypes.CDLL | None = None):
    """The oracle at sampled output positions ``(rows[i], cols[i])``."""
    lib = lib or load()
    ldx = K if ldx is None else ldx
    ldw = K if ldw is None else ldw
    r = np.ascontiguousarray(rows, dtype=np.int32)
    c = np.ascontiguousarray(cols, dtype=np.int32)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    Xf = _u16(X).reshape(-1)
    Wf = _u16(W).reshape(-1)
    y = np.empty(r.size, np.float64)
    a = np.empty(r.size, np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.skinny_oracle_gemm_points(Xf.ctypes.data_as(u16p), ldx, Wf.ctypes.data_as(u16p), ldw,
                                  K, r.ctypes.data_as(i32p), c.ctypes.data_as(i32p), r.size,
                                  y.ctypes.data_as(f64p), a.ctypes.data_as(f64p))
    return y, a


def gemm_f32w(X: np.ndarray, W: np.ndarray, M: int, N: int, K: int,
              ldx: int | None = None, ldw: int | None = None, lib: ctypes.CDLL | None = None):
    """``Y = X . W^T`` with X bf16 bit patterns ``[M, ldx]`` and W float32
    ``[N, ldw]`` (fp32 router weights); returns ``(Y, A)`` in fp64, A the sum of
    |x * w| per output."""
    lib = lib or load()
    ldx = K if ldx is None else ldx
    ldw = K if ldw is None else ldw
    Xf = _u16(X).reshape(-1)
    Wf = np.ascontiguousarray(W, dtype=np.float32).reshape(-1)
    if M and Xf.size < (M - 1) * ldx + K:
        raise ValueError("X too small")
    if N and Wf.size < (N - 1) * ldw + K:
        raise ValueError("W too small")
    Y = np.zeros((M, N), np.float64)
    A = np.zeros((M, N), np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.skinny_oracle_gemm_f32w(Xf.ctypes.data_as(u16p), ldx, Wf.ctypes.data_as(f32p), ldw,
                                Y.ctypes.data_as(f64p), N, A.ctypes.data_as(f64p), N, M, N, K)
    return Y, A


def rmsnorm(X: np.ndarray, G: np.ndarray, eps: float, M: int, K: int, ldx: int | None = None,
            lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Unrounded fp64 RMS norm ``x * r * g`` of the bf16 rows of X (``[M, ldx]``
    bit patterns) with bf16 gains G ``[K]``; see ``skinny_oracle.c``."""
    lib = lib or load()
    ldx = K if ldx is None else ldx
    Xf = _u16(X).reshape(-1)
    Gf = _u16(G).reshape(-1)
    XN = np.zeros((M, K), np.float64)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    lib.skinny_oracle_rmsnorm(Xf.ctypes.data_as(u16p), ldx, Gf.ctypes.data_as(u16p), float(eps), M, K,
                              XN.ctypes.data_as(f64p), K)
    return XN


def router_topk(logits: np.ndarray, k: int, renormalize: bool = False, lib: ctypes.CDLL | None = None):
    """Softmax over each row of the float32 ``logits [M, N]`` and its ``k``
    largest entries: returns ``(weights [M, k] fp64, ids [M, k] int32)``, ids in
    descending order of the float32 logit, equal logits by ascending index
    (the router epilogue in ``skinny_oracle.c``)."""
    lib = lib or load()
    L = np.ascontiguousarray(logits, dtype=np.float32)
    if L.ndim != 2:
        raise ValueError("logits must be [M, N]")
    M, N = L.shape
    if not 1 <= k <= N:
        raise ValueError("need 1 <= k <= N")
    w = np.empty((M, k), np.float64)
    ids = np.empty((M, k), np.int32)
    scratch = np.empty(N, np.uint8)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.skinny_oracle_router_topk(L.ctypes.data_as(f32p), N, M, N, k, 1 if renormalize else 0,
                                  w.ctypes.data_as(f64p), k, ids.ctypes.data_as(i32p), k,
                                  scratch.ctypes.data_as(u8p))
    return w, ids


SOURCE_PATH = _SRC
