"""GB300-native low-latency skinny BF16 GEMM, ``Y[M,N] = X[M,K] . W[N,K]^T``.

bf16 inputs, fp32 accumulation, fp32 (or bf16) output, as used for the MoE
router logits and the small-batch decode projections.  M = 1..16 (decode
sized) runs on every kernel; M = 17..64 runs on the tensor cores only: the
tcgen05 kernel (tensor-memory accumulator, W by tensor-map TMA; any K, 16-byte
aligned rows), the tensor-core dot-product and the cluster split-K kernel's
mma.sync consumer, chosen per shape by the measured tuning table.  The
router's softmax / top-k epilogue, fp32 router weights and the query RMS norm
in front of the q_b projection (a norm kernel chained to the GEMM, or, with
the ``fuse_norm`` option, fused into the tcgen05 GEMM for M <= 16) have entry
points of their own.

This module is a thin ctypes binding over ``libskinny_gemm.so`` (the C ABI in
``include/skinny_gemm.h``): the functions below carry the C names and only
marshal arguments.  Every step of the GEMM runs in the library's sm_103a
kernels; there is no CPU or library fallback, and importing the binding
raises if the compiled library is missing.  PyTorch is used only by the
tensor convenience wrapper :func:`gemm` (device memory and streams).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "SkinnyError", "load_library", "library_path",
    "skinny_gemm_bf16", "skinny_gemm_bf16_bf16out", "skinny_init", "skinny_query_plan", "skinny_plan_for",
    "skinny_set_option", "skinny_get_option", "skinny_get_device_status",
    "skinny_status_string", "skinny_version", "skinny_router_topk", "skinny_router_bf16_topk",
    "skinny_gemm_bf16_f32w", "skinny_plan_for_f32w", "skinny_rmsnorm_gemm_bf16", "gemm", "router_topk",
    "rmsnorm_gemm", "options",
]

# ---- constants mirrored from include/skinny_gemm.h
SKINNY_MAX_M = 64
SKINNY_OK = 0
SKINNY_ERR_INVALID_VALUE = 1
SKINNY_ERR_UNSUPPORTED = 2
SKINNY_ERR_MISALIGNED = 3
SKINNY_ERR_LAUNCH = 4
SKINNY_ERR_DEVICE_TIMEOUT = 5
SKINNY_ERR_NO_DEVICE = 6

SKINNY_BACKEND_AUTO = 0
SKINNY_BACKEND_DOTPROD = 1
SKINNY_BACKEND_SPLITK = 2
SKINNY_BACKEND_STREAM = 3
SKINNY_BACKEND_TCGEN05 = 4
SKINNY_CONSUMER_AUTO = 0
SKINNY_CONSUMER_FMA = 1
SKINNY_CONSUMER_MMA = 2

SKINNY_OPT_PDL = 1
SKINNY_OPT_FORCE_BACKEND = 2
SKINNY_OPT_FORCE_CONSUMER = 3
SKINNY_OPT_FORCE_SPLIT_K = 4
SKINNY_OPT_FORCE_BLOCK_N = 5
SKINNY_OPT_FORCE_STAGES = 6
SKINNY_OPT_WAIT_TIMEOUT_US = 7
SKINNY_OPT_LOG = 8
SKINNY_OPT_FORCE_CLUSTERS = 9
SKINNY_OPT_FORCE_STAGE_K = 10
SKINNY_OPT_FUSE_NORM = 11
SKINNY_OPT_LATE_TRIGGER = 12

EXPORTED_SYMBOLS = (
    "skinny_gemm_bf16", "skinny_gemm_bf16_bf16out", "skinny_init", "skinny_query_plan", "skinny_plan_for",
    "skinny_set_option", "skinny_get_option", "skinny_get_device_status",
    "skinny_status_string", "skinny_version", "skinny_router_topk", "skinny_router_bf16_topk",
    "skinny_gemm_bf16_f32w", "skinny_plan_for_f32w", "skinny_rmsnorm_gemm_bf16",
)


class SkinnyError(RuntimeError):
    """A non-zero skinny_status_t."""

    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {skinny_status_string(status)} ({status})" if what else
                         f"{skinny_status_string(status)} ({status})")


class _Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "backend", "consumer", "vec_elems", "block_n", "split_k", "stages", "stage_k", "k_chunk",
        "grid_x", "grid_y", "threads", "smem_bytes", "pdl", "tuned")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.skinny_gemm_bf16.argtypes = [vp, i, vp, i, vp, i, i, i, i, vp]
    lib.skinny_gemm_bf16.restype = i
    lib.skinny_gemm_bf16_bf16out.argtypes = [vp, i, vp, i, vp, i, i, i, i, vp]
    lib.skinny_gemm_bf16_bf16out.restype = i
    lib.skinny_gemm_bf16_f32w.argtypes = [vp, i, vp, i, vp, i, i, i, i, vp]
    lib.skinny_gemm_bf16_f32w.restype = i
    lib.skinny_plan_for_f32w.argtypes = [vp, i, vp, i, vp, i, i, i, i, i, ctypes.POINTER(_Plan)]
    lib.skinny_plan_for_f32w.restype = i
    lib.skinny_rmsnorm_gemm_bf16.argtypes = [vp, i, vp, ctypes.c_float, vp, i, vp, i, vp, i, i, i, i, vp]
    lib.skinny_rmsnorm_gemm_bf16.restype = i
    lib.skinny_router_topk.argtypes = [vp, i, i, i, i, i, vp, i, vp, i, vp]
    lib.skinny_router_topk.restype = i
    lib.skinny_router_bf16_topk.argtypes = [vp, i, vp, i, vp, i, i, i, i, i, i, vp, i, vp, i, vp]
    lib.skinny_router_bf16_topk.restype = i
    lib.skinny_init.argtypes = [i]
    lib.skinny_init.restype = i
    lib.skinny_query_plan.argtypes = [vp, i, vp, i, vp, i, i, i, i, ctypes.POINTER(_Plan)]
    lib.skinny_query_plan.restype = i
    lib.skinny_plan_for.argtypes = [vp, i, vp, i, vp, i, i, i, i, i, ctypes.POINTER(_Plan)]
    lib.skinny_plan_for.restype = i
    lib.skinny_set_option.argtypes = [i, i]
    lib.skinny_set_option.restype = i
    lib.skinny_get_option.argtypes = [i, ctypes.POINTER(i)]
    lib.skinny_get_option.restype = i
    lib.skinny_get_device_status.argtypes = [vp, ctypes.POINTER(i)]
    lib.skinny_get_device_status.restype = i
    lib.skinny_status_string.argtypes = [i]
    lib.skinny_status_string.restype = ctypes.c_char_p
    lib.skinny_version.argtypes = []
    lib.skinny_version.restype = i
    return lib


def load_library(build_if_missing: bool = False) -> ctypes.CDLL:
    """The loaded ``libskinny_gemm.so``.  Raises if it has not been built
    (``__graft_entry__.build()`` or ``python -m latency_skinny_bf16_gb300._build``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                if not build_if_missing:
                    raise ImportError(f"{path} is missing: build the CUDA library first "
                                      "(python -c 'import __graft_entry__ as g; g.build()')")
                _build.build()
            _lib = _bind(ctypes.CDLL(path))
        return _lib


# ---------------------------------------------------------------- C-named wrappers (raw pointers)

def skinny_gemm_bf16(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                     M: int, N: int, K: int, stream: int = 0) -> int:
    """Raw C call: device pointers as ints; returns the skinny_status_t."""
    return load_library().skinny_gemm_bf16(X, ldx, W, ldw, Y, ldy, M, N, K, stream)


def skinny_gemm_bf16_f32w(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                          M: int, N: int, K: int, stream: int = 0) -> int:
    """Raw C call with fp32 weights (ldw in fp32 elements); returns the skinny_status_t."""
    return load_library().skinny_gemm_bf16_f32w(X, ldx, W, ldw, Y, ldy, M, N, K, stream)


def skinny_plan_for_f32w(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                         M: int, N: int, K: int, num_sms: int) -> dict:
    p = _Plan()
    st = load_library().skinny_plan_for_f32w(X, ldx, W, ldw, Y, ldy, M, N, K, num_sms, ctypes.byref(p))
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_plan_for_f32w")
    return p.as_dict()


def skinny_rmsnorm_gemm_bf16(X: int, ldx: int, gamma: int, eps: float, XN: int, ldxn: int, W: int, ldw: int,
                             Y: int, ldy: int, M: int, N: int, K: int, stream: int = 0) -> int:
    """Raw C call: RMS norm of X into XN, then Y = XN . W^T; returns the skinny_status_t."""
    return load_library().skinny_rmsnorm_gemm_bf16(X, ldx, gamma, float(eps), XN, ldxn, W, ldw, Y, ldy, M, N, K,
                                                   stream)


def skinny_router_topk(L: int, ldl: int, M: int, N: int, k: int, renormalize: int,
                       weights: int, ldw: int, ids: int, ldid: int, stream: int = 0) -> int:
    """Raw C call of the router epilogue (softmax + top-k); returns the skinny_status_t."""
    return load_library().skinny_router_topk(L, ldl, M, N, k, renormalize, weights, ldw, ids, ldid, stream)


def skinny_router_bf16_topk(X: int, ldx: int, W: int, ldw: int, L: int, ldl: int, M: int, N: int, K: int,
                            k: int, renormalize: int, weights: int, ldwt: int, ids: int, ldid: int,
                            stream: int = 0) -> int:
    """Raw C call of the whole router (GEMM into L, then softmax + top-k)."""
    return load_library().skinny_router_bf16_topk(X, ldx, W, ldw, L, ldl, M, N, K, k, renormalize,
                                                  weights, ldwt, ids, ldid, stream)


def skinny_gemm_bf16_bf16out(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                             M: int, N: int, K: int, stream: int = 0) -> int:
    """Raw C call with a bf16 Y (bit patterns); returns the skinny_status_t."""
    return load_library().skinny_gemm_bf16_bf16out(X, ldx, W, ldw, Y, ldy, M, N, K, stream)


def skinny_init(device: int = 0) -> int:
    return load_library().skinny_init(device)


def skinny_query_plan(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                      M: int, N: int, K: int) -> dict:
    p = _Plan()
    st = load_library().skinny_query_plan(X, ldx, W, ldw, Y, ldy, M, N, K, ctypes.byref(p))
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_query_plan")
    return p.as_dict()


def skinny_plan_for(X: int, ldx: int, W: int, ldw: int, Y: int, ldy: int,
                    M: int, N: int, K: int, num_sms: int) -> dict:
    p = _Plan()
    st = load_library().skinny_plan_for(X, ldx, W, ldw, Y, ldy, M, N, K, num_sms, ctypes.byref(p))
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_plan_for")
    return p.as_dict()


def skinny_set_option(option: int, value: int) -> None:
    st = load_library().skinny_set_option(option, int(value))
    if st != SKINNY_OK:
        raise SkinnyError(st, f"skinny_set_option({option}, {value})")


def skinny_get_option(option: int) -> int:
    v = ctypes.c_int(0)
    st = load_library().skinny_get_option(option, ctypes.byref(v))
    if st != SKINNY_OK:
        raise SkinnyError(st, f"skinny_get_option({option})")
    return v.value


def skinny_get_device_status(stream: int = 0) -> int:
    """Synchronise ``stream``, read and clear the device status word."""
    v = ctypes.c_int(0)
    st = load_library().skinny_get_device_status(stream, ctypes.byref(v))
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_get_device_status")
    return v.value


def skinny_status_string(status: int) -> str:
    return load_library().skinny_status_string(int(status)).decode()


def skinny_version() -> int:
    return load_library().skinny_version()


class options:
    """Context manager that sets library options and restores them on exit."""

    def __init__(self, **kw):
        names = {"pdl": SKINNY_OPT_PDL, "backend": SKINNY_OPT_FORCE_BACKEND,
                 "consumer": SKINNY_OPT_FORCE_CONSUMER, "split_k": SKINNY_OPT_FORCE_SPLIT_K,
                 "block_n": SKINNY_OPT_FORCE_BLOCK_N, "stages": SKINNY_OPT_FORCE_STAGES,
                 "wait_timeout_us": SKINNY_OPT_WAIT_TIMEOUT_US, "log": SKINNY_OPT_LOG,
                 "clusters": SKINNY_OPT_FORCE_CLUSTERS, "stage_k": SKINNY_OPT_FORCE_STAGE_K,
                 "fuse_norm": SKINNY_OPT_FUSE_NORM, "late_trigger": SKINNY_OPT_LATE_TRIGGER}
        self._set = [(names[k], int(v)) for k, v in kw.items()]
        self._old = []

    def __enter__(self):
        for opt, v in self._set:
            self._old.append((opt, skinny_get_option(opt)))
            skinny_set_option(opt, v)
        return self

    def __exit__(self, *exc):
        for opt, v in reversed(self._old):
            skinny_set_option(opt, v)
        self._old.clear()
        return False


# ---------------------------------------------------------------- tensor convenience

def gemm(x, w, out=None, stream=None):
    """``out[:M, :N] = x . w^T`` for CUDA tensors: x bf16 [M, K], w bf16 [N, K]
    (unit stride along K), out fp32 or bf16 [M, N] (any row stride >= N, unit
    column stride; bf16 is the fp32 result rounded to nearest-even).  Runs on ``stream`` (default: torch's current stream)."""
    import torch
    if x.dtype != torch.bfloat16 or w.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("x must be bfloat16 and w bfloat16 or float32")
    if x.dim() != 2 or w.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, w {tuple(w.shape)}")
    if not (x.is_cuda and w.is_cuda):
        raise ValueError("x and w must be CUDA tensors")
    M, K = x.shape
    N = w.shape[0]
    if (K > 1 and (x.stride(1) != 1 or w.stride(1) != 1)):
        raise ValueError("x and w need unit stride along K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if out.dtype not in (torch.float32, torch.bfloat16) or out.dim() != 2 or tuple(out.shape) != (M, N):
        raise ValueError("out must be fp32 or bf16 [M, N]")
    if N > 1 and out.stride(1) != 1:
        raise ValueError("out needs unit column stride")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ldx = x.stride(0) if M > 1 else max(K, 1)
    ldw = w.stride(0) if N > 1 else max(K, 1)
    ldy = out.stride(0) if M > 1 else max(N, 1)
    if w.dtype == torch.float32:
        if out.dtype != torch.float32:
            raise TypeError("fp32 weights give an fp32 output")
        call = skinny_gemm_bf16_f32w
    else:
        call = skinny_gemm_bf16 if out.dtype == torch.float32 else skinny_gemm_bf16_bf16out
    st = call(x.data_ptr(), ldx, w.data_ptr(), ldw, out.data_ptr(), ldy, M, N, K, s)
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_gemm_bf16")
    return out


def router_topk(logits, k, renormalize=False, weights=None, ids=None, stream=None):
    """Softmax over each row of the CUDA fp32 ``logits [M, N]`` (unit column
    stride) and its ``k`` largest entries: returns ``(weights fp32 [M, k],
    ids int32 [M, k])``; see ``skinny_router_topk`` in include/skinny_gemm.h."""
    import torch
    if logits.dtype != torch.float32 or logits.dim() != 2 or not logits.is_cuda:
        raise ValueError("logits must be a CUDA fp32 [M, N] tensor")
    M, N = logits.shape
    if N > 1 and logits.stride(1) != 1:
        raise ValueError("logits need unit column stride")
    if weights is None:
        weights = torch.empty((M, k), dtype=torch.float32, device=logits.device)
    if ids is None:
        ids = torch.empty((M, k), dtype=torch.int32, device=logits.device)
    if stream is None:
        stream = torch.cuda.current_stream(logits.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    ldl = logits.stride(0) if M > 1 else max(N, 1)
    st = skinny_router_topk(logits.data_ptr(), ldl, M, N, k, 1 if renormalize else 0,
                            weights.data_ptr(), weights.stride(0) if M > 1 else max(k, 1),
                            ids.data_ptr(), ids.stride(0) if M > 1 else max(k, 1), s)
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_router_topk")
    return weights, ids


def rmsnorm_gemm(x, gamma, eps, w, out=None, xn=None, stream=None):
    """``xn = bf16(rmsnorm(x) * gamma)`` and ``out = xn . w^T`` for CUDA bf16
    tensors x [M, K], gamma [K], w [N, K] (unit stride along K); returns
    ``(out fp32 [M, N], xn bf16 [M, K])``; see ``skinny_rmsnorm_gemm_bf16``."""
    import torch
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or gamma.dtype != torch.bfloat16:
        raise TypeError("x, gamma and w must be bfloat16")
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    if xn is None:
        xn = torch.empty((M, K), dtype=torch.bfloat16, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = skinny_rmsnorm_gemm_bf16(x.data_ptr(), x.stride(0) if M > 1 else max(K, 1), gamma.data_ptr(), eps,
                                  xn.data_ptr(), xn.stride(0) if M > 1 else max(K, 1),
                                  w.data_ptr(), w.stride(0) if N > 1 else max(K, 1),
                                  out.data_ptr(), out.stride(0) if M > 1 else max(N, 1), M, N, K, s)
    if st != SKINNY_OK:
        raise SkinnyError(st, "skinny_rmsnorm_gemm_bf16")
    return out, xn
