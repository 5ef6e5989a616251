"""Helpers for the GPU parity tests: device buffers (allocated by torch), the
raw C-ABI call, and the comparison against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import latency_skinny_bf16_gb300 as sk
import oracle
import skinny_inputs as si

CANARY = -7777.0          # written into the gaps of a strided Y; must survive every call
RTOL = 1e-5               # |y - y_ref| <= RTOL * sum_k |x*w| + ATOL  (elementwise)
ATOL = 1e-6
COS_MIN = 0.99999


def dev_bits(flat_u16: np.ndarray, extra: int = 0) -> torch.Tensor:
    """uint16 bit patterns -> CUDA int16 tensor (with `extra` spare elements)."""
    t = torch.zeros(flat_u16.size + extra + 8, dtype=torch.int16)
    t[: flat_u16.size] = torch.from_numpy(flat_u16.view(np.int16).copy())
    return t.cuda()


class Buffers:
    """X, W and Y of one case on the device, with optional strides / offsets."""

    def __init__(self, case: si.Case, X: np.ndarray, W: np.ndarray, ldx=None, ldw=None, ldy=None,
                 w_offset: int = 0, x_offset: int = 0):
        self.M, self.N, self.K = case.M, case.N, case.K
        self.ldx = ldx or case.lx
        self.ldw = ldw or case.lw
        self.ldy = ldy or case.ly
        xs = si.embed_rows(X, self.ldx) if self.M else np.zeros(1, np.uint16)
        ws = si.embed_rows(W, self.ldw) if self.N else np.zeros(1, np.uint16)
        self.x_dev = dev_bits(np.concatenate([np.zeros(x_offset, np.uint16), xs]))
        self.w_dev = dev_bits(np.concatenate([np.zeros(w_offset, np.uint16), ws]))
        self.x_ptr = self.x_dev.data_ptr() + 2 * x_offset
        self.w_ptr = self.w_dev.data_ptr() + 2 * w_offset
        self.y_dev = torch.full((max(self.M, 1) * self.ldy + 64,), CANARY, dtype=torch.float32, device="cuda")
        self.y_ptr = self.y_dev.data_ptr()

    def run(self, stream: int = 0) -> int:
        return sk.skinny_gemm_bf16(self.x_ptr, self.ldx, self.w_ptr, self.ldw, self.y_ptr, self.ldy,
                                   self.M, self.N, self.K, stream)

    def y(self) -> np.ndarray:
        torch.cuda.synchronize()
        return self.y_dev.cpu().numpy()

    def y_mat(self) -> np.ndarray:
        return self.y()[: self.M * self.ldy].reshape(self.M, self.ldy)[:, : self.N]

    def canary_ok(self) -> bool:
        y = self.y()
        body = y[: self.M * self.ldy].reshape(self.M, self.ldy)
        return bool(np.all(body[:, self.N:] == CANARY) and np.all(y[self.M * self.ldy:] == CANARY))

    def plan(self) -> dict:
        return sk.skinny_query_plan(self.x_ptr, self.ldx, self.w_ptr, self.ldw, self.y_ptr, self.ldy,
                                    self.M, self.N, self.K)


def reference(case: si.Case, X: np.ndarray, W: np.ndarray):
    return oracle.gemm(X, W, case.M, case.N, case.K)


def check_parity(y: np.ndarray, yref: np.ndarray, A: np.ndarray, what: str = "") -> float:
    """Elementwise tolerance and cosine similarity; returns max |err| / (A + eps)."""
    y64 = y.astype(np.float64)
    finite = np.isfinite(yref)
    assert np.array_equal(np.isfinite(y64), finite), f"{what}: non-finite pattern differs"
    err = np.abs(y64[finite] - yref[finite])
    bound = RTOL * A[finite] + ATOL
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements out of tolerance, worst err {err[bad].max():.3e} "
                           f"vs bound {bound[bad][np.argmax(err[bad])]:.3e}")
    a, b = y64[finite].ravel(), yref[finite].ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na > 0 and nb > 0:
        cos = float(a @ b / (na * nb))
        assert cos >= COS_MIN, f"{what}: cosine {cos}"
    return float(np.max(err / (A[finite] + 1e-30))) if err.size else 0.0


def run_and_check(case: si.Case, **buf_kw) -> Buffers:
    X, W = si.make_inputs(case)
    b = Buffers(case, X, W, **buf_kw)
    st = b.run()
    assert st == sk.SKINNY_OK, f"{case.name}: {sk.skinny_status_string(st)}"
    yref, A = reference(case, X, W)
    check_parity(b.y_mat(), yref, A, case.name)
    assert b.canary_ok(), f"{case.name}: wrote outside Y[:M, :N]"
    return b
