"""Shared helpers for the GPU parity tests: padded device buffers with canaries,
direct C-ABI calls, and the acceptance criteria.

Acceptance (per element, against the binary64 oracle C_ref and
D = sum_k |a_ik b_kj|):
  * FP32 output:  |C - C_ref| <= 1e-5 * D   (and C == 0 exactly where D == 0).
  * BF16 output:  the FP32 result (within 1e-5 * D) is rounded once to bf16,
    which moves it by at most half a bf16 ulp of the FP32 value, so
    |C - C_ref| <= 1e-5 * D + ulp_bf16(|C_ref| + 1e-5 * D) / 2.
  * Integer-exact inputs (every partial sum an integer below 2^24): bitwise.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import deterministic_invariant_gemm_gb300 as dig
import oracle

REL_TOL = 1e-5
F32_CANARY = float("nan")
BF16_CANARY_BITS = 0x7FC5          # a quiet-NaN pattern the kernels never produce


def round_up(x: int, m: int) -> int:
    return ((x + m - 1) // m) * m


def device_matrix(t: torch.Tensor, ld: int, extra_rows: int = 0) -> torch.Tensor:
    """Copy a CPU [rows, cols] tensor into a CUDA buffer [rows + extra_rows, ld]
    whose padding holds a NaN canary; returns the whole buffer."""
    rows, cols = t.shape
    buf = torch.full((rows + extra_rows, ld), float("nan"), dtype=t.dtype, device="cuda")
    buf[:rows, :cols] = t.to("cuda")
    return buf


def output_buffer(M: int, N: int, ldc: int, bf16: bool, extra_rows: int = 3) -> torch.Tensor:
    if bf16:
        buf = torch.full((M + extra_rows, ldc), 0, dtype=torch.int16, device="cuda")
        buf.fill_(BF16_CANARY_BITS)
        return buf.view(torch.bfloat16)
    return torch.full((M + extra_rows, ldc), F32_CANARY, dtype=torch.float32, device="cuda")


def canary_intact(buf: torch.Tensor, M: int, N: int) -> bool:
    """True if nothing outside the [M, N] block of the output buffer was written."""
    if buf.dtype == torch.bfloat16:
        bits = buf.view(torch.int16)
        pad_cols = bits[:M, N:]
        pad_rows = bits[M:, :]
        return bool((pad_cols == BF16_CANARY_BITS).all()) and bool((pad_rows == BF16_CANARY_BITS).all())
    return bool(torch.isnan(buf[:M, N:]).all()) and bool(torch.isnan(buf[M:, :]).all())


def run_gemm(A: torch.Tensor, B: torch.Tensor, M: int, N: int, K: int, split_k: int = 1,
             bf16_out: bool = False, lda: int | None = None, ldb: int | None = None,
             ldc: int | None = None, atomic: bool = False, extra_rows: int = 3):
    """Run one product through the C ABI on padded device buffers.

    A, B: CPU bf16 tensors [M, K], [K, N].  Returns (C [M, N] on the device as a
    view of the padded output buffer, the whole output buffer)."""
    lda = round_up(max(K, 1), 8) if lda is None else lda
    ldb = round_up(max(N, 1), 8) if ldb is None else ldb
    ldc = round_up(max(N, 1), 8 if bf16_out else 4) if ldc is None else ldc
    Ad = device_matrix(A, lda)
    Bd = device_matrix(B, ldb)
    Cbuf = output_buffer(M, N, ldc, bf16_out, extra_rows)
    if atomic:
        dig.bigemm_run_atomic_splitk(Ad, Bd, Cbuf, M, N, K, lda, ldb, ldc, split_k)
    else:
        need = dig.bigemm_workspace_bytes(M, N, K, split_k)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if need else None
        fn = dig.bigemm_run_bf16out if bf16_out else dig.bigemm_run
        fn(Ad, Bd, Cbuf, M, N, K, lda, ldb, ldc, split_k, ws, need)
    torch.cuda.synchronize()
    return Cbuf[:M, :N], Cbuf


def to_f64(C: torch.Tensor) -> np.ndarray:
    return C.float().cpu().double().numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 ulp of |x| (2^(E-7) / 2, E the unbiased exponent, with the
    smallest normal exponent for tiny values)."""
    a = np.abs(x)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7 - 1).astype(np.int64))


def check_tolerance(C: np.ndarray, Cref: np.ndarray, D: np.ndarray, bf16_out: bool, what: str):
    err = np.abs(C - Cref)
    tol = REL_TOL * D
    if bf16_out:
        tol = tol + bf16_half_ulp(np.abs(Cref) + REL_TOL * D)
    bad = ~(err <= tol)          # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        raise AssertionError(
            "%s: %d of %d elements outside tolerance; first at (%d, %d): got %r, oracle %r, "
            "D %r, tol %r" % (what, len(idx), C.size, i, j, C[i, j], Cref[i, j], D[i, j], tol[i, j]))
    # worst relative error, for the log
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(D > 0, err / D, 0.0)
    return float(rel.max()) if rel.size else 0.0


def oracle_rows(A: torch.Tensor, B: torch.Tensor, M: int, N: int, K: int, rows=None):
    return oracle.gemm_rows(A, B, M, N, K, rows=rows)


def sample_rows(M: int, count: int, seed: int = 0) -> list[int]:
    """First and last rows, rows on both sides of every 128-row tile boundary
    (up to a cap), and random rows."""
    rows = {0, M - 1}
    for b in range(128, M, 128):
        if len(rows) >= count // 2:
            break
        rows.update((b - 1, b))
    rng = np.random.default_rng(seed)
    while len(rows) < min(count, M):
        rows.add(int(rng.integers(0, M)))
    return sorted(rows)


def bits_equal(x: torch.Tensor, y: torch.Tensor) -> bool:
    """Bitwise equality of two same-shaped fp32/bf16 tensors (any strides)."""
    if x.shape != y.shape or x.dtype != y.dtype:
        return False
    it = torch.int32 if x.dtype == torch.float32 else torch.int16
    return bool(torch.equal(x.contiguous().view(it), y.contiguous().view(it)))


def log2_ceil(x: int) -> int:
    return int(math.ceil(math.log2(x)))


def expected_launches(M: int, N: int, K: int, split_k: int, fp8: bool = False) -> int:
    """Kernels bigemm_run (or a linear entry point) launches for this shape on
    the current device: 2 on the workspace path (partial + reduction), else 1."""
    path = dig.bigemm_split_path(M, N, K, split_k, fp8)
    assert path >= 0
    return 2 if path == dig.PATH_WORKSPACE else 1
