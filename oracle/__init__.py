"""CPU oracle for the deterministic, batch-invariant BF16 GEMM.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product path (``deterministic_invariant_gemm_gb300``) never imports it and
shares no code with it; the two meet only on inputs drawn from ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C, binary64); this module compiles
it with gcc on first use and wraps it with ctypes.  Every function states the
passage of the pages it follows in ``oracle.c``'s header:

* :func:`gemm_rows` -- C_ij = sum_k A_ik B_kj in binary64, k ascending, plus
  D_ij = sum_k |A_ik B_kj| (Tencent AI-infra article, "Batch Invariance の由来").
* :func:`decode` / :func:`encode_rne` -- IEEE-754 binary16 / bfloat16 codecs
  with round-to-nearest-even (same article, "背景": 2048 + 1 in FP16).
* :func:`ulp` -- ULP(x) = 2^(E - M) (same section).
* :func:`splitk_reduce_f32` -- the split-K workspace reduction in serial order
  (same article, "Split-K").
* :func:`decode8` / :func:`linear8_rows` -- 8-bit float (E5M2, E4M3) codecs and
  an 8-bit linear layer (the FP8 matmul of the cuTile article's benchmark,
  techplay.jp "TileGymで行列積ベンチマーク").
* :func:`linear_rows` -- a linear layer, C = A W^T + b (same article, "vLLM に
  おける GEMM の Batch Invariance サポート": linear_batch_invariant(x, weight,
  bias)).
* :func:`ozaki_rho`, :func:`ozaki_split`, :func:`ozaki_pairs`,
  :func:`ozaki_gemm`, :func:`ozaki_fast_d` -- the Ozaki scheme's binary64
  product from bfloat16 slices (cuTile article, "倍精度行列積エミュレーション":
  the Veltkamp split of eqs. (1)-(5), the slice-pair products of eqs.
  (10)-(11), Fast Mode's d, fixed or chosen per element).

Pins (tests/test_oracle.py) tie each function to something other than itself:
identity and permutation products, small-integer products checked against
exact integer arithmetic, brute force with exact rationals, the FP16 worked
example, exhaustive codec round trips and hand-computed binary32 sums.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FMT_FP16 = 0
FMT_BF16 = 1
FMT_E5M2 = 2
FMT_E4M3 = 3

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, OpenMP when present)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle: no C compiler (gcc) on PATH")
    base = [cc, "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared"]
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    try:
        last = None
        for extra in (["-fopenmp"], []):
            r = subprocess.run(base + extra + ["-o", tmp, _SRC, "-lm"],
                               capture_output=True, text=True)
            if r.returncode == 0:
                os.replace(tmp, _LIB)   # atomic: concurrent builders are safe
                return _LIB
            last = r.stderr
        raise RuntimeError("oracle: gcc failed:\n" + (last or ""))
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    i64, u32, dbl = ctypes.c_int64, ctypes.c_uint32, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_decode.argtypes = [ctypes.c_int, u32]
    lib.oracle_decode.restype = dbl
    lib.oracle_encode_rne.argtypes = [ctypes.c_int, dbl]
    lib.oracle_encode_rne.restype = u32
    lib.oracle_ulp.argtypes = [ctypes.c_int, dbl]
    lib.oracle_ulp.restype = dbl
    lib.oracle_gemm_rows.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, i64, vp, vp]
    lib.oracle_gemm_rows.restype = ctypes.c_int
    lib.oracle_linear8_rows.argtypes = [vp, vp, ctypes.c_int, ctypes.c_int, i64, i64, i64, i64, i64,
                                        vp, i64, vp, vp]
    lib.oracle_linear8_rows.restype = ctypes.c_int
    lib.oracle_splitk_reduce_f32.argtypes = [vp, i64, i64, vp]
    lib.oracle_splitk_reduce_f32.restype = ctypes.c_int
    lib.oracle_decode_array.argtypes = [ctypes.c_int, vp, i64, vp]
    lib.oracle_decode_array.restype = None
    lib.oracle_encode_rne_array.argtypes = [ctypes.c_int, vp, i64, vp]
    lib.oracle_encode_rne_array.restype = None
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_ozaki_rho.argtypes = [i64]
    lib.oracle_ozaki_rho.restype = ctypes.c_int
    lib.oracle_ozaki_pairs.argtypes = [ctypes.c_int, ctypes.c_int]
    lib.oracle_ozaki_pairs.restype = i64
    lib.oracle_ozaki_split.argtypes = [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       vp, vp, vp]
    lib.oracle_ozaki_split.restype = ctypes.c_int
    lib.oracle_ozaki_gemm.argtypes = [vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, vp, i64, vp]
    lib.oracle_ozaki_gemm.restype = ctypes.c_int
    lib.oracle_ozaki_fast_d.argtypes = [vp, vp, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                        vp, vp, vp]
    lib.oracle_ozaki_fast_d.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _bits16(x) -> np.ndarray:
    """Accept a numpy uint16/int16 array or a torch bf16/fp16 tensor (CPU)."""
    if hasattr(x, "detach"):                     # torch tensor
        import torch
        t = x.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle: inputs must live in host memory")
        if t.dtype in (torch.bfloat16, torch.float16):
            t = t.view(torch.int16)
        x = t.contiguous().numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle: expected 16-bit patterns, got %s" % a.dtype)
    return a


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def decode(fmt: int, bits) -> np.ndarray:
    b = _bits16(np.asarray(bits, dtype=np.uint16) if not hasattr(bits, "detach") else bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_decode_array(fmt, _ptr(b), b.size, _ptr(out))
    return out


def encode_rne(fmt: int, x) -> np.ndarray:
    v = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_encode_rne_array(fmt, _ptr(v), v.size, _ptr(out))
    return out


def ulp(fmt: int, x: float) -> float:
    return float(_load().oracle_ulp(fmt, float(x)))


def fp16_add(a: float, b: float) -> float:
    """a + b rounded once to binary16 (a, b themselves first rounded to binary16)."""
    qa = decode(FMT_FP16, encode_rne(FMT_FP16, [a]))[0]
    qb = decode(FMT_FP16, encode_rne(FMT_FP16, [b]))[0]
    return float(decode(FMT_FP16, encode_rne(FMT_FP16, [qa + qb]))[0])


def gemm_rows(A, B, M: int, N: int, K: int, lda: int | None = None,
              ldb: int | None = None, rows=None):
    """(C, D) for the selected rows of A (all rows when ``rows`` is None).

    A: bf16 patterns [M, lda]; B: bf16 patterns [K, ldb].  Returns binary64
    arrays C, D of shape [len(rows), N].
    """
    a = _bits16(A).reshape(-1)
    b = _bits16(B).reshape(-1)
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    if rows is None:
        r = None
        nrows = M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.size
    C = np.empty((nrows, N), dtype=np.float64)
    D = np.empty((nrows, N), dtype=np.float64)
    rc = _load().oracle_gemm_rows(_ptr(a), _ptr(b), M, N, K, lda, ldb,
                                  None if r is None else _ptr(r), nrows,
                                  _ptr(C), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_gemm_rows: bad arguments")
    return C, D


def linear_rows(A, W, bias, M: int, N: int, K: int, rows=None):
    """(C, D) of a linear layer for the selected rows of A:
    C_ij = sum_k A_ik W_jk + b_j (binary64; the K terms k-ascending, then b_j),
    D_ij = sum_k |A_ik W_jk| + |b_j|, the scale of all the terms summed.
    W: bf16 patterns [N, K]; bias: bf16 patterns [N] or None.  W^T is formed
    by moving the 16-bit patterns (exact) and the product is gemm_rows'."""
    w = _bits16(W).reshape(N, K)
    wt = np.ascontiguousarray(w.T)
    C, D = gemm_rows(A, wt, M, N, K, rows=rows)
    if bias is not None:
        b = decode(FMT_BF16, _bits16(bias).reshape(N))
        C = C + b[None, :]
        D = D + np.abs(b)[None, :]
    return C, D


def _bits8(x) -> np.ndarray:
    """Accept a numpy uint8/int8 array or a torch 8-bit float / uint8 tensor (CPU)."""
    if hasattr(x, "detach"):
        import torch
        t = x.detach()
        if t.device.type != "cpu":
            raise ValueError("oracle: inputs must live in host memory")
        if t.element_size() != 1:
            raise TypeError("oracle: expected 8-bit patterns")
        x = t.contiguous().view(torch.uint8).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.int8:
        a = a.view(np.uint8)
    if a.dtype != np.uint8:
        raise TypeError("oracle: expected 8-bit patterns, got %s" % a.dtype)
    return a


def decode8(fmt: int, bits) -> np.ndarray:
    """Values of 8-bit float patterns (FMT_E5M2 / FMT_E4M3)."""
    b = _bits8(np.asarray(bits, dtype=np.uint8) if not hasattr(bits, "detach") else bits)
    lib = _load()
    return np.array([lib.oracle_decode(fmt, int(v)) for v in b.reshape(-1)],
                    dtype=np.float64).reshape(b.shape)


def linear8_rows(A, W, fmt_a: int, fmt_b: int, M: int, N: int, K: int, scale: float = 1.0,
                 bias=None, rows=None):
    """(C, D) of an 8-bit float linear layer for the selected rows of A:
    C_ij = scale * sum_k A_ik W_jk + b_j   (binary64, k ascending, then the
    scale, then the bias), D_ij = |scale| * sum_k |A_ik W_jk| + |b_j|.
    A: [M, K] bytes, W: [N, K] bytes (weight layout), bias: bf16 [N] or None."""
    a = _bits8(A).reshape(M, K)
    w = _bits8(W).reshape(N, K)
    if rows is None:
        r, nrows = None, M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = r.size
    C = np.empty((nrows, N), dtype=np.float64)
    D = np.empty((nrows, N), dtype=np.float64)
    rc = _load().oracle_linear8_rows(_ptr(a), _ptr(w), fmt_a, fmt_b, M, N, K, K, K,
                                     None if r is None else _ptr(r), nrows, _ptr(C), _ptr(D))
    if rc != 0:
        raise ValueError("oracle_linear8_rows: bad arguments")
    C = C * scale
    D = D * abs(scale)
    if bias is not None:
        b = decode(FMT_BF16, _bits16(bias).reshape(N))
        C = C + b[None, :]
        D = D + np.abs(b)[None, :]
    return C, D


def splitk_reduce_f32(W: np.ndarray) -> np.ndarray:
    """Serial binary32 reduction over the leading axis of W ([S, ...])."""
    w = np.ascontiguousarray(W, dtype=np.float32)
    S = w.shape[0]
    count = w.size // S
    out = np.empty(w.shape[1:], dtype=np.float32)
    rc = _load().oracle_splitk_reduce_f32(_ptr(w), S, count, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_splitk_reduce_f32: bad arguments")
    return out


def bf16_round(x) -> np.ndarray:
    """Round binary64 values to bfloat16 (ties to even); returns binary64 values."""
    return decode(FMT_BF16, encode_rne(FMT_BF16, x))


# --------------------------------------------------------------- Ozaki --

OZ_M1, OZ_M2, OZ_M3 = 53, 8, 24      # binary64, bfloat16, binary32 significand bits


def ozaki_rho(k: int) -> int:
    """rho = max(ceil(m1 - (m3 - log2 k) / 2), m1 - m2) for inner length k."""
    return int(_load().oracle_ozaki_rho(int(k)))


def ozaki_default_slices(rho: int) -> int:
    """Slices whose bits reach 2^-53 below a vector's maximum: with beta =
    m1 - rho bits in the first slice and beta + 1 in each later one,
    s (beta + 1) - 1 >= m1."""
    beta = OZ_M1 - rho
    return -(-(OZ_M1 + 1) // (beta + 1))


def ozaki_pairs(slices: int, d: int) -> int:
    """Slice pairs (p, q) kept by Fast Mode: 0 <= p, q < slices, p + q < d."""
    return int(_load().oracle_ozaki_pairs(int(slices), int(d)))


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def ozaki_split(X, axis: int, rho: int, slices: int):
    """Split the rows (axis 0) or columns (axis 1) of X into bfloat16 slices.
    Returns (S [slices, rows, cols] float64 slice values, c1 int32 per vector,
    R [rows, cols] the residual after the last slice)."""
    x = _f64(X)
    rows, cols = x.shape
    S = np.empty((slices, rows, cols), dtype=np.float64)
    c1 = np.empty(rows if axis == 0 else cols, dtype=np.int32)
    R = np.empty((rows, cols), dtype=np.float64)
    st = _load().oracle_ozaki_split(_ptr(x), rows, cols, cols, axis, rho, slices, _ptr(S), _ptr(c1),
                                    _ptr(R))
    if st != 0:
        raise ValueError("oracle_ozaki_split failed")
    return S, c1, R


def ozaki_fast_d(A, B, rho: int | None = None, slices: int | None = None):
    """Fast Mode's automatic d for every element of A B (cuTile article,
    "Fast Mode（GEMMの削減）"; the per-element reading in oracle.c): returns
    (D [M, N] int32, T_a [M] and T_b [N] uint64, the vectors' integer masses
    sum_k floor(|x_k| 2^(40 - c^(1))))."""
    a, b = _f64(A), _f64(B)
    M, K = a.shape
    N = b.shape[1]
    rho = ozaki_rho(max(K, 1)) if rho is None else rho
    slices = ozaki_default_slices(rho) if slices is None else slices
    D = np.empty((M, N), dtype=np.int32)
    Ta = np.empty(M, dtype=np.uint64)
    Tb = np.empty(N, dtype=np.uint64)
    st = _load().oracle_ozaki_fast_d(_ptr(a), _ptr(b), M, N, K, K, N, rho, slices, _ptr(D), _ptr(Ta),
                                     _ptr(Tb))
    if st != 0:
        raise ValueError("oracle_ozaki_fast_d failed")
    return D, Ta, Tb


def ozaki_gemm(A, B, rho: int | None = None, slices: int | None = None, d: int | None = None):
    """C = A B (binary64) by the Ozaki scheme; returns (C, inexact) where
    inexact counts slice-pair sums that a binary32 accumulation could round
    (0 when rho fits K).  d = -1: Fast Mode's automatic d per element
    (ozaki_fast_d)."""
    a, b = _f64(A), _f64(B)
    M, K = a.shape
    K2, N = b.shape
    assert K == K2
    rho = ozaki_rho(max(K, 1)) if rho is None else rho
    slices = ozaki_default_slices(rho) if slices is None else slices
    d = slices if d is None else d
    C = np.empty((M, N), dtype=np.float64)
    bad = np.zeros(1, dtype=np.int64)
    st = _load().oracle_ozaki_gemm(_ptr(a), _ptr(b), M, N, K, K, N, rho, slices, d, _ptr(C), N,
                                   _ptr(bad))
    if st != 0:
        raise ValueError("oracle_ozaki_gemm failed")
    return C, int(bad[0])
