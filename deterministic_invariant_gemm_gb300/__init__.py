"""Deterministic, batch-invariant BF16 GEMM for NVIDIA GB300 (sm_103a).

A thin ctypes binding over ``libbigemm.so`` (declared in ``include/bigemm.h``).
Every computation runs in that library's CUDA kernels; this module only turns
torch tensors (or raw integers) into pointers, sizes and a stream handle, and
uses torch to allocate outputs and workspaces.  There is no fallback: if the
library is missing or the device is not sm_103, calls raise.

The operation is C = A * B with A [M, K] and B [K, N] in bf16 and FP32
accumulation; row i of C is bit-for-bit a function of (row i of A, B, K,
split_k, output dtype) only -- independent of M, of the rest of the batch and
of the run (Tencent AI-infra article "腾讯エンジニア：大規模モデルの出力を確定
させるための AI インフラ手法", sections "Batch Invariance の由来" and "Split-K").

Low-level functions keep the C names and argument order::

    bigemm_run(A, B, C, M, N, K, lda, ldb, ldc, split_k, workspace, workspace_bytes, stream)

where the pointer arguments accept a torch tensor, an integer address or None
and ``stream`` accepts a ``torch.cuda.Stream``, an integer handle or None (the
current torch stream).  :func:`matmul` is the convenience wrapper.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH, build as build_library  # noqa: F401

__all__ = [
    "BigemmError", "load", "library_path", "BLOCK_K", "TILE_M", "TILE_N",
    "bigemm_version", "bigemm_status_string", "bigemm_max_split_k",
    "bigemm_default_split_k", "bigemm_effective_split_k", "bigemm_workspace_ld",
    "bigemm_workspace_bytes", "bigemm_partial_workspace_bytes", "bigemm_run",
    "bigemm_run_bf16out", "bigemm_run_partial", "bigemm_splitk_reduce",
    "bigemm_run_atomic_splitk", "bigemm_device_status", "bigemm_last_launch_count",
    "bigemm_run_splitk_static", "bigemm_linear", "bigemm_fp8_effective_split_k",
    "bigemm_fp8_workspace_bytes", "bigemm_linear_fp8", "bigemm_split_is_folded", "bigemm_split_path", "bigemm_tile_n",
    "bigemm_cluster_capacity", "bigemm_ozaki_rho", "bigemm_ozaki_default_slices",
    "bigemm_ozaki_pairs", "bigemm_ozaki_workspace_bytes", "bigemm_ozaki_split", "bigemm_ozaki_dgemm",
    "ozaki_matmul", "bigemm_selftest_timeout", "bigemm_selftest_ozaki_order_timeout", "PATH_UNSPLIT", "PATH_WORKSPACE", "PATH_FOLDED", "PATH_CLUSTER", "PATH_SKINNY", "FP8_E4M3",
    "FP8_E5M2", "FOLD_MIN_ROWS", "FOLD_MIN_TILES", "SKINNY_MAX_ROWS", "SKINNY_MAX_SPLIT",
    "STATIC_SCRATCH_BYTES", "matmul", "linear", "linear_fp8", "EXPORTED_SYMBOLS",
]

BLOCK_K = 64
TILE_M = 128
TILE_N = 256

STATUS_NAMES = {
    0: "BIGEMM_OK", 1: "BIGEMM_ERR_ARG", 2: "BIGEMM_ERR_ALIGN", 3: "BIGEMM_ERR_WORKSPACE",
    4: "BIGEMM_ERR_UNSUPPORTED", 5: "BIGEMM_ERR_CUDA", 6: "BIGEMM_ERR_TIMEOUT",
    7: "BIGEMM_ERR_STATIC_LIMIT",
}

STATIC_SCRATCH_BYTES = 16 << 20

# a split product with at least this many rows and output tiles sums its
# segments inside the CTA (no workspace); see bigemm_split_is_folded
FOLD_MIN_ROWS = 97
FOLD_MIN_TILES = 128

# a bf16 product of at most this many rows and at most this many K segments
# runs the few-row kernel, which sums its segments in one launch (no
# workspace); see bigemm_split_path (PATH_SKINNY)
SKINNY_MAX_ROWS = 32
SKINNY_MAX_SPLIT = 8

EXPORTED_SYMBOLS = (
    "bigemm_version", "bigemm_status_string", "bigemm_max_split_k", "bigemm_default_split_k",
    "bigemm_effective_split_k", "bigemm_workspace_ld", "bigemm_workspace_bytes",
    "bigemm_partial_workspace_bytes", "bigemm_run", "bigemm_run_bf16out", "bigemm_run_partial",
    "bigemm_splitk_reduce", "bigemm_run_atomic_splitk", "bigemm_device_status",
    "bigemm_last_launch_count", "bigemm_run_splitk_static", "bigemm_linear",
    "bigemm_fp8_effective_split_k", "bigemm_fp8_workspace_bytes", "bigemm_linear_fp8",
    "bigemm_split_is_folded", "bigemm_split_path", "bigemm_tile_n", "bigemm_cluster_capacity",
    "bigemm_uses_pair", "bigemm_set_pair_mode", "bigemm_pair_capacity",
    "bigemm_fp8_kn_workspace_bytes", "bigemm_run_fp8",
    "bigemm_ozaki_rho", "bigemm_ozaki_default_slices", "bigemm_ozaki_pairs",
    "bigemm_ozaki_workspace_bytes", "bigemm_ozaki_split", "bigemm_ozaki_dgemm",
    "bigemm_selftest_timeout", "bigemm_selftest_ozaki_order_timeout",
)

FP8_E4M3 = 0
FP8_E5M2 = 1


class BigemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__("%s: %s" % (where, bigemm_status_string(status)))


_lib = None


def library_path() -> str:
    return LIB_PATH


def load():
    """Load libbigemm.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libbigemm.so is not built; run `python -m deterministic_invariant_gemm_gb300.build` "
            "(needs nvcc) -- there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    i64, vp, i32, sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "bigemm_version": ([], i32),
        "bigemm_status_string": ([i32], ctypes.c_char_p),
        "bigemm_max_split_k": ([i64], i32),
        "bigemm_default_split_k": ([i64], i32),
        "bigemm_effective_split_k": ([i64, i32], i32),
        "bigemm_workspace_ld": ([i64], i64),
        "bigemm_workspace_bytes": ([i64, i64, i64, i32], sz),
        "bigemm_split_is_folded": ([i64, i64, i64, i32], i32),
        "bigemm_split_path": ([i64, i64, i64, i32, i32], i32),
        "bigemm_tile_n": ([i64, i64, i64, i32, i32], i32),
        "bigemm_cluster_capacity": ([i32], i32),
        "bigemm_uses_pair": ([i64, i64, i64, i32, i32], i32),
        "bigemm_set_pair_mode": ([i32], i32),
        "bigemm_pair_capacity": ([], i32),
        "bigemm_fp8_kn_workspace_bytes": ([i64, i64, i64, i32], sz),
        "bigemm_run_fp8": ([vp, vp, i32, i32, ctypes.c_float, vp, vp, i64, i64, i64, i64, i64,
                            i64, i32, i32, vp, sz, vp], i32),
        "bigemm_ozaki_rho": ([i64], i32),
        "bigemm_selftest_timeout": ([vp], i32),
        "bigemm_selftest_ozaki_order_timeout": ([vp], i32),
        "bigemm_ozaki_default_slices": ([i64], i32),
        "bigemm_ozaki_pairs": ([i32, i32], i64),
        "bigemm_ozaki_workspace_bytes": ([i64, i64, i64, i32], sz),
        "bigemm_ozaki_split": ([vp, i64, i64, i64, i32, i32, i32, vp, i64, i64, vp, vp], i32),
        "bigemm_ozaki_dgemm": ([vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, i32, vp, sz, vp], i32),
        "bigemm_partial_workspace_bytes": ([i64, i64, i64, i32], sz),
        "bigemm_run": ([vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, vp, sz, vp], i32),
        "bigemm_run_bf16out": ([vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, vp, sz, vp], i32),
        "bigemm_run_partial": ([vp, vp, i64, i64, i64, i64, i64, i32, vp, sz, vp], i32),
        "bigemm_splitk_reduce": ([vp, i32, i64, i64, vp, i64, i32, vp], i32),
        "bigemm_run_atomic_splitk": ([vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, vp], i32),
        "bigemm_device_status": ([i32], i32),
        "bigemm_run_splitk_static": ([vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, vp], i32),
        "bigemm_linear": ([vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, i32, i32, vp, sz, vp], i32),
        "bigemm_fp8_effective_split_k": ([i64, i32], i32),
        "bigemm_fp8_workspace_bytes": ([i64, i64, i64, i32], sz),
        "bigemm_linear_fp8": ([vp, vp, i32, i32, ctypes.c_float, vp, vp, i64, i64, i64, i64, i64,
                               i64, i32, i32, vp, sz, vp], i32),
        "bigemm_last_launch_count": ([], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


# ------------------------------------------------------------ marshalling --

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    raise TypeError("expected a tensor, an integer address or None, got %r" % type(x))


def _current_raw_stream() -> int:
    """torch's current CUDA stream on the current device, as a cudaStream_t.
    The raw accessor costs about 0.1 us per call against about 3 us for
    torch.cuda.current_stream(), which builds a Stream object; the public
    call stays as the fallback."""
    import torch
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return int(raw(torch.cuda.current_device()))
    return int(torch.cuda.current_stream().cuda_stream)


def _stream(s) -> int | None:
    if s is None:
        return _current_raw_stream()
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    raise TypeError("expected a torch.cuda.Stream, an integer handle or None")


def _check(status: int, where: str) -> None:
    if status != 0:
        raise BigemmError(status, where)


# ------------------------------------------------------ C functions, same names --

def bigemm_version() -> int:
    return int(load().bigemm_version())


def bigemm_status_string(status: int) -> str:
    if _lib is None and not os.path.exists(LIB_PATH):
        return STATUS_NAMES.get(int(status), "BIGEMM_ERR_UNKNOWN")
    return load().bigemm_status_string(int(status)).decode()


def bigemm_max_split_k(K: int) -> int:
    return int(load().bigemm_max_split_k(K))


def bigemm_default_split_k(K: int) -> int:
    return int(load().bigemm_default_split_k(K))


def bigemm_effective_split_k(K: int, split_k: int) -> int:
    return int(load().bigemm_effective_split_k(K, split_k))


def bigemm_workspace_ld(N: int) -> int:
    return int(load().bigemm_workspace_ld(N))


def bigemm_workspace_bytes(M: int, N: int, K: int, split_k: int) -> int:
    return int(load().bigemm_workspace_bytes(M, N, K, split_k))


def bigemm_split_is_folded(M: int, N: int, K: int, split_k: int) -> bool:
    return bool(load().bigemm_split_is_folded(M, N, K, split_k))


PATH_UNSPLIT, PATH_WORKSPACE, PATH_FOLDED, PATH_CLUSTER, PATH_SKINNY = 0, 1, 2, 3, 4


def bigemm_cluster_capacity(splits: int) -> int:
    return int(load().bigemm_cluster_capacity(splits))


def bigemm_split_path(M: int, N: int, K: int, split_k: int, fp8: bool = False) -> int:
    """How a direct-output product of this shape runs on the current device:
    PATH_UNSPLIT, PATH_WORKSPACE, PATH_FOLDED, PATH_CLUSTER or PATH_SKINNY
    (-1: invalid)."""
    return int(load().bigemm_split_path(M, N, K, split_k, 1 if fp8 else 0))


def bigemm_uses_pair(M: int, N: int, K: int, split_k: int, fp8: bool = False) -> int:
    """1 when a product of this shape runs the 2-SM kernel (256 x 256 tiles
    on CTA pairs), 0 when single CTAs (-1: invalid)."""
    return int(load().bigemm_uses_pair(M, N, K, split_k, 1 if fp8 else 0))


PAIR_NEVER, PAIR_AUTO, PAIR_ALWAYS = 0, 1, 2


def bigemm_set_pair_mode(mode: int) -> int:
    """When the 2-SM kernel runs for later products: PAIR_NEVER, PAIR_AUTO
    (the default rule) or PAIR_ALWAYS (every shape it serves); returns the
    previous mode."""
    prev = int(load().bigemm_set_pair_mode(int(mode)))
    if prev < 0:
        raise ValueError("pair mode must be 0, 1 or 2")
    return prev


def bigemm_pair_capacity() -> int:
    return int(load().bigemm_pair_capacity())


def bigemm_tile_n(M: int, N: int, K: int, split_k: int, fp8: bool = False) -> int:
    """Output-tile width (256, 128 or 64 columns) a product of this shape runs
    with on the current device (-1: invalid)."""
    return int(load().bigemm_tile_n(M, N, K, split_k, 1 if fp8 else 0))


def bigemm_partial_workspace_bytes(M: int, N: int, K: int, split_k: int) -> int:
    return int(load().bigemm_partial_workspace_bytes(M, N, K, split_k))


def bigemm_run(A, B, C, M, N, K, lda, ldb, ldc, split_k, workspace=None, workspace_bytes=0,
               stream=None, check=True) -> int:
    st = load().bigemm_run(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, split_k,
                           _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_run")
    return st


def bigemm_linear(A, W, bias, C, M, N, K, lda, ldw, ldc, split_k, c_is_bf16, workspace=None,
                  workspace_bytes=0, stream=None, check=True) -> int:
    st = load().bigemm_linear(_ptr(A), _ptr(W), _ptr(bias), _ptr(C), M, N, K, lda, ldw, ldc,
                              split_k, int(bool(c_is_bf16)), _ptr(workspace), workspace_bytes,
                              _stream(stream))
    if check:
        _check(st, "bigemm_linear")
    return st


def bigemm_fp8_effective_split_k(K: int, split_k: int) -> int:
    return int(load().bigemm_fp8_effective_split_k(K, split_k))


def bigemm_fp8_workspace_bytes(M: int, N: int, K: int, split_k: int) -> int:
    return int(load().bigemm_fp8_workspace_bytes(M, N, K, split_k))


def bigemm_linear_fp8(A, W, fmt_a, fmt_w, scale, bias, C, M, N, K, lda, ldw, ldc, split_k,
                      c_is_bf16, workspace=None, workspace_bytes=0, stream=None, check=True) -> int:
    st = load().bigemm_linear_fp8(_ptr(A), _ptr(W), fmt_a, fmt_w, float(scale), _ptr(bias), _ptr(C),
                                  M, N, K, lda, ldw, ldc, split_k, int(bool(c_is_bf16)),
                                  _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_linear_fp8")
    return st


def bigemm_run_bf16out(A, B, C, M, N, K, lda, ldb, ldc, split_k, workspace=None,
                       workspace_bytes=0, stream=None, check=True) -> int:
    st = load().bigemm_run_bf16out(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, split_k,
                                   _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_run_bf16out")
    return st


def bigemm_run_partial(A, B, M, N, K, lda, ldb, split_k, workspace, workspace_bytes,
                       stream=None, check=True) -> int:
    st = load().bigemm_run_partial(_ptr(A), _ptr(B), M, N, K, lda, ldb, split_k,
                                   _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_run_partial")
    return st


def bigemm_splitk_reduce(workspace, splits, M, N, C, ldc, c_is_bf16, stream=None,
                         check=True) -> int:
    st = load().bigemm_splitk_reduce(_ptr(workspace), splits, M, N, _ptr(C), ldc,
                                     int(bool(c_is_bf16)), _stream(stream))
    if check:
        _check(st, "bigemm_splitk_reduce")
    return st


def bigemm_run_atomic_splitk(A, B, C, M, N, K, lda, ldb, ldc, split_k, stream=None,
                             check=True) -> int:
    st = load().bigemm_run_atomic_splitk(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc,
                                         split_k, _stream(stream))
    if check:
        _check(st, "bigemm_run_atomic_splitk")
    return st


def bigemm_run_splitk_static(A, B, C, M, N, K, lda, ldb, ldc, split_k, stream=None,
                             check=True) -> int:
    """bigemm_run without a workspace argument and without any allocation: the
    split-K partials go to the library's built-in 16 MiB device array.  For
    callers that may not allocate device memory per call; calls that can
    overlap on the GPU share that array and must be ordered."""
    st = load().bigemm_run_splitk_static(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc,
                                         split_k, _stream(stream))
    if check:
        _check(st, "bigemm_run_splitk_static")
    return st


def bigemm_device_status(reset: bool = True) -> int:
    return int(load().bigemm_device_status(int(bool(reset))))


def bigemm_last_launch_count() -> int:
    return int(load().bigemm_last_launch_count())


# ----------------------------------------------------------- convenience --

def matmul(A, B, out_dtype=None, split_k: int = 1, out=None, workspace=None, stream=None,
           atomic: bool = False):
    """C = A @ B for bf16 CUDA tensors A [M, K] and B [K, N] (row-major, unit
    column stride; leading dimensions may be padded).  ``out_dtype`` is
    torch.float32 (default) or torch.bfloat16.  ``split_k``: 1 = none, 0 = the
    K-only default, S > 1 = S segments added in a fixed order (through a
    workspace, allocated here with torch when one is needed and not given, or
    inside the CTA or a cluster; see bigemm_split_path).  ``atomic=True`` runs
    the nondeterministic atomic-add contrast instead (fp32 only)."""
    import torch
    if A.dtype != torch.bfloat16 or B.dtype != torch.bfloat16:
        raise TypeError("A and B must be bfloat16")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shapes do not compose: %s x %s" % (tuple(A.shape), tuple(B.shape)))
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B need unit column stride (row-major)")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=A.device)
    if out.dtype != out_dtype or out.stride(1) != 1 or tuple(out.shape) != (M, N):
        raise ValueError("bad output tensor")
    lda = A.stride(0) if M > 1 else max(K, 8 * ((K + 7) // 8))
    ldb = B.stride(0) if K > 1 else max(N, 8 * ((N + 7) // 8))
    ldc = out.stride(0) if M > 1 else max(N, 8 * ((N + 7) // 8))
    if lda % 8 or ldb % 8 or ldc % (8 if out_dtype == torch.bfloat16 else 4):
        raise ValueError(
            "row strides must be multiples of 8 elements for A and B (16-byte rows for the "
            "tensor memory accelerator) and of %d for C; got lda=%d ldb=%d ldc=%d -- store the "
            "matrices with padded rows" % (8 if out_dtype == torch.bfloat16 else 4, lda, ldb, ldc))
    if atomic:
        if out_dtype != torch.float32:
            raise ValueError("the atomic contrast writes fp32")
        bigemm_run_atomic_splitk(A, B, out, M, N, K, lda, ldb, ldc, split_k, stream)
        return out
    # (an unsplit product never needs a workspace: skip the query)
    need = 0 if split_k == 1 else bigemm_workspace_bytes(M, N, K, split_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if out_dtype == torch.float32:
        bigemm_run(A, B, out, M, N, K, lda, ldb, ldc, split_k, workspace, wbytes, stream)
    elif out_dtype == torch.bfloat16:
        bigemm_run_bf16out(A, B, out, M, N, K, lda, ldb, ldc, split_k, workspace, wbytes, stream)
    else:
        raise TypeError("out_dtype must be float32 or bfloat16")
    return out


def linear(x, weight, bias=None, out_dtype=None, split_k: int = 1, out=None, workspace=None,
           stream=None):
    """y = x @ weight.T + bias for bf16 CUDA tensors x [M, K], weight [N, K] and
    bias [N] (or None), through bigemm_linear.  ``out_dtype`` float32 (default)
    or bfloat16; ``split_k`` as in :func:`matmul`."""
    import torch
    if x.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("x and weight must be bfloat16")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.dim() != 1 or bias.stride(0) != 1):
        raise TypeError("bias must be a contiguous bfloat16 vector")
    if x.dim() != 2 or weight.dim() != 2 or x.shape[1] != weight.shape[1]:
        raise ValueError("shapes do not compose: %s x %s^T" % (tuple(x.shape), tuple(weight.shape)))
    if x.stride(1) != 1 or weight.stride(1) != 1:
        raise ValueError("x and weight need unit column stride (row-major)")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    M, K = x.shape
    N = weight.shape[0]
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias has %d entries, weight has %d rows" % (bias.shape[0], N))
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    lda = x.stride(0) if M > 1 else max(K, 8 * ((K + 7) // 8))
    ldw = weight.stride(0) if N > 1 else max(K, 8 * ((K + 7) // 8))
    ldc = out.stride(0) if M > 1 else max(N, 8 * ((N + 7) // 8))
    bf16 = out_dtype == torch.bfloat16
    if lda % 8 or ldw % 8 or ldc % (8 if bf16 else 4):
        raise ValueError("row strides must be multiples of 8 elements for x and weight and of %d "
                         "for the output; got %d, %d, %d" % (8 if bf16 else 4, lda, ldw, ldc))
    need = 0 if split_k == 1 else bigemm_workspace_bytes(M, N, K, split_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    bigemm_linear(x, weight, bias, out, M, N, K, lda, ldw, ldc, split_k, bf16, workspace, wbytes,
                  stream)
    return out


def linear_fp8(x, weight, scale=1.0, bias=None, out_dtype=None, split_k: int = 1, out=None,
               workspace=None, stream=None):
    """y = scale * (x @ weight.T) + bias for 8-bit float CUDA tensors x [M, K] and
    weight [N, K] (torch.float8_e4m3fn or torch.float8_e5m2, each), through
    bigemm_linear_fp8.  bias: bf16 [N] or None; output float32 (default) or
    bfloat16."""
    import torch
    fmts = {torch.float8_e4m3fn: FP8_E4M3, torch.float8_e5m2: FP8_E5M2}
    if x.dtype not in fmts or weight.dtype not in fmts:
        raise TypeError("x and weight must be float8_e4m3fn or float8_e5m2")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.dim() != 1 or bias.stride(0) != 1):
        raise TypeError("bias must be a contiguous bfloat16 vector")
    if x.dim() != 2 or weight.dim() != 2 or x.shape[1] != weight.shape[1]:
        raise ValueError("shapes do not compose: %s x %s^T" % (tuple(x.shape), tuple(weight.shape)))
    if x.stride(1) != 1 or weight.stride(1) != 1:
        raise ValueError("x and weight need unit column stride (row-major)")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    M, K = x.shape
    N = weight.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=x.device)
    lda = x.stride(0) if M > 1 else max(K, 16 * ((K + 15) // 16))
    ldw = weight.stride(0) if N > 1 else max(K, 16 * ((K + 15) // 16))
    ldc = out.stride(0) if M > 1 else max(N, 8 * ((N + 7) // 8))
    bf16 = out_dtype == torch.bfloat16
    if lda % 16 or ldw % 16 or ldc % (8 if bf16 else 4):
        raise ValueError("row strides must be multiples of 16 bytes for x and weight and of %d "
                         "elements for the output; got %d, %d, %d" % (8 if bf16 else 4, lda, ldw, ldc))
    need = 0 if split_k == 1 else bigemm_fp8_workspace_bytes(M, N, K, split_k)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    bigemm_linear_fp8(x, weight, fmts[x.dtype], fmts[weight.dtype], scale, bias, out, M, N, K, lda,
                      ldw, ldc, split_k, bf16, workspace, wbytes, stream)
    return out


def bigemm_fp8_kn_workspace_bytes(M: int, N: int, K: int, split_k: int) -> int:
    return int(load().bigemm_fp8_kn_workspace_bytes(M, N, K, split_k))


def bigemm_run_fp8(A, B, fmt_a, fmt_b, scale, bias, C, M, N, K, lda, ldb, ldc, split_k, c_is_bf16,
                   workspace=None, workspace_bytes=0, stream=None, check=True) -> int:
    st = load().bigemm_run_fp8(_ptr(A), _ptr(B), int(fmt_a), int(fmt_b), float(scale), _ptr(bias),
                               _ptr(C), M, N, K, lda, ldb, ldc, split_k, int(bool(c_is_bf16)),
                               _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_run_fp8")
    return st


def matmul_fp8(a, b, scale=1.0, bias=None, out_dtype=None, split_k: int = 1, out=None,
               workspace=None, stream=None):
    """y = scale * (a @ b) + bias for 8-bit float CUDA tensors a [M, K] and b
    [K, N] (torch.float8_e4m3fn or torch.float8_e5m2, each), through
    bigemm_run_fp8 (b is copied transposed into the workspace, then the
    product is bigemm_linear_fp8's with weight = b^T: the same bits)."""
    import torch
    fmts = {torch.float8_e4m3fn: FP8_E4M3, torch.float8_e5m2: FP8_E5M2}
    if a.dtype not in fmts or b.dtype not in fmts:
        raise TypeError("a and b must be float8_e4m3fn or float8_e5m2")
    if bias is not None and (bias.dtype != torch.bfloat16 or bias.dim() != 1 or bias.stride(0) != 1):
        raise TypeError("bias must be a contiguous bfloat16 vector")
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("shapes do not compose: %s x %s" % (tuple(a.shape), tuple(b.shape)))
    if a.stride(1) != 1 or b.stride(1) != 1:
        raise ValueError("a and b need unit column stride (row-major)")
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    M, K = a.shape
    N = b.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=a.device)
    lda = a.stride(0) if M > 1 else max(K, 16 * ((K + 15) // 16))
    ldb = b.stride(0) if K > 1 else max(N, 16 * ((N + 15) // 16))
    ldc = out.stride(0) if M > 1 else max(N, 8 * ((N + 7) // 8))
    bf16 = out_dtype == torch.bfloat16
    if lda % 16 or ldb % 16 or ldc % (8 if bf16 else 4):
        raise ValueError("row strides must be multiples of 16 bytes for a and b and of %d "
                         "elements for the output; got %d, %d, %d" % (8 if bf16 else 4, lda, ldb, ldc))
    need = bigemm_fp8_kn_workspace_bytes(M, N, K, split_k)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=a.device)
    wbytes = workspace.numel() * workspace.element_size()
    bigemm_run_fp8(a, b, fmts[a.dtype], fmts[b.dtype], scale, bias, out, M, N, K, lda, ldb, ldc,
                   split_k, bf16, workspace, wbytes, stream)
    return out


# ---------------------------------------------------------------- Ozaki --

def bigemm_selftest_timeout(stream=None, check=True) -> int:
    st = load().bigemm_selftest_timeout(_stream(stream))
    if check:
        _check(st, "bigemm_selftest_timeout")
    return st


def bigemm_selftest_ozaki_order_timeout(stream=None, check=True) -> int:
    st = load().bigemm_selftest_ozaki_order_timeout(_stream(stream))
    if check:
        _check(st, "bigemm_selftest_ozaki_order_timeout")
    return st


def bigemm_ozaki_rho(K: int) -> int:
    return int(load().bigemm_ozaki_rho(K))


def bigemm_ozaki_default_slices(K: int) -> int:
    return int(load().bigemm_ozaki_default_slices(K))


def bigemm_ozaki_pairs(slices: int, d: int) -> int:
    return int(load().bigemm_ozaki_pairs(slices, d))


def bigemm_ozaki_workspace_bytes(M: int, N: int, K: int, slices: int = 0) -> int:
    return int(load().bigemm_ozaki_workspace_bytes(M, N, K, slices))


def bigemm_ozaki_split(X, rows, cols, ld, axis, rho, slices, out, out_ld, out_rows, exps,
                       stream=None, check=True) -> int:
    st = load().bigemm_ozaki_split(_ptr(X), rows, cols, ld, axis, rho, slices, _ptr(out), out_ld,
                                   out_rows, _ptr(exps), _stream(stream))
    if check:
        _check(st, "bigemm_ozaki_split")
    return st


def bigemm_ozaki_dgemm(A, B, C, M, N, K, lda, ldb, ldc, slices=0, d=0, workspace=None,
                       workspace_bytes=0, stream=None, check=True) -> int:
    st = load().bigemm_ozaki_dgemm(_ptr(A), _ptr(B), _ptr(C), M, N, K, lda, ldb, ldc, slices, d,
                                   _ptr(workspace), workspace_bytes, _stream(stream))
    if check:
        _check(st, "bigemm_ozaki_dgemm")
    return st


def ozaki_matmul(A, B, slices: int = 0, d: int = 0, out=None, workspace=None, stream=None):
    """C = A @ B for float64 CUDA tensors A [M, K] and B [K, N] (row-major), by
    the Ozaki scheme on the bf16 tensor cores (bigemm_ozaki_dgemm).  slices /
    d: 0 for the defaults (binary64 accuracy); d = -1 for Fast Mode's
    automatic d, chosen per element.  Returns C float64 [M, N]."""
    import torch
    if A.dtype != torch.float64 or B.dtype != torch.float64:
        raise TypeError("A and B must be float64")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError("shapes do not compose: %s x %s" % (tuple(A.shape), tuple(B.shape)))
    if A.stride(1) != 1 or B.stride(1) != 1:
        raise ValueError("A and B need unit column stride (row-major)")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N + (N & 1)), dtype=torch.float64, device=A.device)[:, :N]
    ldc = out.stride(0) if M > 1 else N + (N & 1)
    if ldc % 2:
        raise ValueError("the output's row stride must be even (16-byte vector stores)")
    need = bigemm_ozaki_workspace_bytes(M, N, K, slices)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=A.device)
    wbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lda = A.stride(0) if M > 1 else max(K, 1)
    ldb = B.stride(0) if K > 1 else max(N, 1)
    bigemm_ozaki_dgemm(A, B, out, M, N, K, lda, ldb, ldc, slices, d, workspace, wbytes, stream)
    return out
