"""The C ABI without a GPU: the library builds, loads and exports every symbol
include/bigemm.h declares; the host-side helpers (split count, workspace
sizing) follow their documented formulas; and argument checks return their
error codes before anything touches CUDA."""
import os
import re

import pytest

import deterministic_invariant_gemm_gb300 as dig
from deterministic_invariant_gemm_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bigemm.h")

OK, ARG, ALIGN, WS = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return dig.load()


def header_functions():
    text = open(HEADER, encoding="utf-8").read()
    return sorted(set(re.findall(r"BIGEMM_API[^;(]*?\b(bigemm_\w+)\s*\(", text)))


def test_header_declares_what_the_binding_expects():
    assert header_functions() == sorted(dig.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
    # and nothing of the implementation leaks (hidden visibility)
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", dig.library_path()],
                         capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert exported == set(header_functions())


def test_status_strings(lib):
    for code in range(8):
        s = dig.bigemm_status_string(code)
        assert s.startswith(dig.STATUS_NAMES[code])
    assert dig.bigemm_status_string(99) == "BIGEMM_ERR_UNKNOWN"


def test_split_helpers(lib):
    assert dig.bigemm_max_split_k(0) == 1
    assert dig.bigemm_max_split_k(1) == 1
    assert dig.bigemm_max_split_k(64) == 1
    assert dig.bigemm_max_split_k(65) == 2
    assert dig.bigemm_max_split_k(4096) == 64
    # default split: a function of K only
    assert [dig.bigemm_default_split_k(k) for k in (1, 512, 1023, 1024, 2048, 4096, 8192, 65536)] == \
        [1, 1, 1, 2, 4, 8, 16, 16]
    # effective split: ceil(KB / ceil(KB / S))
    assert dig.bigemm_effective_split_k(4096, 8) == 8
    assert dig.bigemm_effective_split_k(4096, 0) == 8
    assert dig.bigemm_effective_split_k(1000, 3) == 3      # KB=16, L=6 -> 6,6,4
    assert dig.bigemm_effective_split_k(64 * 10, 7) == 5   # KB=10, L=2 -> 5 segments
    assert dig.bigemm_effective_split_k(4096, 65) == 0     # beyond KB
    assert dig.bigemm_effective_split_k(4096, -1) == 0
    assert dig.bigemm_effective_split_k(0, 1) == 1
    for K in (1, 63, 64, 65, 1000, 4096, 65536):
        for S in range(1, min(40, dig.bigemm_max_split_k(K)) + 1):
            kb = -(-K // 64)
            L = -(-kb // S)
            assert dig.bigemm_effective_split_k(K, S) == -(-kb // L)


def test_workspace_sizes(lib):
    assert dig.bigemm_workspace_ld(1) == 4
    assert dig.bigemm_workspace_ld(4096) == 4096
    assert dig.bigemm_workspace_ld(4097) == 4100
    assert dig.bigemm_workspace_bytes(64, 4096, 4096, 8) == 8 * 64 * 4096 * 4
    assert dig.bigemm_workspace_bytes(64, 4096, 4096, 1) == 0
    assert dig.bigemm_partial_workspace_bytes(16, 4096, 4096, 1) == 16 * 4096 * 4
    assert dig.bigemm_workspace_bytes(33, 5, 640, 7) == 5 * 33 * 8 * 4
    assert dig.bigemm_workspace_bytes(-1, 5, 640, 2) == 0
    # a few-row product (M <= 32, at most 8 segments) sums its segments
    # inside one launch: no workspace
    assert dig.bigemm_workspace_bytes(16, 4096, 4096, 8) == 0
    assert dig.bigemm_workspace_bytes(3, 5, 640, 7) == 0
    assert dig.bigemm_workspace_bytes(32, 4096, 4096, 8) == 0
    assert dig.bigemm_workspace_bytes(33, 4096, 4096, 8) == 8 * 33 * 4096 * 4
    assert dig.bigemm_workspace_bytes(16, 4096, 8192, 16) == 16 * 16 * 4096 * 4   # 16 segments
    # the 8-bit entry point has no few-row kernel
    assert dig.bigemm_fp8_workspace_bytes(16, 4096, 8192, 8) == 8 * 16 * 4096 * 4


def test_fold_rule_is_a_function_of_the_shape(lib):
    """A split product folds (no workspace) exactly when it has at least
    FOLD_MIN_ROWS rows and FOLD_MIN_TILES tiles of 128 x 256; K and split_k
    matter only through whether the effective split exceeds 1."""
    def tiles(M, N):
        return -(-M // 128) * -(-N // 256)

    for M in (1, 16, 32, 33, 96, 97, 128, 511, 512, 1024, 1025, 4096, 8192):
        for N in (256, 4096, 4100, 6144, 32768, 65536):
            for K, S in ((4096, 8), (4096, 1), (4096, 0), (65536, 16), (640, 7), (64, 4)):
                s = dig.bigemm_effective_split_k(K, S)
                want = s > 1 and M >= dig.FOLD_MIN_ROWS and tiles(M, N) >= dig.FOLD_MIN_TILES
                assert dig.bigemm_split_is_folded(M, N, K, S) == want, (M, N, K, S)
                ws = dig.bigemm_workspace_bytes(M, N, K, S)
                few_rows = 1 <= M <= dig.SKINNY_MAX_ROWS and s <= dig.SKINNY_MAX_SPLIT
                assert ws == (0 if (s <= 1 or want or few_rows) else s * M * dig.bigemm_workspace_ld(N) * 4)
                s8 = dig.bigemm_fp8_effective_split_k(K, S)
                want8 = s8 > 1 and M >= dig.FOLD_MIN_ROWS and tiles(M, N) >= dig.FOLD_MIN_TILES
                ws8 = dig.bigemm_fp8_workspace_bytes(M, N, K, S)
                assert ws8 == (0 if (s8 <= 1 or want8) else s8 * M * dig.bigemm_workspace_ld(N) * 4)
                # the explicit partial kernel always writes slices (0 bytes for
                # an invalid split, e.g. 4 segments of one K block)
                assert dig.bigemm_partial_workspace_bytes(M, N, K, S) == \
                    s * M * dig.bigemm_workspace_ld(N) * 4
    # the decode shapes never fold; a prefill of 1024 rows at N = 4096 does
    assert not dig.bigemm_split_is_folded(64, 4096, 4096, 8)
    assert dig.bigemm_split_is_folded(1024, 4096, 4096, 8)
    assert not dig.bigemm_split_is_folded(1024, 4096, 4096, 1)
    assert not dig.bigemm_split_is_folded(-1, 4096, 4096, 8)


A16 = 1 << 20      # fake, 16-byte aligned addresses: never dereferenced
B16 = 2 << 20
C16 = 3 << 20
W16 = 4 << 20


@pytest.mark.parametrize("args,code", [
    # (A, B, C, M, N, K, lda, ldb, ldc, split_k, ws, ws_bytes)
    ((A16, B16, C16, -1, 8, 8, 8, 8, 8, 1, None, 0), ARG),
    ((A16, B16, C16, 8, 8, -1, 8, 8, 8, 1, None, 0), ARG),
    ((None, B16, C16, 8, 8, 8, 8, 8, 8, 1, None, 0), ARG),
    ((A16, B16, None, 8, 8, 8, 8, 8, 8, 1, None, 0), ARG),
    ((A16, B16, C16, 8, 8, 16, 8, 8, 8, 1, None, 0), ARG),       # lda < K
    ((A16, B16, C16, 8, 16, 8, 8, 8, 16, 1, None, 0), ARG),      # ldb < N
    ((A16, B16, C16, 8, 16, 8, 8, 16, 8, 1, None, 0), ARG),      # ldc < N
    ((A16, B16, C16, 8, 8, 128, 128, 8, 8, 3, None, 0), ARG),    # split > KB
    ((A16, B16, C16, 8, 8, 128, 128, 8, 8, -2, None, 0), ARG),
    ((A16 + 2, B16, C16, 8, 8, 8, 8, 8, 8, 1, None, 0), ALIGN),
    ((A16, B16 + 8, C16, 8, 8, 8, 8, 8, 8, 1, None, 0), ALIGN),
    ((A16, B16, C16 + 4, 8, 8, 8, 8, 8, 8, 1, None, 0), ALIGN),
    ((A16, B16, C16, 8, 8, 12, 12, 8, 8, 1, None, 0), ALIGN),    # lda % 8
    ((A16, B16, C16, 8, 12, 8, 8, 12, 12, 1, None, 0), ALIGN),   # ldb % 8
    ((A16, B16, C16, 8, 8, 8, 8, 8, 10, 1, None, 0), ALIGN),     # ldc % 4
    # (40 rows: past the few-row kernel, which needs no workspace)
    ((A16, B16, C16, 40, 8, 4096, 4096, 8, 8, 8, None, 0), WS),   # no workspace
    ((A16, B16, C16, 40, 8, 4096, 4096, 8, 8, 8, W16, 100), WS),  # too small
    ((A16, B16, C16, 40, 8, 4096, 4096, 8, 8, 8, W16 + 4, 1 << 20), WS),
    ((A16, B16, C16, 0, 8, 8, 8, 8, 8, 1, None, 0), OK),         # empty: nothing enqueued
    ((A16, B16, C16, 8, 0, 8, 8, 8, 8, 1, None, 0), OK),
])
def test_argument_checks_fp32(lib, args, code):
    A, B, C, M, N, K, lda, ldb, ldc, s, ws, wb = args
    assert dig.bigemm_run(A, B, C, M, N, K, lda, ldb, ldc, s, ws, wb, stream=0, check=False) == code


def test_argument_checks_other_entry_points(lib):
    # bf16 output needs ldc % 8 == 0
    assert dig.bigemm_run_bf16out(A16, B16, C16, 8, 8, 8, 8, 8, 12, 1, None, 0, stream=0,
                                  check=False) == ALIGN
    # the partial kernel needs a workspace even for one slice
    assert dig.bigemm_run_partial(A16, B16, 8, 8, 8, 8, 8, 1, None, 0, stream=0,
                                  check=False) == WS
    assert dig.bigemm_splitk_reduce(W16, 0, 8, 8, C16, 8, 0, stream=0, check=False) == ARG
    assert dig.bigemm_splitk_reduce(W16 + 4, 2, 8, 8, C16, 8, 0, stream=0, check=False) == ALIGN
    assert dig.bigemm_splitk_reduce(W16, 2, 8, 8, C16, 4, 0, stream=0, check=False) == ARG
    assert dig.bigemm_splitk_reduce(W16, 2, 0, 8, C16, 8, 0, stream=0, check=False) == OK
    assert dig.bigemm_run_atomic_splitk(A16, B16, C16, 8, 8, 8, 8, 8, 8, 2, stream=0,
                                        check=False) == ARG
    with pytest.raises(dig.BigemmError):
        dig.bigemm_run(A16, B16, C16, -1, 8, 8, 8, 8, 8, 1, None, 0, stream=0)


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle and has no CPU code path."""
    pkg = os.path.join(ROOT, "deterministic_invariant_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f


def test_ozaki_host_helpers_agree_with_the_oracle(lib):
    """rho, the default slice count and the Fast Mode pair count are host
    arithmetic; the oracle's versions are pinned against the pages."""
    import oracle
    for K in (1, 2, 63, 64, 128, 129, 1000, 4096, 8192, 16384, 1 << 20, 1 << 22):
        rho = dig.bigemm_ozaki_rho(K)
        assert rho == oracle.ozaki_rho(K)
        assert dig.bigemm_ozaki_default_slices(K) == oracle.ozaki_default_slices(rho)
    assert dig.bigemm_ozaki_rho(0) == -1 and dig.bigemm_ozaki_rho((1 << 22) + 1) == -1
    for s in range(1, 12):
        for d in range(0, 2 * s + 1):
            assert dig.bigemm_ozaki_pairs(s, d) == oracle.ozaki_pairs(s, d)
    # workspace: slices of A and B in bf16, then the two exponent vectors,
    # one count per 128 x 256 output tile and the abort word, then Fast
    # Mode's 64-bit masses of the rows of A and the columns of B, 256-byte parts
    M, N, K, s = 100, 70, 300, 0
    s = dig.bigemm_ozaki_default_slices(K)
    up = lambda x: (x + 255) // 256 * 256
    masses = lambda M, N: up(M * 8) + up(N * 8)
    want = up(s * M * 304 * 2) + up(s * 320 * 72 * 2) + up(M * 4) + up(N * 4) + up((1 + 1) * 4)
    assert dig.bigemm_ozaki_workspace_bytes(M, N, K, 0) == want + masses(M, N)
    M, N = 1000, 3000              # 8 x 12 tiles
    want = up(s * M * 304 * 2) + up(s * 320 * 3000 * 2) + up(M * 4) + up(N * 4) + up((96 + 1) * 4)
    assert dig.bigemm_ozaki_workspace_bytes(M, N, K, 0) == want + masses(M, N)
    M, N = 1024, 4096              # 8 x 16 tiles: the abort word starts a second 256-byte block
    want = up(s * M * 304 * 2) + up(s * 320 * 4096 * 2) + up(M * 4) + up(N * 4) + up((128 + 1) * 4)
    assert dig.bigemm_ozaki_workspace_bytes(M, N, K, 0) == want + masses(M, N)
