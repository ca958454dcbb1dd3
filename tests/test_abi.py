"""CPU checks of the C ABI and the binding: the library loads without a GPU, exports exactly what
include/dmuon.h declares, rejects bad arguments before touching a device, and its host-side planning
and flop accounting agree with closed forms."""

import ctypes
import os
import re
import subprocess

import pytest

import newton_schulz_momentum_gb300 as dm
from newton_schulz_momentum_gb300 import build as dmbuild
from tests import _pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    dmbuild.build()
    return dm.lib()


def header_functions():
    with open(os.path.join(ROOT, "include", "dmuon.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"DMUON_API\s+[\w\s\*]+?\b(dmuon_\w+)\s*\(", src)))


def test_exports_match_header(L):
    """Both builds -- libdmuon.so and the checked libdmuon_checked.so -- export exactly what dmuon.h declares."""
    declared = header_functions()
    assert declared, "no declarations found in include/dmuon.h"
    assert sorted(dm.EXPORTS) == declared
    for name in declared:
        assert hasattr(L, name), name
    for path in (dmbuild.LIB, dmbuild.CHECKED_LIB):
        out = subprocess.run(["nm", "-D", "--defined-only", path], check=True, capture_output=True, text=True).stdout
        exported = sorted(set(re.findall(r" T (dmuon_\w+)", out)))
        assert exported == declared, path


def test_checked_build_is_marked_and_regular_build_refuses_the_range_selftest(L):
    """The checked build says so in its version string; the regular build has no device-side range checks
    and refuses their self-test before touching a device."""
    checked = ctypes.CDLL(dmbuild.CHECKED_LIB)
    checked.dmuon_version.restype = ctypes.c_char_p
    assert b"range checks" in checked.dmuon_version()
    assert "range checks" not in dm.version()
    L.dmuon_selftest_range_check.argtypes = [ctypes.c_void_p]
    rc, msg = _status(L, L.dmuon_selftest_range_check(None))
    assert rc == dm.ERR_UNSUPPORTED and "range checks" in msg


def test_version(L):
    assert dm.version().startswith("dmuon-gb300")


def test_tables_match_pages():
    g = _pins.golden_coefficients()
    assert dm.POLAR_EXPRESS == g["POLAR_EXPRESS"]
    assert dm.YOU == g["YOU"]


def _status(L, rc):
    return rc, L.dmuon_last_error().decode()


def test_invalid_arguments_rejected_without_device(L):
    c = (ctypes.c_float * 15)(*[1.0] * 15)
    r = (ctypes.c_int * 1)(2)
    rc, msg = _status(L, L.dmuon_ns(None, 4, 8, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "NULL" in msg
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, c, 5, r, 1, 7, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "backend" in msg
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, c, 0, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "steps" in msg
    bad = (ctypes.c_int * 2)(3, 2)
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, c, 5, bad, 2, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "increasing" in msg
    out = (ctypes.c_int * 1)(5)
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, c, 5, out, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "restart" in msg
    rc, msg = _status(L, L.dmuon_ns(4096, 0, 8, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG
    rc, msg = _status(L, L.dmuon_ns(4100, 4, 8, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "aligned" in msg
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, c, 5, r, 1, 1, -1.0, None))
    assert rc == dm.ERR_INVALID_ARG and "eps" in msg
    nan = (ctypes.c_float * 15)(*([float("nan")] + [1.0] * 14))
    rc, msg = _status(L, L.dmuon_ns(4096, 4, 8, nan, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "finite" in msg
    # GEMM building block
    rc, msg = _status(L, L.dmuon_gemm_f16(8, 9, 16, 4096, 16, 4096, 16, 1, None, 0, 4096, 16, 1.0, 0.0, 0.0, 1, None))
    assert rc == dm.ERR_INVALID_ARG and "M == N" in msg
    rc, msg = _status(L, L.dmuon_gemm_f16(8, 8, 16, 4096, 12, 4096, 16, 1, None, 0, 4096, 16, 1.0, 0.0, 0.0, 0, None))
    assert rc == dm.ERR_INVALID_ARG and "leading" in msg
    rc, msg = _status(L, L.dmuon_gemm_f16(8, 8, 16, 4096, 20, 4096, 16, 1, None, 0, 4096, 16, 1.0, 0.0, 0.0, 0, None))
    assert rc == dm.ERR_INVALID_ARG and "multiples of 8" in msg
    # batched step
    P = (ctypes.c_void_p * 1)(4096)
    rows = (ctypes.c_int64 * 1)(4)
    cols = (ctypes.c_int64 * 1)(8)
    rc, msg = _status(L, L.dmuon_muon_step(1, P, P, 3, P, rows, cols, None, 0.02, 0.95, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "grad_dtype" in msg
    rc, msg = _status(L, L.dmuon_muon_step(0, P, P, 0, P, rows, cols, None, 0.02, 0.95, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_INVALID_ARG and "count" in msg
    # host-gradient step: the host array, each host pointer and the group count are checked first
    H = (ctypes.c_void_p * 1)(8192)
    rc, msg = _status(L, L.dmuon_muon_step_host(1, P, None, P, 1, P, rows, cols, None, 0.02, 0.95, c, 5, r, 1, 1,
                                                1e-7, 0, None))
    assert rc == dm.ERR_INVALID_ARG and "grads_host" in msg
    rc, msg = _status(L, L.dmuon_muon_step_host(1, P, (ctypes.c_void_p * 1)(None), P, 1, P, rows, cols, None, 0.02,
                                                0.95, c, 5, r, 1, 1, 1e-7, 0, None))
    assert rc == dm.ERR_INVALID_ARG and "host gradient" in msg
    rc, msg = _status(L, L.dmuon_muon_step_host(1, P, H, P, 1, P, rows, cols, None, 0.02, 0.95, c, 5, r, 1, 1, 1e-7,
                                                65, None))
    assert rc == dm.ERR_INVALID_ARG and "groups" in msg
    rc, msg = _status(L, L.dmuon_muon_step_host(1, P, H, P, 3, P, rows, cols, None, 0.02, 0.95, c, 5, r, 1, 1, 1e-7,
                                                0, None))
    assert rc == dm.ERR_INVALID_ARG and "grad_dtype" in msg
    # failure-detection self-test: the limit is checked before anything touches a device
    for bad in (0, 999999, 2000000001):
        rc, msg = _status(L, L.dmuon_selftest_bounded_wait(bad, None))
        assert rc == dm.ERR_INVALID_ARG and "limit_ns" in msg


def test_flop_counts_closed_form():
    for m, n in ((4096, 4096), (1024, 4096), (4096, 14336), (128, 512), (7, 3)):
        mm, nn = min(m, n), max(m, n)
        assert dm.gram_flops(m, n) == 6 * mm * mm * nn + 17 * mm ** 3
        assert dm.direct_flops(m, n) == 15 * mm * mm * nn + 5 * mm ** 3
    # no restart: X X^T + 5 R^2 + 4 Q updates + 4 R updates (two symmetric products) + output
    assert dm.gram_flops(10, 20, 5, ()) == 100 * 20 + 5 * 1000 + 4 * 2000 + 4 * 2000 + 2 * 100 * 20


def test_workspace_size_closed_form(L):
    # Gram: two fp16 X buffers (m x roundup(n, 8)) and five fp16 m x roundup(m, 8) buffers per matrix,
    # plus small tables. Direct: two X buffers and two m x m buffers.
    shapes = [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)]
    big = sum(2 * 2 * min(s) * max(s) + 5 * 2 * min(s) ** 2 for s in shapes)
    got = dm.workspace_size(shapes, "gram")
    assert big <= got <= big * 1.001 + (1 << 22)
    small = sum(2 * 2 * min(s) * max(s) + 2 * 2 * min(s) ** 2 for s in shapes)
    got = dm.workspace_size(shapes, "direct")
    assert small <= got <= small * 1.001 + (1 << 22)


def test_workspace_size_of_fused_small_plans(L):
    """A call whose every matrix has m <= 128 and n <= 512 runs the fused small-matrix kernel, which keeps
    X, R, Z and Q in shared memory: its workspace is tables only. One larger matrix sends the whole call to
    the grouped path, which needs the per-matrix buffers again."""
    small = [(128, 512)] * 50 + [(512, 128)] * 50
    for backend in ("gram", "direct", "auto"):
        assert dm.workspace_size(small, backend) < 100 * 1024
    mixed = small[:-1] + [(129, 512)]
    gram = sum(2 * 2 * min(s) * (-(-max(s) // 8) * 8) + 5 * 2 * min(s) * (-(-min(s) // 8) * 8) for s in mixed)
    assert gram <= dm.workspace_size(mixed, "gram") <= gram * 1.001 + (1 << 22)


def test_oversized_dimension_rejected(L):
    c = (ctypes.c_float * 15)(*[1.0] * 15)
    r = (ctypes.c_int * 1)(2)
    rc, msg = _status(L, L.dmuon_ns(4096, 1 << 25, 8, c, 5, r, 1, 1, 1e-7, None))
    assert rc == dm.ERR_UNSUPPORTED and "larger than" in msg


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No CPU fallback: without libdmuon.so every call raises."""
    monkeypatch.setattr(dm, "_lib", None)
    monkeypatch.setattr(dm, "LIB_PATH", str(tmp_path / "libdmuon.so"))
    with pytest.raises(dm.LibraryNotBuilt):
        dm.version()
    with pytest.raises(dm.LibraryNotBuilt):
        dm.set_workspace_limit(0)


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>

#include "dmuon.h"

int main(void) {
  float coeffs[15];
  const int restarts[1] = {2};
  const int64_t rows[3] = {14336, 4096, 1024};
  const int64_t cols[3] = {4096, 4096, 4096};
  int owner[3];
  double loads[2];
  size_t bytes = 0;
  int i, rc;
  for (i = 0; i < 15; ++i) coeffs[i] = 1.0f;
  if (strncmp(dmuon_version(), "dmuon-gb300", 11) != 0) return 1;
  rc = dmuon_ns(NULL, 4, 8, coeffs, 5, restarts, 1, DMUON_NS_GRAM, 1e-7f, NULL);
  if (rc != DMUON_ERR_INVALID_ARG || strstr(dmuon_last_error(), "NULL") == NULL) return 2;
  rc = dmuon_assign_owners(3, rows, cols, NULL, 2, DMUON_COST_GRAM_FLOPS, owner, loads);
  if (rc != DMUON_OK) return 3;
  rc = dmuon_workspace_size(3, rows, cols, DMUON_NS_GRAM, &bytes);
  if (rc != DMUON_OK || bytes == 0) return 4;
  printf("%d %d %d %.17g %.17g %zu\n", owner[0], owner[1], owner[2], loads[0], loads[1], bytes);
  return 0;
}
"""


def test_header_serves_a_plain_c_client(L, tmp_path):
    """include/dmuon.h compiles as strict C99 and a C program links libdmuon.so directly: the host-only
    entry points (version, argument validation, owner assignment, workspace query) answer as they do
    through the Python binding."""
    import shutil

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(dm.LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-L", libdir, "-ldmuon", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    shapes = [(14336, 4096), (4096, 4096), (1024, 4096)]
    owners, loads = dm.assign_owners(shapes, 2, None, "gram_flops")
    assert [int(v) for v in out[:3]] == list(owners)
    assert [float(v) for v in out[3:5]] == list(loads)
    assert int(out[5]) == dm.workspace_size(shapes, "gram")


def test_noalloc_arguments_rejected_without_device(L):
    """dmuon_momentum_normalize_noalloc checks every argument before it looks up its scratch or touches a
    device: NULL buffers, misaligned buffers, a bad gradient type, empty or oversized shapes, non-finite
    beta or eps."""
    f = L.dmuon_momentum_normalize_noalloc
    A, B, C = 4096, 8192, 12288  # 16-byte aligned stand-in addresses (never dereferenced)
    cases = [
        ((None, 0, None, 4, 8, B, C, 0.95, 1e-7), "NULL"),
        ((None, 0, A, 4, 8, None, C, 0.95, 1e-7), "NULL"),
        ((None, 0, A, 4, 8, B, None, 0.95, 1e-7), "NULL"),
        ((None, 2, A, 4, 8, B, C, 0.95, 1e-7), "grad_dtype"),
        ((None, 0, A + 4, 4, 8, B, C, 0.95, 1e-7), "aligned"),
        ((None, 0, A, 4, 8, B + 8, C, 0.95, 1e-7), "aligned"),
        ((A + 8, 1, A, 4, 8, B, C, 0.95, 1e-7), "aligned"),
        ((None, 0, A, 4, 8, B, C + 2, 0.95, 1e-7), "aligned"),
        ((None, 0, A, 0, 8, B, C, 0.95, 1e-7), "rows and cols"),
        ((None, 0, A, 4, -1, B, C, 0.95, 1e-7), "rows and cols"),
        ((None, 0, A, 1 << 20, 1 << 9, B, C, 0.95, 1e-7), "DMUON_NOALLOC_MAX_ELEMS"),
        ((None, 0, A, 4, 8, B, C, float("nan"), 1e-7), "beta"),
        ((None, 0, A, 4, 8, B, C, 0.95, float("inf")), "eps"),
        ((None, 0, A, 4, 8, B, C, 0.95, -1e-7), "eps"),
    ]
    for args, word in cases:
        rc, msg = _status(L, f(*args, None))
        assert rc == dm.ERR_INVALID_ARG and word in msg, (args, msg)
