"""The bounds predicates of the checking build (-DATTN_DEBUG), compiled for the
host from the same header the kernels use, against hand-worked cases; and the
build-flags entry point of the normal library."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "bwd_tcgen05_tma_gb300", "csrc")

# Each line: expected result (0/1) and the C++ expression that computes it.
CASES = [
    # innermost coordinate: 16-byte aligned, box inside the row
    (1, "tma_box_ok(0, 64, 128, 2, 0, 4, 0, 128, 1000, false)"),
    (1, "tma_box_ok(64, 64, 128, 2, 3, 4, 0, 128, 1000, false)"),
    (0, "tma_box_ok(4, 64, 128, 2, 0, 4, 0, 128, 1000, false)"),    # 8 bytes: not 16-aligned
    (1, "tma_box_ok(8, 64, 128, 2, 0, 4, 0, 128, 1000, false)"),    # 16 bytes, box ends at 72
    (0, "tma_box_ok(128, 64, 128, 2, 0, 4, 0, 128, 1000, false)"),  # box past the row end
    (0, "tma_box_ok(-8, 64, 128, 2, 0, 4, 0, 128, 1000, false)"),   # negative x
    (1, "tma_box_ok(4, 32, 128, 4, 0, 4, 0, 64, 1000, false)"),     # fp32: 16 bytes
    (0, "tma_box_ok(2, 32, 128, 4, 0, 4, 0, 64, 1000, false)"),     # fp32: 8 bytes
    # middle index
    (0, "tma_box_ok(0, 64, 128, 2, 4, 4, 0, 128, 1000, false)"),
    (0, "tma_box_ok(0, 64, 128, 2, -1, 4, 0, 128, 1000, false)"),
    # rows of a load: one row of the box inside the tensor
    (1, "tma_box_ok(0, 64, 128, 2, 0, 4, -127, 128, 1000, false)"),
    (0, "tma_box_ok(0, 64, 128, 2, 0, 4, -128, 128, 1000, false)"),
    (1, "tma_box_ok(0, 64, 128, 2, 0, 4, 999, 128, 1000, false)"),
    (0, "tma_box_ok(0, 64, 128, 2, 0, 4, 1000, 128, 1000, false)"),
    # rows of a store or a reduce: never negative, start inside
    (0, "tma_box_ok(0, 64, 128, 2, 0, 4, -1, 128, 1000, true)"),
    (1, "tma_box_ok(0, 64, 128, 2, 0, 4, 0, 128, 1000, true)"),
    (1, "tma_box_ok(0, 64, 128, 2, 0, 4, 999, 128, 1000, true)"),
    (0, "tma_box_ok(0, 64, 128, 2, 0, 4, 1000, 128, 1000, true)"),
    # element ranges
    (1, "span_ok(0, 10, 10)"),
    (0, "span_ok(1, 10, 10)"),
    (0, "span_ok(-1, 1, 10)"),
    (1, "span_ok(9, 1, 10)"),
    (0, "span_ok(10, 1, 10)"),
    (1, "span_ok(10, 0, 10)"),
    (0, "span_ok(INT64_MAX - 1, 4, INT64_MAX)"),  # no overflow in the test
    # row-strided ranges with the vector alignment of the store
    (1, "row_span_ok(5, 6, 32, 16, 64, 4096, 32)"),
    (0, "row_span_ok(6, 6, 32, 16, 64, 4096, 32)"),   # row past the end
    (0, "row_span_ok(5, 6, 56, 16, 64, 4096, 32)"),   # past the row's part
    (0, "row_span_ok(5, 6, 32, 16, 64, 4112, 32)"),   # 16-byte address, 32-byte store
    (1, "row_span_ok(5, 6, 32, 16, 64, 4112, 16)"),
    (0, "row_span_ok(-1, 6, 0, 16, 64, 4096, 16)"),
]


def test_bounds_predicates_on_the_host(tmp_path):
    gxx = shutil.which("g++") or shutil.which("c++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    lines = [f'  if ((int)({expr}) != {want}) {{ std::printf("FAIL %d: {expr.replace(chr(34), "")}\\n", {i}); ++bad; }}'
             for i, (want, expr) in enumerate(CASES)]
    src = ("#include <cstdint>\n#include <cstdio>\n#include \"debug_checks.h\"\n"
           "using namespace attn_dbg;\nint main() {\n  int bad = 0;\n" + "\n".join(lines) +
           "\n  std::printf(\"%d failed\\n\", bad);\n  return bad != 0;\n}\n")
    c = tmp_path / "t.cpp"
    c.write_text(src)
    exe = tmp_path / "t"
    subprocess.check_call([gxx, "-std=c++17", "-O1", "-I" + HEADER_DIR, str(c), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout


def test_normal_library_is_not_the_checking_build():
    from bwd_tcgen05_tma_gb300 import attn as A
    from bwd_tcgen05_tma_gb300 import build

    build.build()
    assert A.load_library().attn_build_flags() & A.BUILD_DEVICE_CHECKS == 0
