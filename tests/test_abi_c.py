"""The boundary from C: include/mm.h compiles as strict C99 and as C++, and a C program
links against libmm.so and gets the documented status codes from calls that need no GPU.
"""
import os
import shutil
import subprocess

import pytest

from dense_packed_bit_gb300 import build as mmbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "dense_packed_bit_gb300")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mm.h"

#define EXPECT(cond) do { if (!(cond)) { printf("FAILED line %d: %s\n", __LINE__, #cond); return 1; } } while (0)

int main(void) {
    int splitk = -7;
    int64_t floats = -7;
    float cb[4] = {-2.0f, -1.0f, 0.0f, 1.0f};
    const float *fake = (const float *)(uintptr_t)0x10000;  /* never dereferenced: validation fails first */

    EXPECT(mm_version() == 100);
    /* argument checks come back before any CUDA call */
    EXPECT(mm_gemm_f32(0, 0, 0, 8, 8, fake, 8, fake, 8, (float *)(uintptr_t)0x20000, 8, NULL) == MM_ERR_INVALID_ARG);
    EXPECT(strlen(mm_last_error()) > 0);
    EXPECT(mm_gemv_packed2(NULL, NULL, NULL, NULL, 8, 8, cb, NULL) == MM_ERR_INVALID_ARG);
    EXPECT(mm_probe_bounded_wait(2, 10000, NULL, NULL) == MM_ERR_INVALID_ARG);
    /* the host-only split plan: the GPT-2 MLP shape runs unsplit, 64 x 3072 x 768 in 12 slices */
    EXPECT(mm_gemm_f32_split_plan(8192, 3072, 768, 152, &splitk, &floats) == MM_OK);
    EXPECT(splitk == 1 && floats == 0);
    EXPECT(mm_gemm_f32_split_plan(64, 3072, 768, 152, &splitk, &floats) == MM_OK);
    EXPECT(splitk == 12 && floats == (int64_t)12 * 64 * 3072);
    EXPECT(mm_gemm_f32_split_plan(0, 3072, 768, 152, &splitk, &floats) == MM_ERR_INVALID_ARG);
    printf("ok\n");
    return 0;
}
"""


def _need(tool):
    if shutil.which(tool) is None:
        pytest.skip(f"{tool} not installed")


def test_header_compiles_as_strict_c99_and_cxx(tmp_path):
    _need("gcc")
    _need("g++")
    src = tmp_path / "h.c"
    src.write_text('#include "mm.h"\nint mm_header_check(void) { return MM_OK + MM_ACT_GELU_TANH; }\n')
    for cc, std in (("gcc", "-std=c99"), ("g++", "-std=c++17")):
        args = [cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE]
        if cc == "g++":
            args += ["-x", "c++"]
        r = subprocess.run(args + ["-c", str(src), "-o", str(tmp_path / f"h_{cc}.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_program_links_and_gets_status_codes(tmp_path):
    _need("gcc")
    lib = mmbuild.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                        "-L", os.path.dirname(lib), "-l:" + os.path.basename(lib),
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
