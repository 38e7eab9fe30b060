"""The boundary as a C program sees it (CPU only): include/gemm.h compiles as
strict C99, a C program that takes the address of every declared function
links against libgemm.so with nothing left unresolved, and the calls that need
no GPU behave as documented when made from C."""
import os
import re
import shutil
import subprocess

import pytest

from dense_gemm_tcgen05_gb300 import build, capi

pytestmark = pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    yield


C_MAIN = r"""
#include <stdio.h>
#include <string.h>
#include "gemm.h"

/* every declared function, by address: the link fails if one is missing */
static void* const fns[] = { %(fns)s };

int main(void) {
    int64_t out[GEMM_PLAN_FIELDS];
    int64_t tm = -1, tn = -1;
    if (sizeof(fns) / sizeof(fns[0]) != %(count)d) return 10;
    /* argument checks run before any CUDA call */
    if (gemm_bf16_tn(-1, 4, 4, 0, 4, 0, 4, 0, 4, NULL) != GEMM_ERR_INVALID_DIM) return 11;
    if (gemm_f32(4, 5, 6, (const float*)0x10000, 5, (const float*)0x10000, 5,
                 (float*)0x10000, 5, NULL) != GEMM_ERR_INVALID_LD) return 12;
    if (gemm_set_option("no such option", 1) != GEMM_ERR_INVALID_OPTION) return 13;
    if (strcmp(gemm_status_string(GEMM_OK), "ok") != 0) return 14;
    /* host-only queries */
    if (gemm_tile_coord(2, 3, 2, 2, 0, &tm, &tn) != GEMM_OK || tm != 0 || tn != 1) return 15;
    if (gemm_tn_plan(GEMM_PLAN_F16, 8192, 8192, 8192,
                     GEMM_PLAN_A_TMA | GEMM_PLAN_B_TMA | GEMM_PLAN_C_TMA | GEMM_PLAN_A_128 |
                     GEMM_PLAN_B_128, 0, 152, out, GEMM_PLAN_FIELDS) != GEMM_OK) return 16;
    if (out[0] != GEMM_OK || out[1] != 1 || out[3] != 256) return 17;
    if (gemm_workspace_bytes(0, 1, 1) != 0) return 18;
    printf("ok\n");
    return 0;
}
"""


def test_header_is_c99_and_links(tmp_path):
    names = capi.declared_symbols()
    src = tmp_path / "main.c"
    src.write_text(C_MAIN % {"fns": ", ".join("(void*)%s" % n for n in names),
                             "count": len(names)})
    exe = tmp_path / "main"
    lib_dir = os.path.dirname(capi.LIB_PATH)
    # the header alone, strictly: ISO C99, every warning an error
    only = tmp_path / "only.c"
    only.write_text('#include "gemm.h"\nint main(void) { return GEMM_OK; }\n')
    res = subprocess.run(["gcc", "-std=c99", "-pedantic-errors", "-Wall", "-Wextra", "-Werror",
                          "-I", os.path.dirname(capi.HEADER), "-c", str(only), "-o",
                          str(tmp_path / "only.o")], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    # the program (function pointers cast to void* are not ISO C, hence no -pedantic)
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror",
           "-I", os.path.dirname(capi.HEADER), str(src), "-o", str(exe), "-L", lib_dir,
           "-l:" + os.path.basename(capi.LIB_PATH), "-Wl,-rpath," + lib_dir]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip() == "ok", (run.returncode, run.stderr)


def test_header_has_no_cpp_outside_its_guard():
    """Outside the __cplusplus guard the header holds C only."""
    text = open(capi.HEADER).read()
    body = re.sub(r"#ifdef __cplusplus.*?#endif", "", text, flags=re.S)
    for token in ("extern \"C\"", "namespace", "template", "class ", "nullptr", "bool "):
        assert token not in body, token
