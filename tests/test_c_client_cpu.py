"""The boundary is a plain C ABI: a C99 program that includes include/q2_0.h
(compiled with -pedantic -Werror) links against libq2_0.so and calls the entry
points that need no GPU — the version, scratch-size queries and argument
checks — and gets the same answers as the Python binding."""
import os
import shutil
import subprocess

import pytest

import bit_ternary_matmul_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "q2_0.h"

int main(void) {
    q2_0_mm_desc d = {0};
    q2_0_mm_plan *mp = 0;
    q2_0_mv_plan *vp = 0;
    int st_mm, st_mv;
    printf("%s\n", q2_0_version());
    printf("%lu\n", (unsigned long)q2_0_mul_mat_vec_workspace_size(2048, 1));
    printf("%lu\n", (unsigned long)q2_0_mul_mat_workspace_size(512, 6144, 2048, Q2_0_PREC_F16_SPLIT));
    printf("%lu\n", (unsigned long)q2_0_mul_mat_workspace_size(0, 4, 512, Q2_0_PREC_F16_SPLIT));
    st_mm = q2_0_mm_plan_create(&d, 1, Q2_0_PREC_F16_SPLIT, &mp);
    st_mv = q2_0_mv_plan_create(0, 1, 1, &vp);
    printf("%d %d %d %d\n", st_mm, mp == 0, st_mv, vp == 0);
    printf("%d %d\n", q2_0_mm_plan_launches(0), q2_0_mv_plan_launches(0));
    printf("%d\n", q2_0_mul_mat(0, 0, 0, 4, 512, 4, Q2_0_PREC_F16_SPLIT, 0, 0, 0));
    printf("%lu\n", (unsigned long)q2_0_split_bytes(4, 64));
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_links_and_calls_the_abi(tmp_path):
    q.build()
    lib = q.library_path()
    src = tmp_path / "client.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    lib, "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    L = q.lib()
    assert out[0] == q.q2_0_version()
    assert int(out[1]) == L.q2_0_mul_mat_vec_workspace_size(2048, 1) > 0
    assert int(out[2]) == L.q2_0_mul_mat_workspace_size(512, 6144, 2048, 0) > 0
    assert int(out[3]) == 0
    assert out[4].split() == [str(q.Q2_0_EINVAL), "1", str(q.Q2_0_EINVAL), "1"]
    assert out[5].split() == ["0", "0"]
    assert int(out[6]) == q.Q2_0_EINVAL
    assert int(out[7]) == L.q2_0_split_bytes(4, 64) > 0
