"""The C ABI from plain C: a C99 program that includes include/kda.h (strict
warnings as errors) links against libkda.so and calls the host-only entry
points.  No GPU is needed: those calls make no CUDA call."""
import os
import shutil
import subprocess

import pytest

from kda_prefill_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "kda.h"

int main(void) {
    /* three sequences of 37, 0 and 59 tokens: chunks (0, 0) and (2, 0) */
    const int32_t cu[4] = {0, 37, 37, 96};
    int32_t seq[8], in_seq[8], off[4];
    int64_t n = -1;
    if (kda_chunk_size() != 64) return 1;
    if (kda_plan_chunks(cu, 3, kda_chunk_size(), seq, in_seq, off, 8, &n) != KDA_OK) return 2;
    if (n != 2 || seq[0] != 0 || seq[1] != 2 || in_seq[0] != 0 || in_seq[1] != 0) return 3;
    if (off[0] != 0 || off[1] != 1 || off[2] != 1 || off[3] != 2) return 4;
    /* too little capacity: the count still comes back */
    n = -1;
    if (kda_plan_chunks(cu, 3, 64, seq, in_seq, off, 1, &n) != KDA_ERR_WORKSPACE || n != 2) return 5;
    /* bounds that do not start at zero */
    {
        const int32_t bad[4] = {1, 37, 37, 96};
        if (kda_plan_chunks(bad, 3, 64, seq, in_seq, off, 8, &n) != KDA_ERR_INVALID_ARG) return 6;
        if (strlen(kda_last_error()) == 0) return 7;
    }
    if (kda_workspace_size(96, 3, 2) == 0 || kda_workspace_size(-1, 3, 2) != 0) return 8;
    if (!kda_kernel_name(0) || kda_kernel_name(4) != NULL) return 9;
    if (kda_check_status(NULL, NULL, NULL) != KDA_ERR_INVALID_ARG) return 10;
    if (kda_cache_entries() != 0) return 11;
    printf("ok %s\n", kda_kernel_name(0));
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_header_compiles_as_c99_and_host_calls_work(tmp_path):
    lib = kbuild.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
           f"-L{libdir}", "-lkda", f"-Wl,-rpath,{libdir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok kda_intra"), (r.returncode, r.stdout,
                                                                        r.stderr)
