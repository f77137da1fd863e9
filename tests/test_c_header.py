"""The boundary is a C ABI: include/repstep.h compiles as strict C11 and as C++17, and a
plain C program links against librepstep.so and calls the entry points that need no
device (sizes, layout, status names, bias corrections, image size, decay-mask bits, and
argument checks that reject before any device is touched)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from bitwise_reproducible_step_gb300 import repstep as rs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <string.h>
#include "repstep.h"

int main(void)
{
    repstep_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n = 12800000u;
    cfg.grad_dtype = REPSTEP_F32;
    cfg.hash_mode = REPSTEP_HASH_PF61;
    size_t ws = repstep_workspace_bytes(&cfg);
    repstep_layout lay;
    int rc = repstep_workspace_layout(&cfg, &lay);
    printf("workspace %zu %d %llu\n", ws, rc, (unsigned long long)lay.total);
    printf("g %llu leaves %llu\n", (unsigned long long)lay.g, (unsigned long long)lay.leaves);

    float bc1 = 0.0f, bc2 = 0.0f;
    repstep_bias_corrections(0.9f, 0.999f, 1, &bc1, &bc2);
    printf("bc %.9g %.9g\n", (double)bc1, (double)bc2);
    printf("image %llu\n", (unsigned long long)repstep_image_bytes(cfg.n));
    printf("status %s %s\n", repstep_strerror(REPSTEP_OK), repstep_strerror(REPSTEP_ERR_ALIGN));

    uint64_t seg_begin[2] = {0, 40};
    uint8_t decay[2] = {0, 1};
    uint32_t mask[3] = {0, 0, 0};
    rc = repstep_decay_mask_from_segments(70, seg_begin, decay, 2, mask);
    printf("mask %d %08x %08x %08x\n", rc, mask[0], mask[1], mask[2]);

    repstep_ctx *ctx = NULL;
    repstep_hparams hp;
    memset(&hp, 0, sizeof hp);
    printf("rejects %d %d %d %d\n",
           repstep_create(&cfg, NULL, ws, NULL, &ctx),
           repstep_step(NULL, NULL, 1, 1, 1, NULL, NULL, NULL, &hp, 1, NULL, NULL),
           repstep_step_from_host(NULL, NULL, 1, NULL, 0, 0, NULL, NULL, NULL, &hp, 1, NULL,
                                  NULL),
           repstep_sync(NULL, NULL));
    return ctx == NULL ? 0 : 1;
}
"""


def _compile(tmp_path, compiler, flags, src_name):
    src = tmp_path / src_name
    src.write_text(PROGRAM)
    exe = tmp_path / (src_name + ".out")
    lib_dir = os.path.dirname(rs.LIB_PATH)
    cmd = [compiler, *flags, "-I", INCLUDE, str(src), "-o", str(exe), "-L", lib_dir,
           "-lrepstep", f"-Wl,-rpath,{lib_dir}", "-lm"]
    out = subprocess.run(cmd, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    return exe


@pytest.mark.parametrize("compiler,flags,src", [
    ("gcc", ["-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic"], "abi.c"),
    ("g++", ["-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic"], "abi.cpp"),
])
def test_plain_program_against_the_c_abi(tmp_path, compiler, flags, src):
    if shutil.which(compiler) is None:
        pytest.skip(f"{compiler} not installed")
    if not os.path.exists(rs.LIB_PATH):
        pytest.skip("librepstep.so is not built")
    exe = _compile(tmp_path, compiler, flags, src)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    lines = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())

    cfg = rs.Config(12_800_000, 0, 0, 0, 0)
    ws = int(rs.lib().repstep_workspace_bytes(rs.C.byref(cfg)))
    assert lines["workspace"].split() == [str(ws), "0", str(ws)]
    assert lines["g"].split()[0] == "0"
    one = np.float32(1.0)
    want_bc = (one - np.float32(0.9), one - np.float32(0.999))   # 1 - b^t at t = 1, in fp32
    assert lines["bc"] == "%.9g %.9g" % (float(want_bc[0]), float(want_bc[1]))
    assert lines["image"] == "153600008"                  # 8 + 12n, the 12.8M example
    assert lines["status"] == f"{rs.strerror(0)} {rs.strerror(2)}"
    # elements 0..39 keep their weight (no decay), 40..69 decay
    assert lines["mask"] == "0 00000000 ffffff00 0000003f"
    assert lines["rejects"] == "1 1 1 1"


def test_readme_c_example_compiles(tmp_path):
    """The C example in README.md compiles as strict C11 against the header."""
    import re
    cuda_inc = "/usr/local/cuda/include"
    if shutil.which("gcc") is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA headers are missing")
    text = open(os.path.join(ROOT, "README.md"), encoding="utf-8").read()
    blocks = re.findall(r"```c\n(.*?)```", text, re.S)
    assert blocks, "README.md has no C example"
    src = tmp_path / "readme_example.c"
    src.write_text(blocks[0])
    out = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                          "-I", INCLUDE, "-I", cuda_inc, "-c", str(src),
                          "-o", str(tmp_path / "readme_example.o")],
                         capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
