"""The C ABI from C: include/sdm.h compiles as strict C99 (and as C++), and a C program linked
against the built libsdm.so calls entry points that fail validation or touch no device (the
version, status strings, argument errors, an empty launch). Nothing here needs a GPU."""

from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from decode_state_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sdm.h"

int main(void) {
    static char fake[64];
    void* p = fake;
    sdm_decode_plan plan;
    int rc;
    printf("version %d\n", sdm_version());
    printf("ok %s\n", sdm_status_string(0));
    /* W = 0: rejected before any CUDA call */
    rc = sdm_decode_seq(p, p, (const float*)p, (const float*)p, (const float*)p, (const float*)p, p,
                        (const float*)p, p, 4, 64, 0, 8, 1, 2, SDM_F32, SDM_I32, NULL);
    printf("width %d %d\n", rc, rc == SDM_EWIDTH);
    /* a bad bank dtype */
    rc = sdm_decode_seq(p, p, (const float*)p, (const float*)p, (const float*)p, (const float*)p, p,
                        (const float*)p, p, 4, 64, 8, 8, 1, 2, 7, SDM_I32, NULL);
    printf("dtype %d\n", rc < 0);
    /* no streams: nothing to do, no pointer read */
    rc = sdm_decode_seq(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 64, 8, 8, 1, 2, SDM_BF16,
                        SDM_I64, NULL);
    printf("empty %d\n", rc);
    /* a plan record into NULL storage */
    rc = sdm_decode_plan_init(NULL, p, p, (const float*)p, (const float*)p, (const float*)p, (const float*)p, p,
                              (const float*)p, p, 4, 64, 8, 8, 1, 2, SDM_F32, SDM_I32);
    printf("plan %d\n", rc < 0);
    printf("record %d\n", (int)sizeof(plan) == SDM_DECODE_PLAN_BYTES);
    printf("message %d\n", strlen(sdm_status_string(SDM_EWIDTH)) > 0);
    return 0;
}
"""


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


def test_header_is_plain_c_and_cxx(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "sdm.h"\nint main(void) { return sdm_version() > 0 ? 0 : 1; }\n')
    for cc, std in ((_compiler("gcc"), "-std=c99"), (_compiler("g++"), "-std=c++17")):
        lang = ["-x", "c++"] if cc.endswith("g++") else []
        r = subprocess.run([cc, *lang, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", INCLUDE, "-fsyntax-only",
                            str(src)], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_c_program_calls_the_library(tmp_path):
    lib = build.build()
    libdir = os.path.dirname(lib)
    src = tmp_path / "abi.c"
    exe = tmp_path / "abi"
    src.write_text(PROGRAM)
    r = subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                        "-L", libdir, "-lsdm", f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    assert lines["version"] == "200"
    assert lines["ok"] == "ok"
    assert lines["width"].split()[1] == "1"
    assert lines["dtype"] == "1"
    assert lines["empty"] == "0"
    assert lines["plan"] == "1"
    assert lines["record"] == "1"
    assert lines["message"] == "1"
