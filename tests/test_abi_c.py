"""The C boundary from plain C: a C99 program compiled against include/neo.h
(no C++, no Python) and linked with libneo.so calls the host-only entry points
and argument checks, which return before any CUDA call. No GPU."""

import os
import shutil
import subprocess

import pytest

from attention_neo_qknorm_gb300.build import BUILD, INCLUDE, build

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "neo.h"

int main(void) {
    if (neo_version() != 100) return 1;
    for (int s = 0; s <= 5; ++s) {
        const char* name = neo_status_string((neo_status)s);
        if (!name || strncmp(name, "NEO_", 4) != 0) return 2;
    }
    float t[11];
    if (neo_time_schedule(t, 10, 1.0f) != NEO_OK || t[0] != 0.0f || t[10] != 1.0f) return 3;
    float sigma = 0.0f;   /* sqrt(64 * 64 / 2^2 / 64) = 4 */
    if (neo_noise_scale(64, 64, 2, 64.0f, 1.0f, NEO_NOISE_RESOLUTION, 16.0f, &sigma) != NEO_OK) return 4;
    if (sigma < 3.999f || sigma > 4.001f) return 5;
    if (neo_flow_euler_step(NULL, NULL, 8, 0.5f, 0.6f, 0.02f, NULL, 0) != NEO_ERR_INVALID_ARG) return 6;
    if (neo_gen_attention(NULL, NULL, NULL, NULL, NULL, NEO_BF16, NULL, 0, 0, 1, 1, 32, 8, 64, NEO_MASK_FULL,
                          NULL, NULL, 0.1f, NULL, NULL, 0) != NEO_ERR_INVALID_ARG) return 7;
    neo_pos_segment seg = {NEO_SEG_TEXT, 0, 4, 0};
    if (neo_build_positions(NULL, 4, &seg, 1, 0) != NEO_ERR_INVALID_ARG) return 8;
    puts("c abi ok");
    return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    return build()


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    pytest.skip("CUDA headers not found")


def test_header_compiles_as_c_and_the_library_links(lib_path, tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no C compiler")
    src = tmp_path / "neo_c_abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "neo_c_abi"
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, "-I", _cuda_include(), str(src),
                    "-L", BUILD, "-lneo", "-Wl,-rpath," + BUILD, "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, f"exit {r.returncode}: {r.stdout}{r.stderr}"
    assert r.stdout.strip() == "c abi ok"
