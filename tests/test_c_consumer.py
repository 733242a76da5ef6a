"""A C program as the library's user: include/sageattn.h compiles as C11 (and as
C++) with warnings as errors, the program links against the built library, and
the host-only entry points (status names, padded length, workspace sizes,
argument rejection before any device work) answer as documented.  No GPU."""
import os
import shutil
import subprocess

import pytest

from sage_attention_forward_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "sageattn.h"

int main(void) {
  int bad = 0;
  if (strcmp(attn_status_name(ATTN_OK), "ATTN_OK") != 0) bad |= 1;
  if (sage_padded_len(76112) != 76160 || sage_padded_len(1) != 128) bad |= 2;
  if (sage_prepare_workspace_size(2, 3) != (size_t)2 * 3 * 128 * 4) bad |= 4;
  if (sage_attention_workspace_size(1, 2, 256, 0, 0, 1) >= sage_attention_workspace_size(1, 2, 256, 0, 0, 0)) bad |= 8;
  {
    const int64_t st[3] = {256 * 2 * 128, 256, 128};
    /* head dimension 64 is refused before anything touches a device */
    attn_status s = attn_fwd_bf16((const void*)0x10000, (const void*)0x10000, (const void*)0x10000, (void*)0x10000,
                                  1, 256, 2, 64, st, st, st, st, 0.088f, (attn_stream_t)0);
    if (s != ATTN_ERR_UNSUPPORTED || attn_last_error()[0] == '\0') bad |= 16;
  }
  printf("c consumer %d\n", bad);
  return bad;
}
"""


def test_c_program_builds_links_and_calls(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = lib_build.build()
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    cudart_dir = "/usr/local/cuda/lib64"
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
           lib, f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{cudart_dir}", f"-L{cudart_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c consumer 0" in r.stdout, (r.stdout, r.stderr[-2000:])


def test_header_compiles_as_cpp(tmp_path):
    if shutil.which("g++") is None:
        pytest.skip("g++ not available")
    src = tmp_path / "consumer.cpp"
    src.write_text('#include "sageattn.h"\nint main() { return sage_padded_len(1) == 128 ? 0 : 1; }\n')
    r = subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I", INCLUDE, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
