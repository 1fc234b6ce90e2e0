"""The boundary is a C ABI: a plain C program includes include/gbattn.h (compiled
as C99 with warnings as errors), links libgbattn.so and calls entry points.
Without a GPU only the paths that end before a launch run: the size queries and
the argument checks, each of which must return its documented status."""
import os
import shutil
import subprocess

import pytest

from tests._util import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include "gbattn.h"

static int expect(const char *what, int got, int want)
{
    if (got != want) {
        printf("%s: got %d, want %d (%s)\n", what, got, want, gbattn_last_error());
        return 1;
    }
    return 0;
}

int main(void)
{
    int bad = 0;
    char buf[64] = {0};
    void *p = buf + (16 - ((size_t)buf & 15));      /* a 16-byte aligned address */
    bad |= expect("attn_fwd d=96", attn_fwd(p, p, p, p, (float *)p, 1, 2, 2, 8, 8, 96, 0, 0, 0.1f, NULL),
                  GBATTN_ERR_UNSUPPORTED);
    bad |= expect("attn_fwd H % H_kv", attn_fwd(p, p, p, p, (float *)p, 1, 3, 2, 8, 8, 128, 0, 0, 0.1f, NULL),
                  GBATTN_ERR_INVALID_ARG);
    bad |= expect("mla_decode H=256", mla_decode(p, p, p, p, p, (float *)p, 1, 256, 64, 512, 64, 0.04f, p, 0, NULL),
                  GBATTN_ERR_UNSUPPORTED);
    bad |= expect("ssd_scan P=32", ssd_scan(p, (const float *)p, (const float *)p, p, p, NULL, (float *)p, NULL,
                                            1, 8, 2, 32, 1, 128, NULL),
                  GBATTN_ERR_UNSUPPORTED);
    bad |= expect("attn_fwd_host buffer", attn_fwd_host(p, p, p, p, (float *)p, 1, 2, 1, 64, 64, 128, 0, 0, 0.1f,
                                                        NULL, 0, NULL),
                  GBATTN_ERR_WORKSPACE);
    if (attn_fwd_host_device_bytes(1, 2, 1, 64, 64, 128) != 2 * 32768 + 2 * 16384 + 512) {
        printf("attn_fwd_host_device_bytes\n");
        bad = 1;
    }
    printf(bad ? "FAIL\n" : "OK\n");
    return bad;
}
"""


def test_c_program_uses_the_abi(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = build_lib()
    src = tmp_path / "caller.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(lib)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-L", libdir, "-lgbattn", f"-Wl,-rpath,{libdir}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK")
