"""The boundary from plain C: a C99 program that includes include/kvc.h and links
libkvc.so (no Python, no torch) calls host-only entry points and gets the documented
answers."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "kvc.h"

int main(void) {
    kvc_desc d = {1, 65536, 8, 128, KVC_Q8_0, KVC_HEAD_MAJOR};
    size_t kq = 0, ks = 0, vq = 0, vs = 0, scratch = 0;
    int32_t chunk = 0;
    int rc = kvc_cache_bytes(&d, &kq, &ks, &vq, &vs);
    rc |= kvc_scratch_bytes(&d, 40, &scratch);
    rc |= kvc_pipeline_chunk(28998, 8192, 4, 1024.0, &chunk);
    printf("%d %zu %zu %zu %zu %zu %d %zu %d\n", rc, kq, ks, vq, vs, scratch, chunk,
           kv_state_size(&d, 100), kvc_pipeline_chunk(0, 8192, 4, 1024.0, &chunk) == KVC_EINVAL);
    printf("%s\n", kvc_strerror(KVC_ENOSPC));
    return 0;
}
"""


def test_a_c99_program_uses_the_library(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from decode_attention_kv_cache_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
    src = tmp_path / "client.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "client"
    libdir = os.path.dirname(b.LIB)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                    "-o", str(exe), b.LIB, "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    f = out[0].split()
    n = 65536 * 8 * 128
    assert f[:5] == ["0", str(n), str(n // 32 * 2), str(n), str(n // 32 * 2)]
    assert int(f[5]) == 40 * 256 * 130 * 4          # n_head_q * splits * (head_dim + 2) floats
    assert f[6] == "3328"                            # the page's chunk for 28,998 tokens on four stages
    assert int(f[7]) == 32 + 100 * 2 * 8 * 4 * 34    # header + records of 8 heads x 4 blocks x 34 bytes
    assert f[8] == "1"
    assert out[1].strip() != ""
