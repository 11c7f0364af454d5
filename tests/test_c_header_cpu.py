"""The C ABI as a C program sees it: include/gclip.h compiles as C99 with
warnings as errors, and a program linked against the in-tree libgclip.so
plans a chunk table and reads status strings without any device."""
import os
import shutil
import subprocess

import pytest

import global_l2_norm_gb300 as g
from global_l2_norm_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "gclip.h"

int main(void) {
    /* Two host-side descriptors (addresses only; nothing is dereferenced):
       10,000 fp32 elements at a 16-byte boundary, 5 bf16 elements after it. */
    clip_tensor_desc_t d[2];
    int64_t n = -1;
    clip_chunk_t table[8];
    d[0].ptr = (void *)(uintptr_t)0x100000; d[0].numel = 10000; d[0].dtype = GCLIP_F32; d[0].reserved = 0;
    d[1].ptr = (void *)(uintptr_t)0x200002; d[1].numel = 5;     d[1].dtype = GCLIP_BF16; d[1].reserved = 0;
    if (clip_plan(d, 2, NULL, 0, &n) != GCLIP_OK) return 1;
    if (n != 3) return 2;                        /* 8192 + 1808 fp32, then 5 bf16 */
    if (clip_plan(d, 2, table, 8, &n) != GCLIP_OK) return 3;
    if (table[0].numel != GCLIP_CHUNK_BYTES / 4 || table[1].numel != 1808) return 4;
    if ((table[2].meta & 0xffu) != GCLIP_BF16 || (table[2].meta >> 8) != 1u) return 5;
    d[1].ptr = (void *)(uintptr_t)0x200001;      /* bf16 at an odd address */
    if (clip_plan(d, 2, NULL, 0, &n) != GCLIP_ERR_INVALID_ARG) return 6;
    if (clip_status_string(GCLIP_ERR_INVALID_ARG) == NULL) return 7;
    if (clip_get_variant(NULL) != -1 || clip_num_chunks(NULL) != -1) return 8;
    printf("ok %lld\n", (long long)n);
    return 0;
}
"""


def test_header_compiles_as_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    g.build()
    lib = _abi.lib_path()
    src = tmp_path / "use_gclip.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_gclip"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        lib, f"-Wl,-rpath,{os.path.dirname(lib)}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok 3", (r.returncode, r.stdout, r.stderr)
