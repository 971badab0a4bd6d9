"""The library from C: a small C99 program that includes both headers, links libattn_fwd.so
and calls entry points whose arguments are rejected before any CUDA call, so it runs on a
host without a GPU. This checks that the headers are plain C and that the exported
symbols have the declared signatures' behaviour when called without any Python in between."""
import os
import shutil
import subprocess

import pytest

import dense_attention_forward_fwd_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include "attn_fwd.h"
#include "attn_bwd.h"

int main(void) {
    /* a fake, 16-byte aligned address: every call below is rejected before the device is used */
    void* a = (void*)(uintptr_t)(1u << 20);
    float* f = (float*)a;
    int rc[10];
    rc[0] = attn_fwd(a, a, a, a, f, 1, 1, 128, 128, 64, 0.125f, NULL);              /* d != 128 */
    rc[1] = attn_fwd(NULL, a, a, a, f, 1, 1, 128, 128, 128, 0.125f, NULL);          /* null q */
    rc[2] = attn_fwd((char*)a + 8, a, a, a, f, 1, 1, 128, 128, 128, 0.125f, NULL);  /* misaligned q */
    rc[3] = attn_fwd_causal(a, a, a, a, f, 1, 1, 256, 128, 128, 0.125f, NULL);      /* Nq > Nk */
    rc[4] = attn_fwd_bias(a, a, a, a, 0, 0, 130, a, f, 1, 1, 128, 130, 128, 0.125f, NULL);  /* bias rows */
    rc[5] = attn_fwd_fp8qk(a, a, a, a, f, 1, 1, 128, 128, 128, 0.125f, 0.0f, 1.0f, NULL);  /* descale 0 */
    rc[6] = attn_fwd_fp8(a, a, a, 120, a, f, 1, 1, 128, 128, 128, 0.125f, 1.0f, 1.0f, 1.0f, NULL);  /* ldv < Nk */
    rc[7] = attn_bwd(a, a, a, a, a, f, a, a, a, 1, 1, 128, 128, 64, 0.125f, NULL);  /* d != 128 */
    rc[8] = attn_fwd(a, a, a, a, f, 0, 1, 128, 128, 128, 0.125f, NULL);             /* empty batch */
    rc[9] = (int)(attn_fwd_kernel_count() + attn_bwd_kernel_count());
    for (int i = 0; i < 10; ++i) printf("%d %s\n", rc[i], i < 9 ? attn_status_string(rc[i]) : "launches");
    return 0;
}
"""


def test_c_program_links_and_gets_the_documented_codes(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    lib = attn.load_library()._name
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    lib, "-Wl,-rpath," + os.path.dirname(lib)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=120).stdout.split("\n")
    got = [line.split()[1] for line in out[:9]]
    assert got == ["ATTN_ERR_UNSUPPORTED", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_MISALIGNED", "ATTN_ERR_INVALID_ARG",
                   "ATTN_ERR_MISALIGNED", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
                   "ATTN_OK"]
    assert out[9].split()[0] == "0"   # nothing was launched
