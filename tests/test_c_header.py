"""include/qlora.h as plain C: a C99 program that includes it compiles with every warning as an
error, links against libqlora.so and runs the calls that need no GPU (size queries, status
strings, the level table, argument checks that fail before any launch)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIBDIR = os.path.join(ROOT, "bit_nf4_quantized_36_b300")

PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <string.h>
#include "qlora.h"

int main(void) {
    /* storage of a 4096 x 4096 matrix: n/2 + nb + 4 ng + 4 bytes */
    const int64_t n = 4096LL * 4096LL, nb = n / 64, ng = (nb + 255) / 256;
    if (qlora_nf4_storage_bytes(4096, 4096) != (size_t)(n / 2 + nb + 4 * ng + 4)) return 1;
    if (qlora_fwd_workspace_bytes(4096, 4096, 4096, 16) == (size_t)-1) return 2;
    if (qlora_bwd_workspace_bytes(4096, 4096, 4096, 16) == (size_t)-1) return 3;
    if (strlen(qlora_status_string(QLORA_ERR_TIMEOUT)) == 0) return 4;
    float lv[16];
    qlora_nf4_levels(lv);
    if (lv[0] != -1.0f || lv[15] != 1.0f || lv[7] != 0.0f) return 5;
    for (int i = 1; i < 16; ++i)
        if (!(lv[i] > lv[i - 1])) return 6;
    /* argument errors are reported before the device is touched */
    qlora_nf4_tensor t;
    memset(&t, 0, sizeof t);
    t.rows = 256;
    t.cols = 100;  /* not a multiple of 64 */
    t.codes = (uint8_t *)0x10000;  /* never dereferenced: the shape is refused first */
    t.scale_codes = (int8_t *)0x20000;
    t.scale_scales = (float *)0x30000;
    t.scale_offset = (float *)0x40000;
    if (nf4_dequantize(&t, (uint16_t *)0x1000, NULL) != QLORA_ERR_UNSUPPORTED_SHAPE) return 7;
    if (nf4_quantize(NULL, &t, NULL, 0, NULL) != QLORA_ERR_INVALID_ARG) return 8;
    if (qlora_test_inject(2u) != QLORA_ERR_INVALID_ARG) return 9;
    if (qlora_launch_count() != 0) return 10;
    printf("ok\n");
    return 0;
}
"""


def test_header_compiles_as_c99_and_links(tmp_path):
    from bit_nf4_quantized_36_b300 import build
    build.build()
    src = tmp_path / "use_qlora.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_qlora"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", LIBDIR, "-lqlora", "-Wl,-rpath," + LIBDIR, "-lm", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
