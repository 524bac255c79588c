"""The boundary from plain C: include/verifyhead.h compiles as C99 with gcc
(-Wall -Werror), and a C program linked against libverifyhead.so gets the
documented results from the host-only paths (sizes, status strings, argument
refusals before any device work).  CPU only."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "verifyhead.h"

int main(void) {
    int bad = 0;
    int32_t ids[1];
    float ml[1];
    char ws[64];
    /* sizes: a 16-byte header, then 8 bytes per row rounded up to 16 */
    if (vh_workspace_bytes(1) != 32) bad |= 1;
    if (vh_workspace_bytes(3) != 48) bad |= 2;
    if (vh_workspace_error_offset() != 4) bad |= 4;
    if (strlen(vh_status_string(VH_OK)) == 0) bad |= 8;
    /* refusals happen on the host, before any device is touched */
    if (mtp_draft_head_argmax(NULL, ws, (const int32_t*)ws, 1, 64, 4, ids, ml, ws, sizeof ws, NULL) != VH_ERR_NULL)
        bad |= 16;
    if (spec_verify_greedy(ws, ws, (const int32_t*)ws, 1, 16, 64, 4, ids, ids, ml, ws, sizeof ws, NULL) != VH_ERR_SHAPE)
        bad |= 32;
    printf("bad=%d version=%d\n", bad, vh_version());
    return bad;
}
"""


def test_header_is_c99_and_the_library_links_from_c(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    import verify_head_gb300 as vh
    lib = vh.build()
    src = tmp_path / "use_abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib)
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(lib),
                        "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert "bad=0" in r.stdout
