"""The boundary is a C ABI: a C11 program that includes include/zeco_gla.h
compiles warning-free, links against the library and calls its host-side entry
points (no GPU work: shape queries and error strings only)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "zeco_gla.h"

int main(void) {
    zeco_shape s;
    memset(&s, 0, sizeof s);
    s.B = 1; s.H = 4; s.T = 1 << 20; s.dk = 256; s.dv = 512;
    s.P = 64; s.K = 8; s.C = 64; s.dtype = ZECO_BF16; s.path = ZECO_PATH_AUTO;
    s.decay = ZECO_DECAY_DIAG;
    /* every entry point's address, so that each declaration is type-checked */
    void (*fns[])(void) = {
        (void (*)(void))zeco_gla_fwd, (void (*)(void))zeco_gla_bwd,
        (void (*)(void))zeco_gla_bwd_noalloc, (void (*)(void))zeco_last_device_status,
        (void (*)(void))zeco_check_device_status, (void (*)(void))zeco_set_overlap,
    };
    (void)fns;
    printf("path %d\n", zeco_gla_resolve_path(&s));
    printf("segments %lld\n", (long long)zeco_gla_segments(&s));
    printf("saved %zu\n", zeco_gla_saved_bytes(&s));
    printf("ws_bwd %zu\n", zeco_gla_workspace_bytes(&s, 1));
    s.dk = 96;
    printf("path_dk96 %d\n", zeco_gla_resolve_path(&s));
    s.T = 1000;
    printf("bad %d %s\n", zeco_gla_resolve_path(&s), zeco_strerror(ZECO_ERR_ARG));
    printf("ws_err %s\n", zeco_strerror(ZECO_ERR_WORKSPACE));
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_c_program_compiles_links_and_queries_shapes(tmp_path):
    from chunked_state_scan_gb300 import build
    lib = build.build()
    src = tmp_path / "use_abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib)
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                           "-L", libdir, "-lzeco_gla", f"-Wl,-rpath,{libdir}"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert got["path"] == "2"          # ZECO_PATH_TC
    assert got["segments"] == "64"
    assert int(got["saved"]) > 0 and int(got["ws_bwd"]) > 0
    assert got["path_dk96"] == "1"     # ZECO_PATH_SIMT
    code, msg = got["bad"].split(" ", 1)
    assert int(code) < 0 and msg
    assert got["ws_err"] == "workspace too small"
