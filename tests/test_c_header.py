"""The boundary is a C ABI: include/h3q.h must compile as plain C99 (no C++
in the declarations), and a C program linked against libh3q.so must reach the
entry points.  The program calls only host-side functions (status strings,
the version, workspace sizes, the host pipeline's chunk plan, and argument
errors reported before any device work), so it runs without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include "h3q.h"

int main(void) {
  int64_t rows[8];
  int64_t n;
  if (h3q_version() < 100) return 1;
  printf("%s|%s\n", h3q_status_string(H3Q_OK), h3q_status_string(H3Q_ERR_TIMEOUT));
  printf("%zu\n", h3q_linear_workspace_bytes(8192, 5376, 5376));
  printf("%zu\n", h3q_linear_grouped_workspace_bytes(5, 8, 8, 64));   /* G out of range: 0 */
  n = h3q_linear_w8a8_grouped_host_chunks(1000, 256, 64, rows, 8);
  printf("%lld:", (long long)n);
  for (int64_t i = 0; i < n && i < 8; ++i) printf(" %lld", (long long)rows[i]);
  printf("\n");
  /* argument errors come back before any device work */
  printf("%d\n", (int)h3q_quantize_act(NULL, 4, 64, NULL, NULL, NULL));
  printf("%d\n", (int)h3q_probe_mma_s8_tops(NULL, NULL));
  printf("%d\n", (int)h3q_probe_mma_f16_pair_tflops(NULL, 0, NULL));
  return 0;
}
"""


def _cuda_include():
    for d in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h")):
            return os.path.join(d, "include")
    return None


def test_header_compiles_as_c99_and_links(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    inc = _cuda_include()
    if not cc or not inc:
        pytest.skip("needs a C compiler and the CUDA headers")
    import w8a8_int8_linear_h3q_gb300 as h3q
    h3q.load()                                   # builds libh3q.so if it is missing
    lib = h3q.lib_path()
    src = tmp_path / "abi.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "abi"
    # -isystem: CUDA's own headers are not pedantic C99; h3q.h and the program are
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           "-isystem", inc, str(src), "-o", str(exe), lib,
           "-Wl,-rpath," + os.path.dirname(lib)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    lines = r.stdout.splitlines()
    assert lines[0] == "ok|device-side wait timed out"
    assert int(lines[1]) == h3q.h3q_linear_workspace_bytes(8192, 5376, 5376)
    assert int(lines[2]) == 0
    assert lines[3] == "6: 64 128 256 256 256 40"
    assert int(lines[4]) == 1                    # H3Q_ERR_INVALID_ARG
    assert int(lines[5]) == 1
    assert int(lines[6]) == 1                    # the FP16 probe: no output pointer
