"""The boundary from plain C: a C11 program that includes only ``include/tpmlp.h`` compiles with warnings as
errors, links against ``libtpmlp.so`` and calls the host-side entry points (status strings, workspace
sizes, argument validation, an empty batch).  No call reaches the CUDA runtime, so no GPU is needed."""
import os
import shutil
import subprocess

import pytest

from tensor_transformer_mlp_tp_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "tpmlp.h"

int main(void) {
  tpmlp_shape s;
  size_t bytes = 0, bytes_sp = 0;
  memset(&s, 0, sizeof(s));
  s.tokens = 8192;
  s.d = 4096;
  s.ffn = 16384;
  s.n_shards = 8;
  s.dtype = TPMLP_BF16;
  if (tpmlp_workspace_size(&s, TPMLP_OP_FWD, &bytes) != TPMLP_OK) return 1;
  if (tpmlp_workspace_size(&s, TPMLP_OP_SP_FWD, &bytes_sp) != TPMLP_OK) return 2;
  /* the forward's workspace holds H [T x F] bf16 at least; the SP forward adds the gathered X */
  if (bytes < (size_t)(8192) * 16384 * 2 || bytes_sp <= bytes) return 3;
  /* invalid shapes are rejected before anything runs */
  s.ffn = 16383;
  if (tpmlp_workspace_size(&s, TPMLP_OP_FWD, &bytes) != TPMLP_ERR_INVALID_ARG) return 4;
  s.ffn = 16384;
  if (tpmlp_forward(NULL, NULL, NULL, NULL, &s, NULL, NULL, NULL, NULL, 0, NULL) != TPMLP_ERR_INVALID_ARG) return 5;
  /* an empty batch is a valid call that launches nothing */
  s.tokens = 0;
  if (tpmlp_forward(NULL, NULL, NULL, NULL, &s, NULL, NULL, NULL, NULL, 0, NULL) != TPMLP_OK) return 6;
  if (strlen(tpmlp_status_string(TPMLP_ERR_WORKSPACE)) == 0) return 7;
  printf("%zu %zu %s\n", bytes, bytes_sp, tpmlp_status_string(TPMLP_OK));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_c_program_compiles_links_and_calls_the_abi(tmp_path):
    lib = build.build()
    src = tmp_path / "client.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "client"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-L", libdir, "-ltpmlp", "-Wl,-rpath," + libdir, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    fwd, sp, ok = r.stdout.split()
    assert int(sp) > int(fwd) > 0 and ok
