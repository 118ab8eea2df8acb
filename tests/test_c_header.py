"""include/asp.h is a C header: it compiles as strict C99 and links against libasp.so.

A tiny C program (written here, compiled with gcc, no GPU needed to build)
includes the header, takes the address of every declared entry point and
checks the version and a host-side argument check through the C ABI.
"""

import os
import shutil
import subprocess

import pytest

from adaptive_sparse_paged_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SRC = r"""
#include <stdio.h>
#include "asp.h"

typedef void (*any_fn)(void);

int main(void) {
  any_fn fns[] = {
%s
  };
  size_t bytes = 0;
  asp_paged_kv kv = {0};
  if (asp_abi_version() != ASP_ABI_VERSION) return 1;
  /* null pointers are rejected on the host, before any device work */
  if (asp_workspace_size(&kv, &bytes) != ASP_EINVAL) return 2;
  if (asp_workspace_size(NULL, &bytes) != ASP_EINVAL) return 3;
  if (asp_status_string(ASP_OK) == NULL) return 4;
  printf("%%d entry points\n", (int)(sizeof(fns) / sizeof(fns[0])));
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
def test_header_is_c99_and_links(tmp_path):
    lib_path = B.LIB_PATH
    if not os.path.exists(lib_path):
        import __graft_entry__ as g
        g.build()
    entries = "\n".join(f"    (any_fn){name}," for name in B.EXPORTED)
    src = tmp_path / "use_asp.c"
    src.write_text(C_SRC % entries)
    exe = tmp_path / "use_asp"
    lib_dir = os.path.dirname(lib_path)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
           "-L", lib_dir, "-lasp", f"-Wl,-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert f"{len(B.EXPORTED)} entry points" in run.stdout
