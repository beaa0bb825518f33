"""include/domino.h as a C caller sees it: the header compiles as strict C11 with every warning an
error, and the layout of domino_cfg that the C compiler picks (size, and offset of every field)
is the one the ctypes binding (comm_overlap_gb300/domino.py) mirrors by hand.  Needs gcc, no GPU."""
import ctypes
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

HEADER_DIR = os.path.join(ROOT, "include")

# the fields of domino_cfg in declaration order, as the header writes them
CFG_FIELDS = ["M", "h", "ffn", "t", "p", "q", "act", "sched", "layers", "ln_eps", "flags", "heads", "seq",
              "reduce_ctas", "attn_ctas"]

C_SOURCE = r"""
#include <stddef.h>
#include <stdio.h>
#include "domino.h"

int main(void) {
  printf("size %zu\n", sizeof(domino_cfg));
%s
  return 0;
}
"""


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    d = tmp_path_factory.mktemp("hdr")
    src = d / "layout.c"
    prints = "\n".join(f'  printf("{f} %zu\\n", offsetof(domino_cfg, {f}));' for f in CFG_FIELDS)
    src.write_text(C_SOURCE.replace("%s", prints))
    exe = d / "layout"
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", HEADER_DIR, str(src),
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return {k: int(v) for k, v in (line.split() for line in out.splitlines())}


def test_header_compiles_as_c11_and_prototypes_are_callable(tmp_path):
    """A C translation unit that calls every path entry point with the header's types."""
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    src = tmp_path / "calls.c"
    src.write_text(r"""
#include <stddef.h>
#include <stdint.h>
#include "domino.h"
int use(domino_handle h, const domino_cfg* c, const uint16_t* x, uint16_t* y, float* g, void* ws, void* st);
int use(domino_handle h, const domino_cfg* c, const uint16_t* x, uint16_t* y, float* g, void* ws, void* st) {
  size_t n = 0;
  int64_t k = 0;
  double ms = 0.0;
  domino_status s = domino_workspace_size(c, DOMINO_PASS_FWD, &n);
  s |= domino_mlp_fwd(h, c, x, x, x, y, NULL, ws, n, st);
  s |= domino_mlp_bwd(h, c, x, x, x, x, x, y, g, g, ws, n, st);
  s |= domino_mlp_fwd_noalloc(h, c, x, x, x, y, NULL, st);
  s |= domino_stack_fwd(h, c, x, x, x, y, ws, n, st);
  s |= domino_shard_sum(g, 2, 4, 8, NULL, 0, y, 8, st);
  s |= domino_timing_read(h, DOMINO_K_SHARD_SUM, &k, &ms);
  return (int)s + (domino_status_string(s)[0] != 0) + (domino_last_error() != NULL);
}
""")
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", HEADER_DIR, "-c",
                        str(src), "-o", str(tmp_path / "calls.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_cfg_layout_matches_the_binding(c_layout):
    from comm_overlap_gb300 import domino as dm
    assert c_layout["size"] == ctypes.sizeof(dm.domino_cfg)
    names = [f[0] for f in dm.domino_cfg._fields_]
    assert names == CFG_FIELDS
    for f in CFG_FIELDS:
        assert c_layout[f] == getattr(dm.domino_cfg, f).offset, f
