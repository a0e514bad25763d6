"""Contract between include/dsb.h and the ctypes binding (no GPU): a small C
program built against the header prints every struct's size and field
offsets, its status codes and its limits, and the binding's declarations must
match them field by field -- a field added, reordered or retyped on one side
only would otherwise pass garbage across the boundary."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = {  # C type -> binding class name
    "dsb_q8_0_mat": "Q8Mat",
    "dsb_kv_cache": "KVCache",
    "dsb_kv_pages": "KVPages",
    "dsb_rope": "RopeC",
    "dsb_model_shape": "ModelShapeC",
    "dsb_layer": "LayerC",
    "dsb_model": "ModelC",
    "dsb_layer_trace": "LayerTraceC",
    "dsb_step_trace": "StepTraceC",
}
MACROS = {"DSB_MAX_SEQS": "MAX_SEQS", "DSB_MAX_TOKENS": "MAX_TOKENS", "DSB_NARROW_MAX": "NARROW_MAX",
          "DSB_ATTN_CHUNK": "ATTN_CHUNK", "DSB_KV_PAGE": "KV_PAGE", "DSB_F16": "DSB_F16", "DSB_BF16": "DSB_BF16",
          "DSB_OK": "DSB_OK", "DSB_ERR_UNSUPPORTED": "DSB_ERR_UNSUPPORTED"}


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from session_decode_step_dsb_gb300 import dsb
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "dsb.h"', 'int main(void) {']
    for ctype, cls in STRUCTS.items():
        lines.append(f'  printf("{ctype} size %zu\\n", sizeof({ctype}));')
        for name, _ in getattr(dsb, cls)._fields_:
            lines.append(f'  printf("{ctype} {name} %zu\\n", offsetof({ctype}, {name}));')
    for macro in MACROS:
        lines.append(f'  printf("macro {macro} %d\\n", (int)({macro}));')
    for name in dsb.STATUS_NAMES.values():
        lines.append(f'  printf("status {name} %d\\n", (int){name});')
    lines += ["  return 0;", "}"]
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        a, b, v = line.split()
        table[(a, b)] = int(v)
    return table


@pytest.mark.parametrize("ctype", sorted(STRUCTS))
def test_struct_layout_matches_the_header(c_layout, ctype):
    from session_decode_step_dsb_gb300 import dsb
    cls = getattr(dsb, STRUCTS[ctype])
    assert ctypes.sizeof(cls) == c_layout[(ctype, "size")], ctype
    for name, _ in cls._fields_:
        assert getattr(cls, name).offset == c_layout[(ctype, name)], (ctype, name)


def test_limits_and_codes_match_the_header(c_layout):
    from session_decode_step_dsb_gb300 import dsb
    for macro, attr in MACROS.items():
        assert getattr(dsb, attr) == c_layout[("macro", macro)], macro
    for code, name in dsb.STATUS_NAMES.items():
        assert c_layout[("status", name)] == code, name
