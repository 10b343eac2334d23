"""The ctypes mirrors of the C-ABI structs have the header's layout.

A small C program including `include/mla_split_kv.h` prints sizeof and the
offset of every field the binding declares; the ctypes structures must agree
field by field, so a field added or reordered on one side only fails here on
the CPU rather than as corrupted arguments on the GPU.
"""
import os
import shutil
import subprocess

import pytest

from mla_split_kv_gb300 import binding as nb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = {
    "mla_chunk_t": nb.mla_chunk_t,
    "mla_device_info_t": nb.mla_device_info_t,
    "mla_plan_t": nb.mla_plan_t,
    "mla_decode_desc_t": nb.mla_decode_desc_t,
}


def c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_split_kv.h"', "int main(void) {"]
    for name, cls in STRUCTS.items():
        lines.append(f'  printf("{name} sizeof %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        struct, field, value = line.split()
        table[(struct, field)] = int(value)
    return table


def test_ctypes_structs_match_the_header(tmp_path):
    table = c_layout(tmp_path)
    import ctypes

    for name, cls in STRUCTS.items():
        assert table[(name, "sizeof")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert table[(name, field)] == getattr(cls, field).offset, (name, field)
