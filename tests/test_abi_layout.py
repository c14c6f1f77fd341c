"""The ctypes structures of the Python binding against the C declarations of
include/kvq.h: a small C program compiled against the header prints each
struct's size and every field's offset, and the binding's ctypes view of the
same struct must agree field by field.  A field added, reordered or retyped on
one side only fails here, on the CPU, before any call can misread memory.
"""

import ctypes
import os
import shutil
import subprocess

import pytest

from quantized_kv_cache_02_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = [B.kvq_config, B.kvq_bytes_t, B.kvq_seq_info, B.kvq_unit_view, B.kvq_decode_opts, B.kvq_compare_t]


def c_layout(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvq.h"', "int main(void) {"]
    for st in STRUCTS:
        name = st.__name__
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in st._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    exe = tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        name, key, value = line.split()
        table[(name, key)] = int(value)
    return table


def test_binding_structs_match_header(tmp_path):
    table = c_layout(tmp_path)
    for st in STRUCTS:
        name = st.__name__
        assert ctypes.sizeof(st) == table[(name, "size")], f"{name}: size"
        for field, _ in st._fields_:
            assert getattr(st, field).offset == table[(name, field)], f"{name}.{field}: offset"
