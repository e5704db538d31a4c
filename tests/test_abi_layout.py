"""The ctypes structures of the Python binding have the C header's layout.

A small C program compiled by the host compiler against include/kvpaged.h prints the
size of every structure the ABI passes by pointer and the offset of every field; the
binding's ctypes definitions must agree field by field (a mismatch would hand the
library shifted arguments without any error).  No GPU is needed."""

import json
import os
import shutil
import subprocess

import ctypes as C
import pytest

from paged_kv_cache_169_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STRUCTS = {"kv_pool_desc": abi.kv_pool_desc, "kv_decode_args": abi.kv_decode_args,
           "kv_alloc_stats_t": abi.kv_alloc_stats_t}


def _probe_source() -> str:
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "kvpaged.h"', "int main(void) {",
             '    printf("{");']
    first = True
    for name, cls in STRUCTS.items():
        fields = [f for f, _ in cls._fields_]
        sep = "" if first else ","
        first = False
        lines.append(f'    printf("{sep}\\"{name}\\": {{\\"size\\": %zu", sizeof({name}));')
        for f in fields:
            lines.append(f'    printf(", \\"{f}\\": %zu", offsetof({name}, {f}));')
        lines.append('    printf("}");')
    lines += ['    printf("}\\n");', "    return 0;", "}"]
    return "\n".join(lines)


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        pytest.skip("no host C compiler")
    d = tmp_path_factory.mktemp("abi_layout")
    src, exe = d / "probe.c", d / "probe"
    src.write_text(_probe_source())
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    return json.loads(subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout)


@pytest.mark.parametrize("name", sorted(STRUCTS))
def test_ctypes_structure_matches_header(c_layout, name):
    cls = STRUCTS[name]
    want = c_layout[name]
    assert C.sizeof(cls) == want["size"], (name, C.sizeof(cls), want["size"])
    for field, _ in cls._fields_:
        assert getattr(cls, field).offset == want[field], (name, field)
