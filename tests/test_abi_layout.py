"""The binding's ctypes mirrors of decode_attn_params and decode_attn_plan
have the C structs' size and field offsets: a small C program built against
include/decode_attn.h with gcc prints them (no GPU, no CUDA headers)."""
import ctypes
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def c_layout(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    import paged_gqa_decode_06_gb300 as pkg
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "decode_attn.h"',
             'int main(void) {']
    for ctype, cls in (("decode_attn_params", pkg.DecodeAttnParams),
                       ("decode_attn_plan", pkg.DecodeAttnPlan)):
        lines.append(f'  printf("{ctype} size %zu\\n", sizeof({ctype}));')
        for name, _ in cls._fields_:
            lines.append(f'  printf("{ctype} {name} %zu\\n", offsetof({ctype}, {name}));')
    lines += ['  return 0;', '}']
    d = tmp_path_factory.mktemp("abi")
    src, exe = d / "layout.c", d / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        ctype, field, value = line.split()
        table[(ctype, field)] = int(value)
    return pkg, table


def test_structs_match_the_header(c_layout):
    pkg, table = c_layout
    for ctype, cls in (("decode_attn_params", pkg.DecodeAttnParams),
                       ("decode_attn_plan", pkg.DecodeAttnPlan)):
        assert ctypes.sizeof(cls) == table[(ctype, "size")], ctype
        for name, _ in cls._fields_:
            assert getattr(cls, name).offset == table[(ctype, name)], (ctype, name)
