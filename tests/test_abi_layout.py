"""The ctypes mirrors of the C ABI structs have the C layout (no GPU needed).

A C program built against include/bs.h prints sizeof and every field's
offsetof; the binding's ctypes Structures must agree field by field, since
a shifted field would hand a kernel a wrong device pointer.
"""

import ctypes
import os
import subprocess

import pytest

from conftest import ROOT, build_lib

STRUCTS = {
    "bs_mesh_info_t": "MeshInfo",
    "bs_gs_dev": "GSDev",
    "bs_plan_dev": "PlanDev",
    "bs_plan_info_t": "PlanInfo",
}


@pytest.fixture(scope="module")
def bs():
    build_lib()
    import order_fem_cg_gb300 as bs
    return bs


def test_struct_layouts_match_header(bs, tmp_path):
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "bs.h"', "int main(void) {"]
    for cname, pyname in STRUCTS.items():
        py = getattr(bs, pyname)
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'printf("{cname} {field} %zu\\n", offsetof({cname}, {field}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "abi.c"
    exe = tmp_path / "abi"
    src.write_text("\n".join(lines))
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe),
                    str(src)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    got = {}
    for line in out.splitlines():
        cname, what, val = line.split()
        got[(cname, what)] = int(val)
    for cname, pyname in STRUCTS.items():
        py = getattr(bs, pyname)
        assert ctypes.sizeof(py) == got[(cname, "size")], cname
        for field, _ in py._fields_:
            assert getattr(py, field).offset == got[(cname, field)], (cname, field)
