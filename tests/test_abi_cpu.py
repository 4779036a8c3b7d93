"""The ctypes binding against the C header, without a GPU: every struct the header declares
has the same field names, offsets and size in the binding as gcc gives it, and the status
codes and kernel kinds match the header's enums."""
import ctypes as C
import os
import re
import shutil
import subprocess

import pytest

from tests.conftest import ROOT

B = pytest.importorskip("packed_rectified_flow_packer_b300.binding")
HEADER = os.path.join(ROOT, "include", "mageflow.h")
STRUCTS = ["mf_sample", "mf_plan_info", "mf_dims", "mf_temb_weights", "mf_stream_weights",
           "mf_block_weights", "mf_stream_weights_fp8", "mf_block_weights_fp8", "mf_stream_grads",
           "mf_block_grads", "mf_trace_entry"]


def _header_fields(name):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"typedef struct \{([^{}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "const void* a; const void* b" are split already; "T x" -> x
        fields.append(re.findall(r"[A-Za-z_]\w*", decl)[-1])
    return fields


@pytest.mark.parametrize("name", STRUCTS)
def test_struct_field_names(name):
    ct = getattr(B, name)
    assert [f[0] for f in ct._fields_] == _header_fields(name)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_struct_layout_matches_gcc(tmp_path):
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "mageflow.h"', "int main(void) {"]
    for name in STRUCTS:
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for f in _header_fields(name):
            lines.append(f'  printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines += ["  return 0;", "}"]
    c = tmp_path / "abi.c"
    c.write_text("\n".join(lines))
    exe = tmp_path / "abi"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            parts = line.split()
            got[(parts[0], parts[1])] = int(parts[2])
    for name in STRUCTS:
        ct = getattr(B, name)
        assert C.sizeof(ct) == got[(name, "size")], name
        for f in _header_fields(name):
            assert getattr(ct, f).offset == got[(name, f)], (name, f)


def _enum(name):
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    m = re.search(r"typedef enum \{([^{}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    return {k: int(v) for k, v in re.findall(r"(\w+)\s*=\s*(\d+)", m.group(1))}


def test_status_and_kind_enums():
    st = _enum("mf_status")
    assert {v: k for k, v in st.items()} == B.STATUS
    kinds = _enum("mf_kernel_kind")
    n = kinds.pop("MF_K_COUNT")
    assert n == len(B.KERNEL_KINDS) == len(kinds)
    assert sorted(kinds.values()) == list(range(n))
