"""The binding's view of the C ABI matches include/kvo.h (host logic, no GPU).

Two checks that need no device: the ctypes structures have the size and field
offsets that a C compiler gives the header's structs (plain gcc on the header
alone), and every entry point is declared to ctypes with as many arguments as
its prototype in the header has.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvo.h")

STRUCTS = {
    "kvo_config": "KvoConfig",
    "kvo_stats": "KvoStats",
    "kvo_lw_config": "KvoLwConfig",
}


def _c_layout(tmp_path):
    """sizeof and offsetof of every field of the header's structs, from gcc."""
    from top_cache_gb300 import kvo
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "kvo.h"', "int main(void) {"]
    for cname, pyname in STRUCTS.items():
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for field, _ in getattr(kvo, pyname)._fields_:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, field, cname, field))
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    exe = tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        cname, field, value = line.split()
        table[(cname, field)] = int(value)
    return table


def test_struct_layouts_match_header(tmp_path):
    from top_cache_gb300 import kvo
    try:
        table = _c_layout(tmp_path)
    except (OSError, subprocess.CalledProcessError) as e:
        pytest.fail("could not compile the header's layout probe: %r" % (e,))
    for cname, pyname in STRUCTS.items():
        cls = getattr(kvo, pyname)
        assert ctypes.sizeof(cls) == table[(cname, "size")], cname
        for field, _ in cls._fields_:
            assert getattr(cls, field).offset == table[(cname, field)], (cname, field)


def _prototypes():
    """name -> number of parameters of every kvo_* prototype in the header."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = {}
    for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(kvo_\w+)\s*\(([^)]*)\)\s*;", src, flags=re.M):
        params = " ".join(m.group(2).split())
        protos[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return protos


def test_argtypes_match_prototypes():
    from top_cache_gb300 import build, kvo
    build.build()
    L = kvo.lib()
    protos = _prototypes()
    assert set(protos) == set(kvo.EXPORTED)
    for name, n in protos.items():
        f = getattr(L, name)
        assert f.argtypes is not None, name
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)
