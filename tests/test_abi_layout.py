"""The ctypes mirrors of the ABI structs (sparse_activation_decode_gb300/_lib.py)
have the C header's field order, offsets and sizes: a small C program built
against include/np.h with the host compiler prints them (no GPU needed)."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

STRUCTS = {"np_model_desc": "ModelDesc", "np_delta_view": "DeltaView", "np_stats": "Stats"}


@pytest.fixture(scope="module")
def c_layout():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no host C compiler")
    from sparse_activation_decode_gb300 import _lib as L
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "np.h"', "int main(void) {"]
    for cname, pyname in STRUCTS.items():
        lines.append(f'  printf("{cname} size %zu\\n", sizeof({cname}));')
        for field, _ in getattr(L, pyname)._fields_:
            lines.append(f'  printf("{cname} {field} %zu %zu\\n", offsetof({cname}, {field}), '
                         f'sizeof((({cname}*)0)->{field}));')
    lines += ["  return 0;", "}"]
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "layout.c"), os.path.join(d, "layout")
        with open(src, "w") as f:
            f.write("\n".join(lines) + "\n")
        subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    table = {}
    for line in out.splitlines():
        parts = line.split()
        if parts[1] == "size":
            table[(parts[0], None)] = (int(parts[2]),)
        else:
            table[(parts[0], parts[1])] = (int(parts[2]), int(parts[3]))
    return table


@pytest.mark.parametrize("cname", list(STRUCTS))
def test_struct_matches_header(c_layout, cname):
    import ctypes
    from sparse_activation_decode_gb300 import _lib as L
    cls = getattr(L, STRUCTS[cname])
    assert ctypes.sizeof(cls) == c_layout[(cname, None)][0]
    for field, _ in cls._fields_:
        off, size = c_layout[(cname, field)]
        desc = getattr(cls, field)
        assert (desc.offset, desc.size) == (off, size), f"{cname}.{field}"


def test_header_fields_all_mirrored():
    # every field the header declares in these structs has a ctypes twin
    import re
    from sparse_activation_decode_gb300 import _lib as L
    with open(os.path.join(ROOT, "include", "np.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    for cname, pyname in STRUCTS.items():
        body = re.search(r"typedef struct \{([^{}]*)\}\s*" + cname + ";", text).group(1)
        names = re.findall(r"(\w+)\s*(?:\[[^\]]*\])?\s*;", body)
        names += re.findall(r"\(\*\s*(\w+)\)", body)  # function pointers
        py = [f for f, _ in getattr(L, pyname)._fields_]
        assert sorted(set(names)) == sorted(set(py)), (cname, sorted(set(names) ^ set(py)))
