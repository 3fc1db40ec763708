"""The C-ABI library loads on a host without a GPU and exports every entry
point include/moe.h declares; shape refusal needs no device."""
import ctypes
import os
import re

import pytest

import block_fp8_mixture_router_gb300 as moe
from block_fp8_mixture_router_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    build()
    return moe.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_refusals_without_a_device(lib):
    ok = moe.moe_config(2048, 256, 8, 512, 512, 128, 1024, 0)
    rc, n = moe.moe_required_bytes(ok)
    assert rc == moe.MOE_OK and n > 768 << 20
    bad = [moe.moe_config(2000, 256, 8, 512, 512, 128, 16, 0),
           moe.moe_config(2048, 256, 8, 500, 512, 128, 16, 0),
           moe.moe_config(2048, 256, 8, 512, 100, 128, 16, 0),
           moe.moe_config(2048, 257, 8, 512, 512, 128, 16, 0),
           moe.moe_config(2048, 4, 8, 512, 512, 128, 16, 0),
           moe.moe_config(2048, 256, 0, 512, 512, 128, 16, 0),
           moe.moe_config(2048, 256, 17, 512, 512, 128, 16, 0),
           moe.moe_config(2048, 256, 8, 512, 512, 256, 16, 0),
           moe.moe_config(2048, 256, 8, 512, 512, 1024, 16, 0),
           moe.moe_config(2048, 256, 8, 512, 512, 128, 0, 0),
           moe.moe_config(2048, 256, 8, 512, 512, 128, 65537, 0)]
    for cfg in bad:
        rc, h = moe.moe_create(cfg, 0)
        assert rc == moe.MOE_ERR_UNSUPPORTED_SHAPE and not h.value
        assert moe.moe_required_bytes(cfg)[0] == moe.MOE_ERR_UNSUPPORTED_SHAPE
    # one activation scale per row (act_group == hidden) is a supported shape
    assert moe.moe_required_bytes(moe.moe_config(2048, 256, 8, 512, 512, 2048, 16, 0))[0] == \
        moe.MOE_OK
    capped = moe.moe_config(2048, 256, 8, 512, 512, 128, 1024, 1 << 20)
    rc, h = moe.moe_create(capped, 0)
    assert rc == moe.MOE_ERR_ALLOC_LIMIT and not h.value
    assert moe.moe_create(ok, -1)[0] == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_forward(None, None, None, 1, 0) == moe.MOE_ERR_INVALID_ARG
    assert moe.moe_add_rmsnorm_quantize(None, None, None, None, 1e-6, 1, None, None, None,
                                        None, 0) == moe.MOE_ERR_INVALID_ARG
    moe.moe_destroy(None)
    assert moe.status_string(moe.MOE_ERR_DEVICE_TIMEOUT) == "device-side wait timed out"


def test_header_constants_match_the_binding():
    """Every MOE_* enumerator of include/moe.h has the same value in the binding."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    found = {}
    for body in re.findall(r"enum\s*\{(.*?)\}", src, flags=re.S):
        for name, value in re.findall(r"(MOE_[A-Z_]+)\s*=\s*(-?\d+)", body):
            found[name] = int(value)
    assert len(found) >= 9
    for name, value in found.items():
        assert getattr(moe, name) == value, name


def test_struct_layouts_match_the_header(tmp_path):
    """moe_config and moe_weights as ctypes lays them out equal the C layout
    of include/moe.h (offsets and sizes printed by a program gcc builds)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = {"moe_config": [f for f, _ in moe.moe_config._fields_],
              "moe_weights": [f for f, _ in moe.moe_weights._fields_]}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "moe.h"', "int main(void) {"]
    for st, names in fields.items():
        lines.append(f'  printf("{st} size %zu\\n", sizeof({st}));')
        for n in names:
            lines.append(f'  printf("{st} {n} %zu\\n", offsetof({st}, {n}));')
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c_layout = {tuple(ln.split()[:2]): int(ln.split()[2]) for ln in out if ln.strip()}
    for st, cls in (("moe_config", moe.moe_config), ("moe_weights", moe.moe_weights)):
        assert c_layout[(st, "size")] == ctypes.sizeof(cls), st
        for n in fields[st]:
            assert c_layout[(st, n)] == getattr(cls, n).offset, (st, n)


def _declaration_comments():
    """(function name, the comment block right above its declaration) for
    every function include/moe.h declares."""
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    out = {}
    for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*(?:enum\s*\{[^}]*\};\s*)?(?:#define [^\n]*\n\s*)?(?:typedef struct \w+ \w+;\s*)?"
                         r"(?:int|void|const char\*)\s+(moe_[a-z_]+)\s*\(", src, flags=re.S):
        out[m.group(2)] = m.group(1)
    return out


def test_every_declaration_cites_its_defining_passage():
    """Each entry point's comment names the passage of the pages that defines
    the operation; the allocation-free router says the pages have no
    counterpart instead, as does the workspace-poisoning test entry."""
    comments = _declaration_comments()
    assert set(comments) == set(declared_functions())
    for name, text in comments.items():
        flat = " ".join(text.split())
        if name in ("moe_route_static", "moe_debug_poison_workspace"):
            assert "no counterpart" in flat, name
            assert "Defined by:" not in flat, name
            continue
        assert "Defined by:" in flat, name
        cited = flat.split("Defined by:", 1)[1]
        assert re.search(r'(PR #9\d\d|commit ")', cited), (name, cited)
