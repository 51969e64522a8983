"""The C-ABI library without a GPU: it builds, loads, exports every function
include/qtts.h declares, the binding's struct layouts match the header, and
host-side argument checks answer before any device work."""
import ctypes as C
import os
import re
import subprocess

import pytest

from codebook_decode_gb300 import qtts

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qtts.h")


@pytest.fixture(scope="module")
def lib():
    from codebook_decode_gb300 import build
    build.build()
    return qtts.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qtts_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(n for n, _, _ in qtts.SIGNATURES) == names


def declared_arities():
    """Parameter count of every function the header declares."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"#define[^\n]*", "", src)
    out = {}
    for name, params in re.findall(r"\b(qtts_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", src):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arities_match_header():
    decl = declared_arities()
    for name, _, args in qtts.SIGNATURES:
        assert len(args) == decl[name], (name, len(args), decl[name])


def test_exports_with_nm(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", qtts.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (qtts_\w+)", out))
    assert set(declared_functions()) <= exported


def test_struct_layouts_match_header(tmp_path):
    prog = tmp_path / "sz.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "qtts.h"\n'
                    'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(qtts_config), sizeof(qtts_tensor),'
                    ' sizeof(qtts_session), sizeof(qtts_rng), offsetof(qtts_config, kv_pool_pages),'
                    ' offsetof(qtts_tensor, data)); return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    vals = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    assert vals == [C.sizeof(qtts.Config), C.sizeof(qtts.Tensor), C.sizeof(qtts.Session), C.sizeof(qtts.Rng),
                    qtts.Config.kv_pool_pages.offset, qtts.Tensor.data.offset]
    assert C.sizeof(qtts.Session) == 32 and C.sizeof(qtts.Rng) == 16


def test_abi_version_and_host_side_errors(lib):
    assert qtts.qtts_abi_version() == 1
    # null model / bad config answer on the host, before any CUDA call
    assert lib.qtts_frame_step(None, 1, *([None] * 2), 1, *([None] * 8)) == qtts.QTTS_E_INVALID
    assert lib.qtts_set_option(None, 1, 1) == qtts.QTTS_E_INVALID
    cfg = qtts.Config()
    m = C.c_void_p()
    assert lib.qtts_create(C.byref(cfg), 0, C.byref(m)) == qtts.QTTS_E_INVALID
    assert b"must be positive" in lib.qtts_last_error(None)
