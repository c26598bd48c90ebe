"""The C-ABI library builds, loads, and exports every symbol the header
declares (no GPU needed: no compute call is made)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparsecos.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(ss_[a-z_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from sparse_embedding_exact_gb300 import build

    build.build()
    from sparse_embedding_exact_gb300 import _abi

    return _abi.load()


def test_header_declares_the_calls():
    names = declared_functions()
    for required in ("ss_create", "ss_row_norms", "ss_build_item_index", "ss_score_chunk",
                     "ss_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from sparse_embedding_exact_gb300 import _abi

    out = subprocess.run(["nm", "-D", "--defined-only", _abi.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(ss_[a-z_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    # and the binding declares a signature for each of them
    assert set(declared_functions()) == set(_abi.SIGNATURES)
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings(lib):
    for code in range(0, 9):
        s = lib.ss_status_string(code)
        assert isinstance(s, bytes) and s
    assert lib.ss_status_string(0) == b"ok"
    assert lib.ss_last_error(None) == b""


def test_null_arguments_are_rejected_without_a_gpu(lib):
    from sparse_embedding_exact_gb300 import _abi

    assert lib.ss_create(None, 0, 10, 8192, 0) == _abi.SS_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert lib.ss_create(ctypes.byref(h), 0, 0, 8192, 0) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_create(ctypes.byref(h), 0, 10, 0, 0) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_create(ctypes.byref(h), 0, 10, _abi.SS_MAX_CHUNK_ROWS + 1, 0) == _abi.SS_ERR_LIMIT
    assert lib.ss_destroy(None) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_row_norms(None, None, None, None) == _abi.SS_ERR_INVALID_ARG
    assert lib.ss_score_chunk(None, None, None, None, None, None, 0, None) == _abi.SS_ERR_INVALID_ARG


def test_library_is_built_for_sm_103a():
    from sparse_embedding_exact_gb300 import build

    assert ["-gencode", "arch=compute_103a,code=sm_103a"] == build.ARCH


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_embedding_exact_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b", text), f
                assert "cosine_oracle" not in text, f


def test_header_is_plain_c_and_every_call_links(lib, tmp_path):
    # A C99 program (no C++ anywhere) that takes the address of every declared
    # call, links against the library and runs the calls that need no device.
    import shutil

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from sparse_embedding_exact_gb300 import _abi

    names = declared_functions()
    src = tmp_path / "abi_check.c"
    src.write_text(
        '#include <stdio.h>\n#include <string.h>\n#include "sparsecos.h"\n'
        "typedef void (*fn)(void);\n"
        "static const fn calls[] = {\n" + "".join(f"  (fn){n},\n" for n in names) + "};\n"
        "int main(void) {\n"
        "  size_t i;\n"
        "  for (i = 0; i < sizeof(calls) / sizeof(calls[0]); ++i) if (!calls[i]) return 2;\n"
        "  for (i = 0; i <= 9; ++i) if (!ss_status_string((ss_status)i)) return 3;\n"
        "  if (ss_destroy(NULL) != SS_ERR_INVALID_ARG) return 4;\n"
        "  if (ss_invalidate(NULL) != SS_ERR_INVALID_ARG) return 5;\n"
        "  if (ss_kernel_launches(NULL) != 0) return 6;\n"
        "  if (strcmp(ss_last_error(NULL), \"\") != 0) return 7;\n"
        "  if (ss_set_device_limit(NULL, 0) != SS_ERR_INVALID_ARG) return 8;\n"
        "  printf(\"%d calls\\n\", (int)(sizeof(calls) / sizeof(calls[0])));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(_abi.library_path())
    libname = os.path.basename(_abi.library_path())[3:-3]  # libX.so -> X
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-L", libdir, "-l" + libname,
                        "-Wl,-rpath," + libdir, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.strip() == f"{len(names)} calls"
