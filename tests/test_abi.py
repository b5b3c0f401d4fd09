"""The C-ABI library builds, loads and exports every entry point include/pagedkv.h declares
(no GPU needed: nothing is called that touches a device)."""
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_core_calls():
    names = declared_functions()
    for n in ("kv_cache_create", "paged_kv_append", "paged_decode_attention", "packed_prefill_attention",
              "paged_slot_mapping", "kv_cache_destroy", "kv_cache_check_error", "pkv_last_error"):
        assert n in names


@pytest.fixture(scope="module")
def built_lib():
    from paged_kv_cache_134_gb300 import build
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    return build.build()


def test_library_exports_every_declared_symbol(built_lib):
    out = subprocess.run(["nm", "-D", "--defined-only", built_lib], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing


def test_library_loads_and_binds(built_lib):
    import paged_kv_cache_134_gb300 as P
    L = P.lib()
    for n in declared_functions():
        assert hasattr(L, n)
    assert L.pkv_last_error() == b""


def test_header_compiles_as_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "pagedkv.h"\nint main(void){ pkv_cache_t c = 0; (void)c; return PKV_OK; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(tmp_path / "t")], check=True)


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_cache_134_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pagedkv_oracle" not in text, f
