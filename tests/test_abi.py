"""The C-ABI library builds, loads, and exports every call include/kvsel.h declares
(CPU only: no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvsel.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvsel_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__.load_builder().build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = _declared()
    for call in ["kvsel_memory_update", "kvsel_rule_scores", "kvsel_topk_retain", "kvsel_redirect_slots",
                 "kvsel_meank_build", "kvsel_block_scores", "kvsel_select_blocks", "kvsel_rerope_scatter"]:
        assert call in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_signatures_cover_header(lib):
    import kv_cache_retention_gb300 as kv
    assert sorted(kv.SIGNATURES) == _declared()
    for name in _declared():
        assert callable(getattr(kv, name))


def test_version_and_null_context(lib):
    lib.kvsel_version.restype = ctypes.c_int
    assert lib.kvsel_version() == 100
    lib.kvsel_last_error_string.restype = ctypes.c_char_p
    lib.kvsel_last_error_string.argtypes = [ctypes.c_void_p]
    assert lib.kvsel_last_error_string(None) == b"null context"
    lib.kvsel_ctx_destroy.argtypes = [ctypes.c_void_p]
    assert lib.kvsel_ctx_destroy(None) == 0
    # every call rejects a null context without touching the device
    lib.kvsel_redirect_slots.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    assert lib.kvsel_redirect_slots(None, None, None, 0, 0, None, None) == -1


def test_no_oracle_in_product_sources():
    """The product library and binding never reference the oracle."""
    pkg = os.path.join(ROOT, "kv_cache_retention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text and "orc_" not in text, f


def test_oracle_shares_nothing_with_the_product():
    """The oracle neither imports the product package nor includes its headers or kernels."""
    odir = os.path.join(ROOT, "oracle")
    for f in os.listdir(odir):
        if f.endswith((".py", ".c", ".h")):
            text = open(os.path.join(odir, f)).read()
            assert "kv_cache_retention_gb300" not in text, f
            assert "kvsel.h" not in text and "kvsel_internal" not in text and "csrc" not in text, f


def test_header_is_plain_c_and_links(lib, tmp_path):
    """A C99 program includes the header with every warning an error, links against the library
    and calls it (version, and a call rejected on a null context)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_kvsel.c"
    src.write_text(
        '#include <stdio.h>\n#include "kvsel.h"\n'
        "int main(void) {\n"
        "    if (kvsel_version() != 100) return 1;\n"
        "    if (kvsel_redirect_slots(NULL, NULL, NULL, 0, 0, NULL, NULL) != KVSEL_ERR_INVALID_ARG) return 2;\n"
        '    printf("%s\\n", kvsel_last_error_string(NULL));\n'
        "    return 0;\n}\n")
    exe = tmp_path / "use_kvsel"
    libdir = os.path.dirname(lib._name)
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lkvsel", "-Wl,-rpath," + libdir],
                   check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True)
    assert out.stdout.strip() == "null context"


def test_binding_fails_loudly_without_a_gpu_path():
    """CPU tensors, unsupported dtypes and a missing device are errors, never a fallback."""
    import torch

    import kv_cache_retention_gb300 as kv
    with pytest.raises(ValueError, match="CUDA tensor"):
        kv._ptr(torch.zeros(3))
    with pytest.raises(TypeError):
        kv._code(torch.zeros(3, dtype=torch.float16))
    assert kv._ptr(None) is None
    if not torch.cuda.is_available():
        with pytest.raises(kv.KvselError):
            kv.Context(0)
