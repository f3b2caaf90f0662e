"""The C ABI library loads without a GPU and exports every function include/g4.h declares;
the binding's struct layouts match the C compiler's (CPU only, no compute calls)."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "g4.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(g4_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def g4():
    from accelerator_decode_gb300 import build
    if not os.path.exists(build.LIB):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("libg4.so not built and no nvcc")
        build.build()
    from accelerator_decode_gb300 import g4 as mod
    return mod


def test_every_declared_symbol_is_exported(g4):
    names = _declared()
    assert "g4_create" in names and "g4_decode_step" in names and "g4_prefill" in names
    for n in names:
        assert hasattr(g4.lib, n), n


def test_status_strings(g4):
    for s in range(0, -8, -1):
        assert g4.status_string(s) != "unknown status"
    assert g4.last_cuda_error() == ""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no gcc")
def test_struct_layout_matches_c(g4, tmp_path):
    src = tmp_path / "sz.c"
    src.write_text('#include "g4.h"\n#include <stdio.h>\n#include <stddef.h>\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(g4_config), '
                   'sizeof(g4_linear), sizeof(g4_layer_weights), sizeof(g4_weights), '
                   'offsetof(g4_config, rms_eps), offsetof(g4_layer_weights, layer_scale), '
                   'offsetof(g4_config, table_format), offsetof(g4_weights, ple_table_scales));return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()))
    want = [ctypes.sizeof(g4.g4_config), ctypes.sizeof(g4.g4_linear), ctypes.sizeof(g4.g4_layer_weights),
            ctypes.sizeof(g4.g4_weights), g4.g4_config.rms_eps.offset, g4.g4_layer_weights.layer_scale.offset,
            g4.g4_config.table_format.offset, g4.g4_weights.ple_table_scales.offset]
    assert got == want


def test_invalid_arguments_are_rejected_on_the_host(g4):
    """Host-checkable errors return before any device work (safe without a GPU)."""
    h = ctypes.c_void_p()
    assert g4.lib.g4_create(None, None, 0, ctypes.byref(h)) == g4.G4_ERR_INVALID_ARG
    cfg = g4.g4_config()
    assert g4.lib.g4_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == g4.G4_ERR_INVALID_ARG
    assert g4.lib.g4_decode_step(None, None, 1, None, None, None, None, None) == g4.G4_ERR_INVALID_ARG
    assert g4.lib.g4_prefill(None, None, 1, None, None, None, None, None, None) == g4.G4_ERR_INVALID_ARG
    assert g4.lib.g4_linear_forward(None, None, 1, None, None) == g4.G4_ERR_INVALID_ARG
    assert g4.lib.g4_argmax_rows(0, None, 0, 5, None, None) == g4.G4_ERR_INVALID_ARG
    g4.lib.g4_free(None)
