"""The C-ABI library loads and exports every symbol include/*.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import glob
import os
import re

from transformer_encoder_layer_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(tl_\w+)\s*\(", src):
            names.add(m.group(1))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("tl_encoder_create", "tl_encoder_forward", "tl_encoder_destroy",
              "tl_encoder_workspace_size", "tl_encoder_get_status", "tl_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol():
    path = build.build()
    lib = ctypes.CDLL(path)
    missing = [n for n in sorted(declared_symbols()) if not hasattr(lib, n)]
    assert not missing, missing
    # The binding declares a signature for every exported entry point.
    assert declared_symbols() <= set(binding.SIGNATURES)


def test_status_strings_without_gpu():
    lib = binding.load(build.build())
    for code in range(8):
        assert lib.tl_status_string(code)
    assert lib.tl_encoder_destroy(None) == 0
    # Argument validation happens before any CUDA call.
    h = ctypes.c_void_p()
    assert lib.tl_encoder_create(None, 1, 128, 4, 512, 1, ctypes.byref(h)) == 1
    assert lib.tl_encoder_workspace_size(None, 1, 1, None) == 1
    assert lib.tl_encoder_forward(None, None, 1, 1, None, None, None, 0, None) == 1
