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
    assert lib.tl_encoder_forward_host(None, None, 1, 1, None, None, None, 0, None) == 1
    assert lib.tl_encoder_host_workspace_size(None, 1, 1, None) == 1
    assert lib.tl_encoder_set_path(None, 0) == 1
    assert lib.tl_encoder_set_host_chunks(None, 0) == 1
    assert lib.tl_encoder_plan(None, 1, 1, None) == 1
    assert lib.tl_encoder_set_attention_split(None, 0) == 1
    assert lib.tl_encoder_attention_split(None, 1, 1, None) == 1
    assert lib.tl_encoder_set_graphs(None, 1) == 1
    assert lib.tl_encoder_set_gemm_pairs(None, 1) == 1
    assert lib.tl_encoder_set_mega_assist(None, 1) == 1
    assert lib.tl_encoder_mega_assisted(None, 1, 1, None) == 1
    assert lib.tl_encoder_graph_stats(None, None, None) == 1
    # Shape checks at create time also come before any CUDA call (the weight
    # pointers are not read when the shape is refused).
    dummy = ctypes.create_string_buffer(12 * 8)
    for d_model, heads, d_ff, dtype, want in [(100, 4, 512, 1, 2),   # d_model % 16
                                              (2048, 16, 512, 1, 2),  # d_model > 1024
                                              (128, 3, 512, 1, 2),    # heads do not divide
                                              (128, 4, 520, 1, 2),    # d_ff % 16
                                              (128, 4, 512, 7, 1),    # no such dtype
                                              (8, 1, 512, 1, 1)]:     # d_model < 16
        assert lib.tl_encoder_create(dummy, 1, d_model, heads, d_ff, dtype, ctypes.byref(h)) == want


def test_header_compiles_as_plain_c(tmp_path):
    """The boundary header is plain C99 (no C++ or CUDA types leak into it)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        import pytest
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "tl_encoder.h"\n'
                   "int main(void) {\n"
                   "  tl_layer_weights w = {0};\n"
                   "  tl_encoder *h = 0;\n"
                   "  (void)w;\n"
                   "  return tl_encoder_destroy(h) == TL_OK ? 0 : 1;\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src),
                        "-o", str(tmp_path / "use_header.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_no_cpu_fallback_without_a_gpu():
    """Without a CUDA device the product path raises; nothing computes on the
    host in its place."""
    import pytest
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    from transformer_encoder_layer_gb300.inputs import make_inputs, tiny_shape
    s = tiny_shape(dtype="f16", batch=1, seq_len=4, vl_lo=4, vl_hi=4, d_model=32)
    inp = make_inputs(s, seed=0)
    with pytest.raises(binding.TLError) as e:
        binding.Encoder(inp.layers, 32, 2, 128, "f16")
    assert e.value.code == 3  # TL_ERR_CUDA
    with pytest.raises(Exception):
        binding.run_forward(inp)
