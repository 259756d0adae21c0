"""ctypes binding of the C ABI in ``include/tl_encoder.h``.

Argument marshalling only: torch tensors supply device memory and the CUDA
stream; every step of the forward runs in the library's CUDA kernels.  There
is no fallback: if the shared library has not been built (``build.build()``),
``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libtl_encoder.so")

TL_F32, TL_F16, TL_BF16 = 0, 1, 2
DTYPE_CODES = {"f32": TL_F32, "f16": TL_F16, "bf16": TL_BF16}
PATHS = {"auto": 0, "simt": 1, "layered": 2, "mega": 3, "dag": 4}
PATH_NAMES = {v: k for k, v in PATHS.items()}
STATUS = {0: "TL_OK", 1: "TL_ERR_INVALID_ARG", 2: "TL_ERR_UNSUPPORTED_SHAPE", 3: "TL_ERR_CUDA",
          4: "TL_ERR_OUT_OF_MEMORY", 5: "TL_ERR_WORKSPACE_TOO_SMALL", 6: "TL_ERR_BAD_VALID_LEN",
          7: "TL_ERR_DEVICE_TIMEOUT"}

# Every symbol the header declares, with its ctypes signature.
_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "tl_encoder_create": (_i, [_vp, _i, _i, _i, _i, _i, ctypes.POINTER(_vp)]),
    "tl_encoder_set_path": (_i, [_vp, _i]),
    "tl_encoder_set_host_chunks": (_i, [_vp, _i]),
    "tl_encoder_plan": (_i, [_vp, _i, _i, ctypes.POINTER(_i)]),
    "tl_encoder_set_attention_split": (_i, [_vp, _i]),
    "tl_encoder_set_graphs": (_i, [_vp, _i]),
    "tl_encoder_set_gemm_pairs": (_i, [_vp, _i]),
    "tl_encoder_set_mega_assist": (_i, [_vp, _i]),
    "tl_encoder_mega_assisted": (_i, [_vp, _i, _i, ctypes.POINTER(_i)]),
    "tl_encoder_graph_stats": (_i, [_vp, ctypes.POINTER(ctypes.c_longlong),
                                    ctypes.POINTER(ctypes.c_longlong)]),
    "tl_encoder_attention_split": (_i, [_vp, _i, _i, ctypes.POINTER(_i)]),
    "tl_encoder_workspace_size": (_i, [_vp, _i, _i, ctypes.POINTER(_sz)]),
    "tl_encoder_forward": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "tl_encoder_host_workspace_size": (_i, [_vp, _i, _i, ctypes.POINTER(_sz)]),
    "tl_encoder_forward_host": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _sz, _vp]),
    "tl_encoder_get_status": (_i, [_vp, _vp]),
    "tl_encoder_destroy": (_i, [_vp]),
    "tl_status_string": (ctypes.c_char_p, [_i]),
    "tl_encoder_forward_static": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp]),
    "tl_encoder_enable_timing": (_i, [_vp, _i, _i]),
    "tl_encoder_read_timing": (_i, [_vp, _i, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_i)]),
    "tl_encoder_reset_timing": (_i, [_vp]),
    "tl_kernel_class_name": (ctypes.c_char_p, [_i]),
    "tl_eval_gelu": (_i, [_vp, _vp, _vp, _sz, _vp]),
}
TL_KERNEL_CLASSES = 16


class TLError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)}")
        self.code = code


class _LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "w_qkv", "b_qkv", "w_o", "b_o", "ln1_g", "ln1_b",
        "w_1", "b_1", "w_2", "b_2", "ln2_g", "ln2_b")]


_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library (once) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing (run build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        raise TLError(code, what)


def _torch():
    import torch
    return torch


def torch_dtype(dtype: str):
    torch = _torch()
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]


def _stream_ptr(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


class Encoder:
    """One library handle: packed weights of an n-layer encoder on the current
    CUDA device.  ``layers`` holds per-layer dicts of host arrays (numpy, any
    float dtype: values are cast to ``dtype`` storage) or torch tensors."""

    def __init__(self, layers: Sequence[Dict[str, np.ndarray]], d_model: int, n_heads: int,
                 d_ff: int, dtype: str):
        from .inputs import PARAM_NAMES, to_storage
        self.lib = load()
        self.d_model, self.n_heads, self.d_ff, self.dtype = d_model, n_heads, d_ff, dtype
        self.n_layers = len(layers)
        keep: List[np.ndarray] = []
        arr = (_LayerWeights * self.n_layers)()
        for li, p in enumerate(layers):
            for name in PARAM_NAMES:
                v = p[name]
                if hasattr(v, "data_ptr"):
                    ptr = v.data_ptr()
                    keep.append(v)
                else:
                    a = to_storage(np.asarray(v, dtype=np.float64), dtype)
                    keep.append(a)
                    ptr = a.ctypes.data
                setattr(arr[li], name, ptr)
        h = ctypes.c_void_p()
        _check(self.lib.tl_encoder_create(ctypes.cast(arr, ctypes.c_void_p), self.n_layers, d_model,
                                          n_heads, d_ff, DTYPE_CODES[dtype], ctypes.byref(h)),
               "tl_encoder_create")
        self.handle = h
        self._ws = None

    def close(self):
        if getattr(self, "handle", None):
            self.lib.tl_encoder_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_path(self, path: str):
        _check(self.lib.tl_encoder_set_path(self.handle, PATHS[path]), "tl_encoder_set_path")

    def plan(self, B: int, L: int) -> str:
        p = ctypes.c_int()
        _check(self.lib.tl_encoder_plan(self.handle, B, L, ctypes.byref(p)), "tl_encoder_plan")
        return PATH_NAMES[p.value]

    def set_attention_split(self, key_tiles: int):
        """-1 automatic (default), 0 never, k > 0 chunks of k 64-key tiles."""
        _check(self.lib.tl_encoder_set_attention_split(self.handle, key_tiles),
               "tl_encoder_set_attention_split")

    def set_gemm_pairs(self, enable):
        """-1 automatic (default), 0 / False none, 1 / True every GEMM."""
        _check(self.lib.tl_encoder_set_gemm_pairs(self.handle, int(enable)),
               "tl_encoder_set_gemm_pairs")

    def set_mega_assist(self, enable: int):
        """-1 automatic (default), 0 never, 1 wherever possible."""
        _check(self.lib.tl_encoder_set_mega_assist(self.handle, int(enable)),
               "tl_encoder_set_mega_assist")

    def mega_assisted(self, B: int, L: int) -> bool:
        v = ctypes.c_int()
        _check(self.lib.tl_encoder_mega_assisted(self.handle, B, L, ctypes.byref(v)),
               "tl_encoder_mega_assisted")
        return bool(v.value)

    def set_graphs(self, enable: bool):
        _check(self.lib.tl_encoder_set_graphs(self.handle, int(enable)), "tl_encoder_set_graphs")

    def graph_stats(self):
        c, r = ctypes.c_longlong(), ctypes.c_longlong()
        _check(self.lib.tl_encoder_graph_stats(self.handle, ctypes.byref(c), ctypes.byref(r)),
               "tl_encoder_graph_stats")
        return c.value, r.value

    def attention_split(self, B: int, L: int) -> int:
        k = ctypes.c_int()
        _check(self.lib.tl_encoder_attention_split(self.handle, B, L, ctypes.byref(k)),
               "tl_encoder_attention_split")
        return k.value

    def workspace_size(self, B: int, L: int) -> int:
        n = ctypes.c_size_t()
        _check(self.lib.tl_encoder_workspace_size(self.handle, B, L, ctypes.byref(n)),
               "tl_encoder_workspace_size")
        return n.value

    def set_host_chunks(self, chunks: int):
        """Batch slices forward_host pipelines (0 = automatic, 1 = off)."""
        _check(self.lib.tl_encoder_set_host_chunks(self.handle, chunks), "tl_encoder_set_host_chunks")

    def host_workspace_size(self, B: int, L: int) -> int:
        n = ctypes.c_size_t()
        _check(self.lib.tl_encoder_host_workspace_size(self.handle, B, L, ctypes.byref(n)),
               "tl_encoder_host_workspace_size")
        return n.value

    def workspace(self, nbytes: int):
        torch = _torch()
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        return self._ws

    def forward(self, x, valid_len, out=None, workspace=None, stream=None, check: bool = True):
        """x: CUDA tensor [B, L, d] in the handle's dtype; valid_len: CUDA int32
        [B].  Enqueues the forward on ``stream`` (default: current stream) and
        returns ``out``.  check=True also reads the device status word (a
        stream synchronisation)."""
        torch = _torch()
        B, L, d = x.shape
        assert d == self.d_model and x.is_cuda and x.is_contiguous()
        assert valid_len.dtype == torch.int32 and valid_len.is_cuda
        if out is None:
            out = torch.empty_like(x)
        nbytes = self.workspace_size(B, L)
        ws = workspace if workspace is not None else self.workspace(nbytes)
        sp = _stream_ptr(stream)
        _check(self.lib.tl_encoder_forward(self.handle, x.data_ptr(), B, L, valid_len.data_ptr(),
                                           out.data_ptr(), ws.data_ptr() if nbytes else None,
                                           ws.numel() if nbytes else 0, sp), "tl_encoder_forward")
        if check:
            _check(self.lib.tl_encoder_get_status(self.handle, sp), "device status")
        return out

    def forward_static(self, x, valid_len, out=None, stream=None, check: bool = True):
        """The forward with the library's static scratch array instead of a
        caller workspace (allocates nothing; see tl_encoder_forward_static)."""
        torch = _torch()
        B, L, d = x.shape
        if out is None:
            out = torch.empty_like(x)
        sp = _stream_ptr(stream)
        _check(self.lib.tl_encoder_forward_static(self.handle, x.data_ptr(), B, L,
                                                  valid_len.data_ptr(), out.data_ptr(), sp),
               "tl_encoder_forward_static")
        if check:
            _check(self.lib.tl_encoder_get_status(self.handle, sp), "device status")
        return out

    def forward_host(self, x_host, valid_len_host, out_host, workspace=None, stream=None):
        """The same forward on host (ideally pinned) torch CPU tensors; the
        call copies in, runs, copies out and synchronises."""
        B, L, d = x_host.shape
        nbytes = self.host_workspace_size(B, L)
        ws = workspace if workspace is not None else self.workspace(nbytes)
        _check(self.lib.tl_encoder_forward_host(self.handle, x_host.data_ptr(), B, L,
                                                valid_len_host.data_ptr(), out_host.data_ptr(),
                                                ws.data_ptr(), ws.numel(), _stream_ptr(stream)),
               "tl_encoder_forward_host")
        return out_host

    def enable_timing(self, enable: bool = True, capacity: int = 4096):
        _check(self.lib.tl_encoder_enable_timing(self.handle, int(enable), capacity),
               "tl_encoder_enable_timing")

    def reset_timing(self):
        _check(self.lib.tl_encoder_reset_timing(self.handle), "tl_encoder_reset_timing")

    def read_timing(self) -> Dict[str, tuple]:
        """{kernel class name: (total ms, launches)} for classes that ran."""
        out = {}
        for k in range(TL_KERNEL_CLASSES):
            name = self.lib.tl_kernel_class_name(k).decode()
            if not name:
                continue
            ms, n = ctypes.c_float(), ctypes.c_int()
            _check(self.lib.tl_encoder_read_timing(self.handle, k, ctypes.byref(ms), ctypes.byref(n)),
                   "tl_encoder_read_timing")
            if n.value:
                out[name] = (ms.value, n.value)
        return out

    def get_status(self, stream=None) -> int:
        return self.lib.tl_encoder_get_status(self.handle, _stream_ptr(stream))


def run_forward(inp, path: str = "auto", device: str = "cuda") -> np.ndarray:
    """Convenience for tests: build an Encoder from an EncoderInputs, run it
    on the GPU and return the output as fp64 numpy."""
    torch = _torch()
    from .inputs import from_storage, to_storage
    s = inp.shape
    enc = Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    try:
        if path != "auto":
            enc.set_path(path)
        xs = to_storage(inp.x, s.dtype)
        if s.dtype == "bf16":
            x = torch.from_numpy(xs.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            x = torch.from_numpy(xs).to(device)
        vl = torch.from_numpy(np.asarray(inp.valid_len, dtype=np.int32)).to(device)
        out = enc.forward(x, vl)
        torch.cuda.synchronize()
        o = out.cpu()
        if s.dtype == "bf16":
            return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16")
        return from_storage(o.numpy(), s.dtype)
    finally:
        enc.close()
