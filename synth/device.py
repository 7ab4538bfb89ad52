"""ctypes wrapper of the device generator (synth_gen.cu) and its build step."""

from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

from . import WORKLOADS, Workload, outlier_mask_words  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth_gen.cu")
_SO = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-shared", "-cudart", "shared", _SRC, "-o", tmp], check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            L.synth_gen_kv.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.synth_gen_kv.restype = ctypes.c_int
            L.synth_gen_q.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p]
            L.synth_gen_q.restype = ctypes.c_int
            _lib = L
    return _lib


class DeviceGenerator:
    """Fills torch device tensors with a workload's keys, values and queries."""

    def __init__(self, w: Workload, device="cuda"):
        import torch

        self.w = w
        self.torch = torch
        self.device = torch.device(device)
        self.masks = {}

    def _mask(self, layer: int):
        if layer not in self.masks:
            words = outlier_mask_words(self.w.seed, layer, self.w.n_kv, self.w.n_out, self.w.d_head)
            self.masks[layer] = self.torch.from_numpy(words.view(np.int64)).to(self.device)
        return self.masks[layer]

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def kv(self, layer: int, t0: int, nt: int, b0: int = 0, nb: int | None = None, out_k=None, out_v=None):
        """(k, v) [nb][nt][n_kv][d] float16 for tokens [t0, t0+nt)."""
        w = self.w
        nb = w.batch if nb is None else nb
        shape = (nb, nt, w.n_kv, w.d_head)
        k = out_k if out_k is not None else self.torch.empty(shape, dtype=self.torch.float16, device=self.device)
        v = out_v if out_v is not None else self.torch.empty(shape, dtype=self.torch.float16, device=self.device)
        s = self._stream()
        rc = lib().synth_gen_kv(w.seed, 0, layer, b0, nb, t0, nt, w.n_kv, w.d_head, self._mask(layer).data_ptr(),
                                int(w.gain), int(round(w.shift * 65536)), k.data_ptr(), s)
        assert rc == 0, rc
        rc = lib().synth_gen_kv(w.seed, 1, layer, b0, nb, t0, nt, w.n_kv, w.d_head, None, 0, 0, v.data_ptr(), s)
        assert rc == 0, rc
        return k, v

    def q(self, layer: int, step_token: int, b0: int = 0, nb: int | None = None, out=None):
        """Queries [nb][n_q][d] float16 of the decode step at token index ``step_token``."""
        w = self.w
        nb = w.batch if nb is None else nb
        q = out if out is not None else self.torch.empty((nb, w.n_q, w.d_head), dtype=self.torch.float16,
                                                         device=self.device)
        rc = lib().synth_gen_q(w.seed, layer, b0, nb, w.n_q, w.d_head, step_token, q.data_ptr(), self._stream())
        assert rc == 0, rc
        return q
