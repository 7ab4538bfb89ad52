"""ctypes binding of libkvq (the C ABI in include/kvq.h).

Argument marshalling only: every step of the quantized-KV path runs in the CUDA
kernels of ``libkvq.so``. Each function keeps the C name and raises ``KVQError``
on a non-OK status. Pointers are plain integers (``tensor.data_ptr()``) and the
stream is a ``cudaStream_t`` value (``torch.cuda.current_stream().cuda_stream``).
Loading fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkvq.so")

KVQ_OK = 0
STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_UNSUPPORTED", 3: "KVQ_ERR_CAPACITY",
                4: "KVQ_ERR_WORKSPACE", 5: "KVQ_ERR_CUDA"}
BUFFER_NAMES = ("k_codes", "k_meta", "k_resid", "v_codes", "v_meta")
DECODE_AUTO, DECODE_SIMT, DECODE_MMA = 0, 1, 2
DECODE_EARLY_PREFETCH = 1  # flag bits of kvq_decode_attention_ex / kvq_decode_step_ex
DECODE_ZERO_WAIT_LIMIT = 2
DECODE_ERR_WAIT_TIMEOUT = 1  # bit of the decode error word
EXPORTED = ("kvq_buffer_sizes", "kvq_quantize_append", "kvq_dequantize", "kvq_decode_workspace_size",
            "kvq_decode_attention", "kvq_decode_attention_impl", "kvq_decode_num_splits", "kvq_status_string",
            "kvq_version", "kvq_decode_attention_noalloc", "kvq_decode_step", "kvq_decode_attention_ex",
            "kvq_decode_step_ex", "kvq_decode_error", "kvq_decode_noalloc_error")


class KVQError(RuntimeError):
    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)} ({message})")
        self.status = status


class KVQDeviceError(RuntimeError):
    """A decode launch reported a device-side error in its workspace error word."""

    def __init__(self, word: int):
        names = [n for bit, n in ((DECODE_ERR_WAIT_TIMEOUT, "a wait for staged cache tiles timed out"),) if word & bit]
        super().__init__(f"decode error word 0x{word:x}: {'; '.join(names) or 'unknown bits'}")
        self.word = word


class kvq_config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "batch", "n_kv_heads", "gqa_ratio", "d_head",
                                               "max_seq_len", "bits", "k_group", "v_group", "residual_len",
                                               "v_bits", "symmetric", "k_outliers")]


class kvq_buffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in BUFFER_NAMES]


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libkvq.so; raises if it is missing (build it with bit_kv_cache_09_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libkvq.so not found at {path}: run `python -m bit_kv_cache_09_gb300.build` "
                               "(the quantized-KV path has no fallback)")
        L = ctypes.CDLL(path)
        cfgp, bufp, vp = ctypes.POINTER(kvq_config), ctypes.POINTER(kvq_buffers), ctypes.c_void_p
        L.kvq_buffer_sizes.argtypes = [cfgp, ctypes.POINTER(ctypes.c_size_t)]
        L.kvq_buffer_sizes.restype = ctypes.c_int
        L.kvq_quantize_append.argtypes = [cfgp, bufp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, vp, vp, vp]
        L.kvq_quantize_append.restype = ctypes.c_int
        L.kvq_dequantize.argtypes = [cfgp, bufp, ctypes.c_int32, ctypes.c_int64, vp, vp, vp]
        L.kvq_dequantize.restype = ctypes.c_int
        L.kvq_decode_workspace_size.argtypes = [cfgp, ctypes.c_int64]
        L.kvq_decode_workspace_size.restype = ctypes.c_size_t
        L.kvq_decode_attention.argtypes = [cfgp, bufp, ctypes.c_int32, ctypes.c_int64, vp, ctypes.c_float, vp, vp,
                                           ctypes.c_size_t, vp]
        L.kvq_decode_attention.restype = ctypes.c_int
        L.kvq_decode_attention_impl.argtypes = L.kvq_decode_attention.argtypes + [ctypes.c_int]
        L.kvq_decode_attention_impl.restype = ctypes.c_int
        L.kvq_decode_attention_noalloc.argtypes = [cfgp, bufp, ctypes.c_int32, ctypes.c_int64, vp, ctypes.c_float,
                                                   vp, vp]
        L.kvq_decode_attention_noalloc.restype = ctypes.c_int
        L.kvq_decode_step.argtypes = [cfgp, bufp, ctypes.c_int32, ctypes.c_int64, vp, vp, vp, ctypes.c_float, vp, vp,
                                      ctypes.c_size_t, vp]
        L.kvq_decode_step.restype = ctypes.c_int
        L.kvq_decode_attention_ex.argtypes = L.kvq_decode_attention.argtypes + [ctypes.c_uint32]
        L.kvq_decode_attention_ex.restype = ctypes.c_int
        L.kvq_decode_step_ex.argtypes = L.kvq_decode_step.argtypes + [ctypes.c_uint32]
        L.kvq_decode_step_ex.restype = ctypes.c_int
        L.kvq_decode_error.argtypes = [vp, ctypes.c_size_t, vp, ctypes.POINTER(ctypes.c_uint32)]
        L.kvq_decode_error.restype = ctypes.c_int
        L.kvq_decode_noalloc_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
        L.kvq_decode_noalloc_error.restype = ctypes.c_int
        L.kvq_decode_num_splits.argtypes = [cfgp, ctypes.c_int64]
        L.kvq_decode_num_splits.restype = ctypes.c_int32
        L.kvq_status_string.argtypes = [ctypes.c_int]
        L.kvq_status_string.restype = ctypes.c_char_p
        L.kvq_version.argtypes = []
        L.kvq_version.restype = ctypes.c_char_p
        _lib = L
        return L


def _check(fn: str, status: int) -> None:
    if status != KVQ_OK:
        raise KVQError(fn, status, kvq_status_string(status))


def make_config(*, n_layers, batch, n_kv_heads, gqa_ratio, d_head, max_seq_len, bits, k_group, v_group,
                residual_len, v_bits=0, symmetric=0, k_outliers=0) -> kvq_config:
    return kvq_config(n_layers, batch, n_kv_heads, gqa_ratio, d_head, max_seq_len, bits, k_group, v_group,
                      residual_len, v_bits, int(symmetric), int(k_outliers))


def make_buffers(ptrs) -> kvq_buffers:
    """ptrs: five device addresses (ints) in the order k_codes, k_meta, k_resid, v_codes, v_meta."""
    return kvq_buffers(*[ctypes.c_void_p(int(p)) for p in ptrs])


def kvq_status_string(status: int) -> str:
    return load().kvq_status_string(int(status)).decode()


def kvq_version() -> str:
    return load().kvq_version().decode()


def kvq_buffer_sizes(cfg: kvq_config) -> list[int]:
    out = (ctypes.c_size_t * 5)()
    _check("kvq_buffer_sizes", load().kvq_buffer_sizes(ctypes.byref(cfg), out))
    return [int(v) for v in out]


def kvq_quantize_append(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, n_new: int, k_f16: int,
                        v_f16: int, stream: int = 0) -> None:
    _check("kvq_quantize_append", load().kvq_quantize_append(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur,
                                                             n_new, k_f16, v_f16, stream))


def kvq_dequantize(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, k_out: int, v_out: int,
                   stream: int = 0) -> None:
    _check("kvq_dequantize", load().kvq_dequantize(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, k_out,
                                                   v_out, stream))


def kvq_decode_workspace_size(cfg: kvq_config, s_cur: int) -> int:
    return int(load().kvq_decode_workspace_size(ctypes.byref(cfg), s_cur))


def kvq_decode_num_splits(cfg: kvq_config, s_cur: int) -> int:
    return int(load().kvq_decode_num_splits(ctypes.byref(cfg), s_cur))


def kvq_decode_attention(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, q_f16: int,
                         softmax_scale: float, out: int, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check("kvq_decode_attention", load().kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur,
                                                               q_f16, softmax_scale, out, ws, ws_bytes, stream))


def kvq_decode_attention_impl(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, q_f16: int,
                              softmax_scale: float, out: int, ws: int, ws_bytes: int, stream: int = 0,
                              impl: int = DECODE_AUTO) -> None:
    _check("kvq_decode_attention_impl",
           load().kvq_decode_attention_impl(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, q_f16, softmax_scale,
                                            out, ws, ws_bytes, stream, impl))


def kvq_decode_step(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, k_f16: int, v_f16: int, q_f16: int,
                    softmax_scale: float, out: int, ws: int, ws_bytes: int, stream: int = 0) -> None:
    _check("kvq_decode_step", load().kvq_decode_step(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, k_f16, v_f16,
                                                     q_f16, softmax_scale, out, ws, ws_bytes, stream))


def kvq_decode_attention_ex(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, q_f16: int,
                            softmax_scale: float, out: int, ws: int, ws_bytes: int, stream: int = 0,
                            flags: int = 0) -> None:
    _check("kvq_decode_attention_ex",
           load().kvq_decode_attention_ex(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, q_f16, softmax_scale,
                                          out, ws, ws_bytes, stream, flags))


def kvq_decode_step_ex(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, k_f16: int, v_f16: int,
                       q_f16: int, softmax_scale: float, out: int, ws: int, ws_bytes: int, stream: int = 0,
                       flags: int = 0) -> None:
    _check("kvq_decode_step_ex", load().kvq_decode_step_ex(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, k_f16,
                                                           v_f16, q_f16, softmax_scale, out, ws, ws_bytes, stream,
                                                           flags))


def kvq_decode_attention_noalloc(cfg: kvq_config, bufs: kvq_buffers, layer: int, s_cur: int, q_f16: int,
                                 softmax_scale: float, out: int, stream: int = 0) -> None:
    """Decode attention with the library's static 16 MiB device scratch instead of a
    caller workspace (for callers that cannot allocate; calls must not overlap)."""
    _check("kvq_decode_attention_noalloc",
           load().kvq_decode_attention_noalloc(ctypes.byref(cfg), ctypes.byref(bufs), layer, s_cur, q_f16,
                                               softmax_scale, out, stream))


def kvq_decode_error(ws: int, ws_bytes: int, stream: int = 0) -> int:
    """The decode error word of workspace `ws` (synchronizes `stream`, then clears it)."""
    word = ctypes.c_uint32(0)
    _check("kvq_decode_error", load().kvq_decode_error(ws, ws_bytes, stream, ctypes.byref(word)))
    return int(word.value)


def kvq_decode_noalloc_error(stream: int = 0) -> int:
    """The error word of the last kvq_decode_attention_noalloc call on the current device."""
    word = ctypes.c_uint32(0)
    _check("kvq_decode_noalloc_error", load().kvq_decode_noalloc_error(stream, ctypes.byref(word)))
    return int(word.value)
