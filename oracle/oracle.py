"""ctypes/numpy wrapper of the C++ oracle (test infrastructure only).

Every function here marshals arguments to ``kvq_oracle.cpp``; none of the
method's arithmetic is restated in Python.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libkvq_oracle.so")
_lock = threading.Lock()
_lib = None

CXXFLAGS = ["-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the oracle library with g++ if it is missing or older than its source."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["g++", *CXXFLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _SO)
    return _SO


_u8p = ctypes.POINTER(ctypes.c_uint8)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            so = build()
            L = ctypes.CDLL(so)
            L.orc_f32_from_f16.argtypes = [ctypes.c_uint16]
            L.orc_f32_from_f16.restype = ctypes.c_float
            L.orc_f16_from_f32_rne.argtypes = [ctypes.c_float]
            L.orc_f16_from_f32_rne.restype = ctypes.c_uint16
            L.orc_f16_from_f32_ru.argtypes = [ctypes.c_float]
            L.orc_f16_from_f32_ru.restype = ctypes.c_uint16
            L.orc_qmin.argtypes = [ctypes.c_int]
            L.orc_qmin.restype = ctypes.c_int
            L.orc_qmax.argtypes = [ctypes.c_int]
            L.orc_qmax.restype = ctypes.c_int
            L.orc_quant_params.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _u16p, _u16p]
            L.orc_quant_params.restype = ctypes.c_int
            L.orc_quantize_values.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint16,
                                              ctypes.c_uint16, _u8p]
            L.orc_quantize_values.restype = ctypes.c_int
            L.orc_dequantize_value.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint16, ctypes.c_uint16]
            L.orc_dequantize_value.restype = ctypes.c_float
            L.orc_kv_bytes.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_double] * 3
            L.orc_kv_bytes.restype = ctypes.c_double
            L.orc_v_pos.argtypes = [ctypes.c_int, ctypes.c_int]
            L.orc_v_pos.restype = ctypes.c_int64
            L.orc_pack_k_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
            L.orc_pack_k_row.restype = None
            L.orc_unpack_k_row.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, _u8p]
            L.orc_unpack_k_row.restype = None
            L.orc_pack_v_token.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _u8p]
            L.orc_pack_v_token.restype = None
            L.orc_unpack_v_token.argtypes = [_u8p, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _u8p]
            L.orc_unpack_v_token.restype = None
            L.orc_cache_state.argtypes = [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_int, _u16p, _u16p, _u8p, _u16p,
                                                               _u16p, _u16p, _u8p, _u16p, _u8p, _u8p]
            L.orc_cache_state.restype = ctypes.c_int64
            L.orc_dequantize_state.argtypes = [ctypes.c_int] * 6 + [ctypes.c_int64, ctypes.c_int, _u8p, _u16p, _u16p,
                                                                    _u16p, _u8p, _u16p, _f32p, _f32p]
            L.orc_dequantize_state.restype = ctypes.c_int
            L.orc_sym_params.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _u16p]
            L.orc_sym_params.restype = ctypes.c_int
            L.orc_sym_quantize.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_uint16, _u8p]
            L.orc_sym_quantize.restype = ctypes.c_int
            L.orc_sym_dequantize_value.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_uint16]
            L.orc_sym_dequantize_value.restype = ctypes.c_float
            L.orc_split_outliers.argtypes = [_u16p, ctypes.c_int, ctypes.c_int, _u16p, _u16p, _u16p]
            L.orc_split_outliers.restype = ctypes.c_int
            L.orc_cache_state_sym.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, _u16p, _u16p, _u8p, _u16p,
                                              _u16p, _u8p, _u16p, _u8p, _u8p]
            L.orc_cache_state_sym.restype = ctypes.c_int
            L.orc_dequantize_state_sym.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, _u8p, _u16p, _u16p,
                                                   _u8p, _u16p, _f32p, _f32p]
            L.orc_dequantize_state_sym.restype = ctypes.c_int
            L.orc_attention.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, _u16p, _f32p, _f32p,
                                        ctypes.c_float, _f32p]
            L.orc_attention.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ct):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ct)


def _as_u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


# ----------------------------------------------------------------------------- scalars
def f32_from_f16(h: int) -> float:
    return float(lib().orc_f32_from_f16(int(h)))


def f16_from_f32_rne(x: float) -> int:
    return int(lib().orc_f16_from_f32_rne(float(np.float32(x))))


def f16_from_f32_ru(x: float) -> int:
    return int(lib().orc_f16_from_f32_ru(float(np.float32(x))))


def qmin(bits: int) -> int:
    return int(lib().orc_qmin(bits))


def qmax(bits: int) -> int:
    return int(lib().orc_qmax(bits))


def quant_params(x, bits: int) -> tuple[int, int]:
    """(scale, zero_point) binary16 bit patterns of one group of binary16 values."""
    x = _as_u16(x).ravel()
    s = ctypes.c_uint16()
    z = ctypes.c_uint16()
    rc = lib().orc_quant_params(_ptr(x, _u16p), x.size, 1, bits, ctypes.byref(s), ctypes.byref(z))
    if rc != 0:
        raise ValueError("bad group")
    return int(s.value), int(z.value)


def quantize_values(x, bits: int, scale_h: int, zp_h: int) -> np.ndarray:
    x = _as_u16(x).ravel()
    u = np.zeros(x.size, np.uint8)
    rc = lib().orc_quantize_values(_ptr(x, _u16p), x.size, 1, bits, scale_h, zp_h, _ptr(u, _u8p))
    if rc != 0:
        raise ValueError("bad arguments")
    return u


def dequantize_value(u: int, bits: int, scale_h: int, zp_h: int) -> float:
    return float(lib().orc_dequantize_value(int(u), bits, scale_h, zp_h))


def kv_bytes(L, n_kv, d_head, S, bits_per_elem, meta_bytes=0.0, group_elems=0.0) -> float:
    return float(lib().orc_kv_bytes(L, n_kv, d_head, S, bits_per_elem, meta_bytes, group_elems))


# ----------------------------------------------------------------------------- layout
def v_pos(d: int, c: int) -> int:
    return int(lib().orc_v_pos(d, c))


def pack_k_row(u, d: int, bits: int) -> np.ndarray:
    u = np.ascontiguousarray(u, np.uint8)
    row = np.zeros(d * bits // 8, np.uint8)
    lib().orc_pack_k_row(_ptr(u, _u8p), d, bits, _ptr(row, _u8p))
    return row


def unpack_k_row(row, d: int, bits: int) -> np.ndarray:
    row = np.ascontiguousarray(row, np.uint8)
    u = np.zeros(d, np.uint8)
    lib().orc_unpack_k_row(_ptr(row, _u8p), d, bits, _ptr(u, _u8p))
    return u


def pack_v_token(u, d: int, bits: int, t: int, pairs: np.ndarray) -> None:
    u = np.ascontiguousarray(u, np.uint8)
    assert pairs.dtype == np.uint8 and pairs.flags["C_CONTIGUOUS"]
    assert pairs.size >= (t // 2 + 1) * 2 * d * bits // 8
    lib().orc_pack_v_token(_ptr(u, _u8p), d, bits, t, _ptr(pairs, _u8p))


def unpack_v_token(pairs, d: int, bits: int, t: int) -> np.ndarray:
    pairs = np.ascontiguousarray(pairs, np.uint8)
    assert pairs.size >= (t // 2 + 1) * 2 * d * bits // 8
    u = np.zeros(d, np.uint8)
    lib().orc_unpack_v_token(_ptr(pairs, _u8p), d, bits, t, _ptr(u, _u8p))
    return u


# ----------------------------------------------------------------------------- cache state
@dataclass
class OracleState:
    """Cache state of one (batch row, kv head) slice after T tokens, in the packed layout."""

    T: int
    Tq: int
    k_codes: np.ndarray  # [Tq][d*b/8] uint8
    k_meta: np.ndarray  # [Tq/G][d][2] uint16 (scale, zp) binary16 bits
    k_resid: np.ndarray  # [R_eff][d] uint16
    v_codes: np.ndarray  # [ceil(T/2)][2*d*b/8] uint8
    v_meta: np.ndarray  # [ceil(T/2)][d/Gv][4] uint16 pair records {s(2p), s(2p+1), zp(2p), zp(2p+1)}
    k_u: np.ndarray  # [Tq][d] unpacked key codes
    v_u: np.ndarray  # [T][d] unpacked value codes
    k_sparse: np.ndarray = None  # isolated key entries [Tq][k][2] (channel, binary16 value), or None


def cache_state(k_hist, v_hist, *, d: int, bits: int, G: int, Gv: int, R: int, v_bits: int = 0,
                k_outliers: int = 0) -> OracleState:
    """Quantized cache of one (b, h) slice from its binary16 token history [T][d]; keys
    with `bits`-bit codes, values with `v_bits`-bit codes (0: the same as the keys). With
    k_outliers > 0 every quantized key row gives up its k farthest entries (k_sparse)
    before the per-channel groups are formed."""
    v_bits = v_bits or bits
    k = _as_u16(k_hist)
    v = _as_u16(v_hist)
    T = k.shape[0]
    assert k.shape == (T, d) and v.shape == (T, d)
    R_eff = R if R > 0 else G
    Tq = (T // R_eff) * R_eff
    rowK = d * bits // 8
    k_codes = np.zeros((Tq, rowK), np.uint8)
    k_meta = np.zeros((Tq // G, d, 2), np.uint16)
    k_resid = np.zeros((R_eff, d), np.uint16)
    v_codes = np.zeros(((T + 1) // 2, 2 * (d * v_bits // 8)), np.uint8)
    v_meta = np.zeros(((T + 1) // 2, d // Gv, 4), np.uint16)
    k_u = np.zeros((Tq, d), np.uint8)
    v_u = np.zeros((T, d), np.uint8)
    k_sparse = np.zeros((Tq, k_outliers, 2), np.uint16)
    # zero-size arrays still need a valid pointer
    bufs = [np.zeros(1, a.dtype) if a.size == 0 else a
            for a in (k_codes, k_meta, k_resid, v_codes, v_meta, k_u, v_u, k_sparse)]
    kk = k if k.size else np.zeros(1, np.uint16)
    vv = v if v.size else np.zeros(1, np.uint16)
    rc = lib().orc_cache_state(d, bits, v_bits, G, Gv, R, T, k_outliers, _ptr(kk, _u16p), _ptr(vv, _u16p),
                               _ptr(bufs[0], _u8p), _ptr(bufs[1], _u16p), _ptr(bufs[7], _u16p), _ptr(bufs[2], _u16p),
                               _ptr(bufs[3], _u8p), _ptr(bufs[4], _u16p), _ptr(bufs[5], _u8p), _ptr(bufs[6], _u8p))
    if rc < 0:
        raise ValueError("bad cache shape")
    assert rc == Tq
    return OracleState(T, Tq, k_codes, k_meta, k_resid, v_codes, v_meta, k_u, v_u,
                       k_sparse if k_outliers > 0 else None)


def value_meta(st: OracleState) -> np.ndarray:
    """The value metadata of a state per token: [T][d/Gv][2] (scale, zero point) binary16
    bits, read out of the pair records (token t sits in record t // 2, half t % 2)."""
    rec = st.v_meta
    t = np.arange(st.T)
    return np.stack([rec[t // 2, :, t % 2], rec[t // 2, :, 2 + t % 2]], axis=-1) if st.T else np.zeros(
        (0, rec.shape[1], 2), np.uint16)


def dequantize_state(st: OracleState, *, d: int, bits: int, G: int, Gv: int, R: int, v_bits: int = 0):
    """(k_hat, v_hat) binary32 [T][d] from a packed slice state (v_bits 0: same as bits)."""
    v_bits = v_bits or bits
    T = st.T
    k_out = np.zeros((max(T, 1), d), np.float32)
    v_out = np.zeros((max(T, 1), d), np.float32)

    def nz(a):
        return np.ascontiguousarray(a) if a.size else np.zeros(1, a.dtype)

    ks = st.k_sparse if st.k_sparse is not None else np.zeros((st.Tq, 0, 2), np.uint16)
    rc = lib().orc_dequantize_state(d, bits, v_bits, G, Gv, R, T, ks.shape[1], _ptr(nz(st.k_codes), _u8p),
                                    _ptr(nz(st.k_meta), _u16p), _ptr(nz(ks), _u16p), _ptr(nz(st.k_resid), _u16p),
                                    _ptr(nz(st.v_codes), _u8p), _ptr(nz(st.v_meta), _u16p), _ptr(k_out, _f32p),
                                    _ptr(v_out, _f32p))
    if rc != 0:
        raise ValueError("bad cache shape")
    return k_out[:T], v_out[:T]


# ----------------------------------------------------------------------------- symmetric scheme
def sym_params(x, bits: int = 8) -> int:
    """Symmetric scale (binary16 bits) of a vector of binary16 values (zero point 0)."""
    x = _as_u16(x).ravel()
    s = ctypes.c_uint16()
    if lib().orc_sym_params(_ptr(x, _u16p), x.size, 1, bits, ctypes.byref(s)) != 0:
        raise ValueError("bad vector")
    return int(s.value)


def sym_quantize(x, bits: int, scale_h: int) -> np.ndarray:
    """Codes u = q - q_min of q = clamp(round(x / scale), q_min, q_max)."""
    x = _as_u16(x).ravel()
    u = np.zeros(max(x.size, 1), np.uint8)
    xx = x if x.size else np.zeros(1, np.uint16)
    if lib().orc_sym_quantize(_ptr(xx, _u16p), x.size, 1, bits, scale_h, _ptr(u, _u8p)) != 0:
        raise ValueError("bad arguments")
    return u[:x.size]


def sym_dequantize_value(u: int, bits: int, scale_h: int) -> float:
    return float(lib().orc_sym_dequantize_value(int(u), bits, scale_h))


def split_outliers(x, k: int):
    """(channels [k], binary16 values [k], dense row) of the dense-and-sparse split."""
    x = _as_u16(x).ravel()
    idx = np.zeros(max(k, 1), np.uint16)
    val = np.zeros(max(k, 1), np.uint16)
    dense = np.zeros(x.size, np.uint16)
    if lib().orc_split_outliers(_ptr(x, _u16p), x.size, k, _ptr(idx, _u16p), _ptr(val, _u16p), _ptr(dense, _u16p)) != 0:
        raise ValueError("bad arguments")
    return idx[:k], val[:k], dense


def cache_state_sym(k_hist, v_hist, *, d: int, k_outliers: int = 0) -> OracleState:
    """Symmetric per-token int8 cache of one (b, h) slice: keys and values each with one
    scale per token and zero point 0, no residual window. k_meta holds the per-token key
    scales [T] (binary16 bits), v_meta [ceil(T/2)][1][4] the value pair records (zero
    points +0); with
    k_outliers > 0, k_sparse [T][k][2] the isolated key entries (channel, binary16)."""
    k = _as_u16(k_hist)
    v = _as_u16(v_hist)
    T = k.shape[0]
    assert k.shape == (T, d) and v.shape == (T, d)
    k_codes = np.zeros((T, d), np.uint8)
    k_meta = np.zeros((T,), np.uint16)
    v_codes = np.zeros(((T + 1) // 2, 2 * d), np.uint8)
    v_meta = np.zeros(((T + 1) // 2, 1, 4), np.uint16)
    k_u = np.zeros((T, d), np.uint8)
    v_u = np.zeros((T, d), np.uint8)
    k_sparse = np.zeros((T, k_outliers, 2), np.uint16)
    bufs = [np.zeros(1, a.dtype) if a.size == 0 else a
            for a in (k_codes, k_meta, v_codes, v_meta, k_u, v_u, k_sparse)]
    kk = k if k.size else np.zeros(1, np.uint16)
    vv = v if v.size else np.zeros(1, np.uint16)
    rc = lib().orc_cache_state_sym(d, T, k_outliers, _ptr(kk, _u16p), _ptr(vv, _u16p), _ptr(bufs[0], _u8p),
                                   _ptr(bufs[1], _u16p), _ptr(bufs[6], _u16p), _ptr(bufs[2], _u8p),
                                   _ptr(bufs[3], _u16p), _ptr(bufs[4], _u8p), _ptr(bufs[5], _u8p))
    if rc != 0:
        raise ValueError("bad cache shape")
    return OracleState(T, T, k_codes, k_meta, np.zeros((0, d), np.uint16), v_codes, v_meta, k_u, v_u, k_sparse)


def dequantize_state_sym(st: OracleState, *, d: int):
    """(k_hat, v_hat) binary32 [T][d] of a symmetric per-token state."""
    T = st.T
    k_out = np.zeros((max(T, 1), d), np.float32)
    v_out = np.zeros((max(T, 1), d), np.float32)

    def nz(a):
        return np.ascontiguousarray(a) if a.size else np.zeros(1, a.dtype)

    ks = st.k_sparse if st.k_sparse is not None else np.zeros((T, 0, 2), np.uint16)
    rc = lib().orc_dequantize_state_sym(d, T, ks.shape[1], _ptr(nz(st.k_codes), _u8p), _ptr(nz(st.k_meta), _u16p),
                                        _ptr(nz(ks), _u16p), _ptr(nz(st.v_codes), _u8p), _ptr(nz(st.v_meta), _u16p),
                                        _ptr(k_out, _f32p), _ptr(v_out, _f32p))
    if rc != 0:
        raise ValueError("bad cache shape")
    return k_out[:T], v_out[:T]


def attention(q, k_hat, v_hat, softmax_scale: float) -> np.ndarray:
    """Exact softmax attention (binary64 inside) of r binary16 queries [r][d]."""
    q = _as_u16(q)
    r, d = q.shape
    k_hat = np.ascontiguousarray(k_hat, np.float32)
    v_hat = np.ascontiguousarray(v_hat, np.float32)
    T = k_hat.shape[0]
    out = np.zeros((r, d), np.float32)
    rc = lib().orc_attention(d, r, T, _ptr(q, _u16p), _ptr(k_hat, _f32p), _ptr(v_hat, _f32p),
                             float(softmax_scale), _ptr(out, _f32p))
    if rc != 0:
        raise ValueError("bad attention arguments")
    return out
