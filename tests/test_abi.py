"""The C-ABI library without a GPU: it loads, exports every declared entry point,
and rejects bad arguments on the host before any launch."""

import ctypes
import os
import re

import pytest

import oracle
from bit_kv_cache_09_gb300 import build as kvq_build
from bit_kv_cache_09_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    kvq_build.build()
    return kvq.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in kvq.EXPORTED
    assert kvq.kvq_version().startswith("kvq ")


def good_cfg(**kw):
    base = dict(n_layers=2, batch=3, n_kv_heads=2, gqa_ratio=4, d_head=128, max_seq_len=1000, bits=4, k_group=32,
                v_group=64, residual_len=128)
    base.update(kw)
    return kvq.make_config(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(bits=3), 2), (dict(bits=16), 2), (dict(d_head=64), 2), (dict(k_group=48), 2), (dict(v_group=16), 2),
    (dict(residual_len=100), 1), (dict(residual_len=2048), 2), (dict(gqa_ratio=9), 2), (dict(batch=0), 1),
    (dict(max_seq_len=0), 1), (dict(n_kv_heads=256), 2), (dict(v_bits=3), 2), (dict(bits=4, v_bits=8), 2),
    (dict(bits=4, v_bits=2), 2), (dict(bits=2, v_bits=4), 2),
    # symmetric per-token int8: 8-bit codes, one value group, no residual window
    (dict(symmetric=2), 1), (dict(symmetric=1, bits=4, v_group=128, residual_len=0), 2),
    (dict(symmetric=1, bits=8, v_bits=4, v_group=128, residual_len=0), 2),
    (dict(symmetric=1, bits=8, v_group=64, residual_len=0), 2), (dict(symmetric=1, bits=8, v_group=128), 1),
    # outlier isolation: 0..4 entries per token; with per-channel keys for r <= 4 only
    (dict(k_outliers=2, gqa_ratio=8), 2), (dict(k_outliers=5), 2),
    (dict(symmetric=1, bits=8, v_group=128, residual_len=0, k_outliers=5), 2),
    (dict(symmetric=1, bits=8, v_group=128, residual_len=0, k_outliers=-1), 2),
])
def test_bad_configs_are_rejected(lib, kw, status):
    sizes = (ctypes.c_size_t * 5)()
    assert lib.kvq_buffer_sizes(ctypes.byref(good_cfg(**kw)), sizes) == status
    assert kvq.kvq_decode_workspace_size(good_cfg(**kw), 10) == 0


def test_buffer_sizes_follow_the_bytes_formula(lib):
    """Code bytes are the pages' 2*L*n_kv*d*S*bits/8 (batch rows count as extra
    sequences); metadata adds one (scale, zero) binary16 pair per group."""
    for bits, G, Gv, R in [(8, 32, 128, 0), (4, 128, 64, 128), (2, 32, 32, 128)]:
        L, B, H, S = 3, 2, 4, 1024
        cfg = good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=bits, k_group=G, v_group=Gv,
                       residual_len=R)
        kc, km, kr, vc, vm = kvq.kvq_buffer_sizes(cfg)
        assert kc + vc == oracle.kv_bytes(L, H * B, 128, S, bits)
        assert km == oracle.kv_bytes(L, H * B, 128, S, 0, 4, G) / 2
        assert vm == oracle.kv_bytes(L, H * B, 128, S, 0, 4, Gv) / 2
        R_eff = R or G
        assert kr == L * B * H * R_eff * 128 * 2


def test_mixed_width_buffer_sizes(lib):
    """8-bit keys with 4-bit values: key codes at 8 bits, value codes at 4 bits per element."""
    L, B, H, S = 3, 2, 4, 1024
    same = kvq.kvq_buffer_sizes(good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=8, k_group=128,
                                         v_group=64, residual_len=128))
    mixed = kvq.kvq_buffer_sizes(good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=8, k_group=128,
                                          v_group=64, residual_len=128, v_bits=4))
    assert mixed[0] == same[0] and mixed[1] == same[1] and mixed[2] == same[2] and mixed[4] == same[4]
    assert mixed[3] == oracle.kv_bytes(L, H * B, 128, S, 4) / 2
    assert kvq.kvq_buffer_sizes(good_cfg(bits=8, v_bits=8)) == kvq.kvq_buffer_sizes(good_cfg(bits=8))


def test_symmetric_buffer_sizes(lib):
    """Symmetric per-token int8: key and value rows of d bytes, one binary16 key scale and
    one (scale, 0) value pair per token, no residual buffer."""
    L, B, H, S = 3, 2, 4, 1000
    S_pad = 1024
    sizes = kvq.kvq_buffer_sizes(good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=8, v_group=128,
                                          residual_len=0, symmetric=1))
    n = L * B * H
    assert sizes == [n * S_pad * 128, n * S_pad * 2, 0, n * S_pad * 128, n * S_pad * 4]
    # the bytes the pages count for an int8 cache, plus 6 metadata bytes per token and head
    assert sizes[0] + sizes[3] == oracle.kv_bytes(L, H * B, 128, S_pad, 8)


def test_outlier_buffer_sizes(lib):
    """k_outliers = k adds k (channel, binary16) entries of 4 bytes per token after the
    per-token key scales."""
    L, B, H, S = 2, 3, 2, 1000
    S_pad, n = 1024, 2 * 3 * 2
    for k in range(5):
        sizes = kvq.kvq_buffer_sizes(good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=8, v_group=128,
                                              residual_len=0, symmetric=1, k_outliers=k))
        assert sizes[1] == n * S_pad * (2 + 4 * k)
        assert sizes[0] == sizes[3] == n * S_pad * 128 and sizes[2] == 0
    # per-channel keys: the entries follow the (scale, zero point) pairs of the key groups
    for k in range(5):
        sizes = kvq.kvq_buffer_sizes(good_cfg(n_layers=L, batch=B, n_kv_heads=H, max_seq_len=S, bits=4, k_group=32,
                                              k_outliers=k))
        assert sizes[1] == n * ((S_pad // 32) * 128 * 4 + S_pad * 4 * k)


def _bufs(ptr=4096):
    return kvq.make_buffers([ptr, ptr + 4096, ptr + 8192, ptr + 12288, ptr + 16384])


def test_append_argument_checks(lib):
    cfg = good_cfg()
    B = ctypes.byref
    bufs = _bufs()
    # wrong layer, negative s_cur, empty append, capacity, null/misaligned inputs: nothing launches
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 2, 0, 1, 4096, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 0, -1, 1, 4096, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 0, 0, 0, 4096, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 0, 999, 2, 4096, 4096, None) == 3
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 0, 0, 1, None, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), B(bufs), 0, 0, 1, 4098, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), B(_bufs(4100)), 0, 0, 1, 4096, 4096, None) == 1
    assert lib.kvq_quantize_append(B(cfg), None, 0, 0, 1, 4096, 4096, None) == 1
    assert lib.kvq_quantize_append(None, B(bufs), 0, 0, 1, 4096, 4096, None) == 1


def test_decode_argument_checks(lib):
    cfg = good_cfg()
    B = ctypes.byref
    bufs = _bufs()
    need = kvq.kvq_decode_workspace_size(cfg, 500)
    assert need > 0
    args = lambda layer, s, q, out, ws, wsb, scale=0.088: (B(cfg), B(bufs), layer, s, q, ctypes.c_float(scale), out,  # noqa: E731
                                                           ws, wsb, None)
    assert lib.kvq_decode_attention(*args(0, 0, 4096, 4096, 4096, need)) == 1  # no tokens
    assert lib.kvq_decode_attention(*args(0, 1001, 4096, 4096, 4096, need)) == 3
    assert lib.kvq_decode_attention(*args(0, 500, 4096, 4096, 4096, need - 1)) == 4
    assert lib.kvq_decode_attention(*args(0, 500, 4096, 4096, None, need)) == 4
    assert lib.kvq_decode_attention(*args(0, 500, 4100, 4096, 4096, need)) == 1
    assert lib.kvq_decode_attention(*args(0, 500, 4096, 4096, 4096, need, float("nan"))) == 1
    assert lib.kvq_decode_attention(*args(5, 500, 4096, 4096, 4096, need)) == 1
    assert lib.kvq_dequantize(B(cfg), B(bufs), 0, 0, 4096, 4096, None) == 1
    assert lib.kvq_dequantize(B(cfg), B(bufs), 0, 1001, 4096, 4096, None) == 3


def test_decode_flag_checks(lib):
    """Unknown flag bits of the _ex entry points are rejected on the host; the early-prefetch
    bit passes the flag check and meets the same argument checks as the plain calls."""
    cfg = good_cfg()
    B = ctypes.byref
    bufs = _bufs()
    need = kvq.kvq_decode_workspace_size(cfg, 500)
    att = lambda s, flags: lib.kvq_decode_attention_ex(B(cfg), B(bufs), 0, s, 4096, ctypes.c_float(0.088), 4096,  # noqa: E731
                                                       4096, need, None, flags)
    step = lambda s, flags: lib.kvq_decode_step_ex(B(cfg), B(bufs), 0, s, 4096, 4096, 4096, ctypes.c_float(0.088),  # noqa: E731
                                                   4096, 4096, need, None, flags)
    assert kvq.DECODE_EARLY_PREFETCH == 1 and kvq.DECODE_ZERO_WAIT_LIMIT == 2
    assert att(500, 4) == 1 and att(500, 0x80000000) == 1
    assert step(499, 4) == 1 and step(499, 7) == 1
    for flag in (kvq.DECODE_EARLY_PREFETCH, kvq.DECODE_ZERO_WAIT_LIMIT):
        assert att(0, flag) == 1      # no tokens
        assert att(1001, flag) == 3   # capacity
        assert step(1000, flag) == 3  # capacity
        assert step(-1, flag) == 1


def test_error_word_reader_checks(lib):
    """kvq_decode_error / kvq_decode_noalloc_error reject a missing output, workspace or a
    workspace too small for the error word on the host, before touching the device."""
    err = ctypes.c_uint32(7)
    assert lib.kvq_decode_error(4096, 4096, None, None) == 1
    assert lib.kvq_decode_error(None, 4096, None, ctypes.byref(err)) == 4
    assert lib.kvq_decode_error(4100, 4096, None, ctypes.byref(err)) == 4
    assert lib.kvq_decode_error(4096, 255, None, ctypes.byref(err)) == 4
    assert lib.kvq_decode_noalloc_error(None, None) == 1
    assert err.value == 7


def test_early_prefetch_flag_follows_the_previous_launch():
    """The cache object sets the early-prefetch bit unless its previous launch on the same
    stream wrote the same layer (host logic only)."""
    from bit_kv_cache_09_gb300.cache import QuantizedKVCache
    c = QuantizedKVCache.__new__(QuantizedKVCache)
    c._last = None
    E = kvq.DECODE_EARLY_PREFETCH
    assert c._early(7, 0, None) == E               # nothing launched yet
    c._last = (7, 0, True)                          # wrote layer 0 on stream 7
    assert c._early(7, 0, None) == 0
    assert c._early(7, 1, None) == E                # another layer
    assert c._early(8, 0, None) == E                # another stream
    assert c._early(7, 1, False) == 0 and c._early(7, 0, True) == E   # explicit choice wins
    c._last = (7, 0, False)                         # read layer 0 only
    assert c._early(7, 0, None) == E


def test_status_strings(lib):
    for s in range(6):
        assert kvq.kvq_status_string(s)
    with pytest.raises(kvq.KVQError):
        kvq.kvq_buffer_sizes(good_cfg(bits=5))
